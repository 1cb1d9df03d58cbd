// kkt_tc.cu -- persistent tcgen05 + TMA kernel (bf16 I/O).  Not built yet:
// reports no supported shapes, so every call takes the SIMT kernel.
#include "kkt_internal.cuh"

namespace kkt {

bool tc_supports(int, int, int, int) { return false; }

int launch_tc(const Problem &) { return KKT_ERR_UNSUPPORTED; }

}  // namespace kkt
