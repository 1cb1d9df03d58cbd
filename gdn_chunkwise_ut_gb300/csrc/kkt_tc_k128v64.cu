// kkt_tc_k128v64.cu -- the tensor-core kernel (kkt_tc.cuh) at d_k = 128, d_v = 64.
// K rows are two 64-column TMA boxes and V rows one: the Gram contracts over 128, and
// D = T~ [K | V] has 192 columns (128 of W, then 64 of U~).
#include "kkt_tc.cuh"

namespace kkt {

int debug_bounds_tc_k128v64(BoundsRecord *out) { return read_bounds_record(out); }

int launch_tc_k128v64(const Problem &p) {
    switch (p.C) {
        case 32: return launch_tc_t<32, 128, 64>(p);
        case 64: return launch_tc_t<64, 128, 64>(p);
        case 128: return launch_tc_t<128, 128, 64>(p);
        default: return KKT_ERR_UNSUPPORTED;
    }
}

}  // namespace kkt
