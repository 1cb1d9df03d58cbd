// kkt_tc_k64v128.cu -- the tensor-core kernel (kkt_tc.cuh) at d_k = 64, d_v = 128.
// K rows are one 64-column TMA box and V rows two: the Gram contracts over 64, and
// D = T~ [K | V] has 192 columns (64 of W, then 128 of U~).
#include "kkt_tc.cuh"

namespace kkt {

int debug_bounds_tc_k64v128(BoundsRecord *out) { return read_bounds_record(out); }

int launch_tc_k64v128(const Problem &p) {
    switch (p.C) {
        case 32: return launch_tc_t<32, 64, 128>(p);
        case 64: return launch_tc_t<64, 64, 128>(p);
        case 128: return launch_tc_t<128, 64, 128>(p);
        default: return KKT_ERR_UNSUPPORTED;
    }
}

}  // namespace kkt
