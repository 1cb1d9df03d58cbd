// kkt_tc_d64.cu -- the tensor-core kernel (kkt_tc.cuh) at head dimension d_k = d_v = 64: K and V
// rows are one 64-column TMA box, the Gram contracts over 64, and D = T~ [K | V] has 128 columns.
#include "kkt_tc.cuh"

namespace kkt {

int debug_bounds_tc_d64(BoundsRecord *out) { return read_bounds_record(out); }

int launch_tc_d64(const Problem &p) {
    switch (p.C) {
        case 32: return launch_tc_t<32, 64, 64>(p);
        case 64: return launch_tc_t<64, 64, 64>(p);
        case 128: return launch_tc_t<128, 64, 64>(p);
        default: return KKT_ERR_UNSUPPORTED;
    }
}

}  // namespace kkt
