// kkt_tc.cu -- the tensor-core kernel (kkt_tc.cuh) at head dimension d_k = d_v = 128, and the
// entry points that choose the head dimension.  The d = 64 instantiations compile in their own
// translation unit (kkt_tc_d64.cu).
#include "kkt_tc.cuh"

namespace kkt {

int launch_tc_d64(const Problem &p);  // kkt_tc_d64.cu

bool tc_supports(int dk, int dv, int C, int io) {
    return io == KKT_IO_BF16 && dk == dv && (dk == 64 || dk == 128) && (C == 32 || C == 64 || C == 128);
}

int debug_bounds_tc(BoundsRecord *out) { return read_bounds_record(out); }

int launch_tc(const Problem &p) {
    if (p.dk == 64) return launch_tc_d64(p);
    switch (p.C) {
        case 32: return launch_tc_t<32, 128>(p);
        case 64: return launch_tc_t<64, 128>(p);
        case 128: return launch_tc_t<128, 128>(p);
        default: return KKT_ERR_UNSUPPORTED;
    }
}

}  // namespace kkt
