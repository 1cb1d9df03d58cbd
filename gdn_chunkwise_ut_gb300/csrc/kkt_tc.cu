// kkt_tc.cu -- the tensor-core kernel (kkt_tc.cuh) at d_k = d_v = 128, and the entry points that
// choose the head dimensions.  The other (d_k, d_v) pairs compile in their own translation units
// (kkt_tc_d64.cu, kkt_tc_k128v64.cu, kkt_tc_k64v128.cu).
#include "kkt_tc.cuh"

namespace kkt {

int launch_tc_d64(const Problem &p);      // kkt_tc_d64.cu
int launch_tc_k128v64(const Problem &p);  // kkt_tc_k128v64.cu
int launch_tc_k64v128(const Problem &p);  // kkt_tc_k64v128.cu

bool tc_supports(int dk, int dv, int C, int io) {
    return io == KKT_IO_BF16 && (dk == 64 || dk == 128) && (dv == 64 || dv == 128) &&
           (C == 32 || C == 64 || C == 128);
}

int debug_bounds_tc(BoundsRecord *out) { return read_bounds_record(out); }

int launch_tc(const Problem &p) {
    if (p.dk != p.dv) return p.dk == 128 ? launch_tc_k128v64(p) : launch_tc_k64v128(p);
    if (p.dk == 64) return launch_tc_d64(p);
    switch (p.C) {
        case 32: return launch_tc_t<32, 128, 128>(p);
        case 64: return launch_tc_t<64, 128, 128>(p);
        case 128: return launch_tc_t<128, 128, 128>(p);
        default: return KKT_ERR_UNSUPPORTED;
    }
}

}  // namespace kkt
