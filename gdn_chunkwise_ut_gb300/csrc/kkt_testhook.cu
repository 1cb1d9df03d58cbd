// kkt_testhook.cu -- test hooks of libkkt (declared in kkt_test.h): code paths that
// correct inputs never reach, made reachable for the tests of failure detection.
#include <cstdint>
#include <cuda_runtime.h>

#include "kkt_internal.cuh"
#include "kkt_test.h"

namespace {
bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

extern "C" int kkt_test_stalled_solve(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                                      int B, int T, int H, int dk, int dv, int C,
                                      float *T_out, void *W_out, void *U_out, struct CUstream_st *stream) {
    if (!k || !v || !beta || !W_out || !U_out) return KKT_ERR_ARG;  // T_out may be NULL
    if (B < 1 || T < 0 || H < 1 || H > 65535) return KKT_ERR_ARG;
    const int which = kkt_select_kernel(dk, dv, C, KKT_IO_BF16, KKT_KERNEL_TC);
    if (which < 0) return -which;
    if (!aligned_to(k, 16) || !aligned_to(v, 16) || !aligned_to(T_out, 16) || !aligned_to(W_out, 16) ||
        !aligned_to(U_out, 16) || !aligned_to(beta, 4) || (cu_seqlens && !aligned_to(cu_seqlens, 4)))
        return KKT_ERR_ALIGN;
    const int64_t ntok = cu_seqlens ? (int64_t)T : (int64_t)B * T;
    if (ntok == 0) return KKT_OK;
    if (ntok / C + B > 0x7fffffffLL) return KKT_ERR_ARG;

    kkt::Problem p;
    p.k = k; p.v = v; p.beta = beta; p.cu_seqlens = cu_seqlens;
    p.nseq = B; p.T = T; p.ntok = ntok;
    p.H = H; p.dk = dk; p.dv = dv; p.C = C;
    p.T_out = T_out; p.W_out = W_out; p.U_out = U_out;
    p.io = KKT_IO_BF16;
    p.stream = reinterpret_cast<cudaStream_t>(stream);
    p.trace = nullptr;
    p.tile_counter = nullptr;  // fixed round robin: no workspace needed
    p.stall_first_tile = 1;
    const int st = kkt::status_ptr(&p.status);
    if (st != KKT_OK) return st;
    return kkt::launch_tc(p);
}
