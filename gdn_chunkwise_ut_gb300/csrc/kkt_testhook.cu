// kkt_testhook.cu -- test hooks of libkkt (declared in kkt_test.h): code paths that
// correct inputs never reach, made reachable for the tests of failure detection.
#include <cstdint>
#include <cuda_runtime.h>

#include "kkt_internal.cuh"
#include "kkt_test.h"

extern "C" int kkt_test_stalled_solve(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                                      int B, int T, int H, int dk, int dv, int C,
                                      float *T_out, void *W_out, void *U_out, struct CUstream_st *stream) {
    kkt::Problem p;
    int which = 0;
    bool empty = false;
    const int st = kkt::make_problem(k, v, beta, nullptr, cu_seqlens, B, T, H, dk, dv, C, T_out, W_out, U_out,
                                     KKT_IO_BF16, KKT_KERNEL_TC, stream, &p, &which, &empty);
    if (st != KKT_OK || empty) return st;
    p.tile_counter = nullptr;  // fixed round robin: no workspace needed
    p.stall_first_tile = 1;
    return kkt::launch_tc(p);
}
