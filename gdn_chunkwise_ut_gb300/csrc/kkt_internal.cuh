// kkt_internal.cuh -- shared host/device definitions of libkkt (not installed).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "kkt.h"

namespace kkt {

// Raises a kernel's dynamic shared-memory limit to `bytes` once per device (the setting persists in
// the context), so that a call makes no such runtime call after the first, and calls made while a
// stream is being captured into a CUDA graph launch only.
template <auto Kern>
inline bool ensure_max_smem(int bytes) {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const unsigned long long bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return true;
    if (cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    done.fetch_or(bit, std::memory_order_acq_rel);
    return true;
}

// Everything a launcher needs, validated by the C entry points.
struct Problem {
    const void *k;
    const void *v;
    const float *beta;
    const float *g = nullptr;   // per-token log decays of the gated variant, or nullptr
    const int32_t *cu_seqlens;  // nullptr: nseq sequences of T tokens each
    int nseq;                   // number of sequences (B)
    int T;                      // tokens per sequence, or the packed total with cu_seqlens
    int64_t ntok;               // rows of the flat token axis (B*T, or T with cu_seqlens)
    int H, dk, dv, C;
    void *T_out;                // fp32, or fp16 with t_f16; nullptr: T is not written
    void *W_out;
    void *U_out;
    int io;                     // KKT_IO_BF16 / KKT_IO_F32
    int t_f16 = 0;              // T_out holds fp16
    cudaStream_t stream;
    int *status;                // device status word of the current device
    void *trace;                // pipeline trace buffer (KKT_TRACE builds only), else nullptr
    unsigned long long *tile_counter;  // zeroed work counter for dynamic scheduling, or nullptr
    int stall_first_tile = 0;   // test hook: the tensor-core kernel never fills its first stage
};

// Device-side error codes (first error wins); a null status records nothing.
__device__ __forceinline__ void record_error(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Work ids and chunks.  Sequence s owns the ids [Q(s), Q(s+1)) with
// Q(s) = floor(start(s) / C) + s.  Q is strictly increasing for nondecreasing
// starts, and a sequence of L tokens starting at a gets
// floor((a mod C + L) / C) + 1 >= ceil(L / C) ids, so every chunk has an id;
// the surplus ids (at most one per sequence) are idle.  Total ids:
// Q(nseq) = floor(ntok / C) + nseq.  No host-side pass over cu_seqlens and no
// device scratch table are needed.
struct Chunk {
    int64_t t0;  // first row in the flat token axis
    int Lc;      // rows in this chunk, 1..C
};

__device__ __forceinline__ int64_t seq_start(const int32_t *cu, int s, int T) {
    return cu ? (int64_t)__ldg(cu + s) : (int64_t)s * T;
}

__host__ __device__ __forceinline__ int64_t total_work_ids(int64_t ntok, int C, int nseq) {
    return ntok / C + nseq;
}

// Maps a work id to its chunk.  Returns false for idle ids and for ids whose
// sequence bounds are malformed (recorded as KKT_ERR_SEQLENS); never touches
// memory outside cu_seqlens[0..nseq].
__device__ __forceinline__ bool map_chunk(int64_t id, const int32_t *cu, int nseq, int T, int64_t ntok,
                                          int C, int *status, Chunk &out) {
    int lo = 0, hi = nseq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int64_t q = seq_start(cu, mid, T) / C + mid;
        if (q <= id) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int64_t a = seq_start(cu, s, T);
    const int64_t b = seq_start(cu, s + 1, T);
    if (a < 0 || b < a || b > ntok) {
        record_error(status, KKT_ERR_SEQLENS);
        return false;
    }
    const int64_t c = id - (a / C + s);
    if (c < 0) {
        record_error(status, KKT_ERR_SEQLENS);
        return false;
    }
    const int64_t t0 = a + c * C;
    if (t0 >= b) return false;
    out.t0 = t0;
    out.Lc = (int)((b - t0) < C ? (b - t0) : C);
    return true;
}

// Checks the global shape of cu_seqlens for sequence s (called once per s).
__device__ __forceinline__ void check_sequence(const int32_t *cu, int s, int nseq, int64_t ntok, int *status) {
    if (!cu) return;
    const int64_t a = __ldg(cu + s), b = __ldg(cu + s + 1);
    bool bad = (a < 0) || (b < a) || (b > ntok);
    if (s == 0 && a != 0) bad = true;
    if (s == nseq - 1 && b != ntok) bad = true;
    if (bad) record_error(status, KKT_ERR_SEQLENS);
}

// Address of the current device's status word (looked up once per device).
int status_ptr(int **out);

// The argument checks every entry point shares.  Validates the call, chooses the kernel (*which,
// KKT_KERNEL_SIMT or KKT_KERNEL_TC) and fills every field of *p except the schedule (tile_counter,
// left null) and the test hook.  Returns KKT_OK or the status the entry point returns without
// launching; *empty is set when the call has no tokens (valid, nothing to launch).
int make_problem(const void *k, const void *v, const float *beta, const float *g, const int32_t *cu_seqlens,
                 int B, int T, int H, int dk, int dv, int C, void *T_out, void *W_out, void *U_out,
                 int io_dtype, int kernel, struct CUstream_st *stream, Problem *p, int *which, bool *empty);

int launch_simt(const Problem &p);
int launch_tc(const Problem &p);

// Bounds-checked debug builds (-DKKT_DEBUG_BOUNDS, kkt_debug.cuh): violation count, kind of the
// first (1 shared memory, 2 array index, 3 global index) and its shared address or index.  Each
// kernel file reads and clears its own record; -1 in the default build.
struct BoundsRecord {
    unsigned int count;
    unsigned int kind;
    unsigned long long first;
};
int debug_bounds_tc(BoundsRecord *out);
int debug_bounds_tc_d64(BoundsRecord *out);
int debug_bounds_tc_k128v64(BoundsRecord *out);
int debug_bounds_tc_k64v128(BoundsRecord *out);
int debug_bounds_simt(BoundsRecord *out);
bool tc_supports(int dk, int dv, int C, int io);

}  // namespace kkt
