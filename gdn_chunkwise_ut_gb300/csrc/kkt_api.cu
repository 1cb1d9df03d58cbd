// kkt_api.cu -- the C entry points of libkkt: argument checks, kernel choice,
// the per-device status word.  Declared in include/kkt.h.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "kkt_internal.cuh"

namespace {

// Per-device status word: first device-side error since the last
// kkt_device_status() (0 = none).
__device__ int g_kkt_status = 0;

// Device address of the status word, per device.  Host threads may fill an entry at the same time;
// they all store the same address, and the atomics make that well defined.  cudaDeviceReset
// invalidates the address (the module is loaded again by the next call's context), so calls after a
// reset of the device are not supported.
constexpr int kMaxDevices = 64;
std::atomic<int *> g_status_ptr[kMaxDevices] = {};

}  // namespace

namespace kkt {

int status_ptr(int **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KKT_ERR_NO_DEVICE;
    int *cached = g_status_ptr[dev].load(std::memory_order_relaxed);
    if (!cached) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_kkt_status) != cudaSuccess || ptr == nullptr) return KKT_ERR_CUDA;
        cached = static_cast<int *>(ptr);
        g_status_ptr[dev].store(cached, std::memory_order_relaxed);
    }
    *out = cached;
    return KKT_OK;
}

}  // namespace kkt

namespace {

#ifdef KKT_TRACE
void *g_trace = nullptr;
#endif

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool head_dim_ok(int d) { return d == 64 || d == 128; }
bool chunk_ok(int C) { return C == 32 || C == 64 || C == 128; }

}  // namespace

extern "C" int kkt_select_kernel(int dk, int dv, int C, int io_dtype, int kernel) {
    io_dtype &= ~KKT_T_OUT_F16;  // the T_out precision does not affect the choice
    if (io_dtype != KKT_IO_BF16 && io_dtype != KKT_IO_F32) return -KKT_ERR_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv) || !chunk_ok(C)) return -KKT_ERR_UNSUPPORTED;
    const bool tc = kkt::tc_supports(dk, dv, C, io_dtype);
    switch (kernel) {
        case KKT_KERNEL_AUTO: return tc ? KKT_KERNEL_TC : KKT_KERNEL_SIMT;
        case KKT_KERNEL_SIMT: return KKT_KERNEL_SIMT;
        case KKT_KERNEL_TC: return tc ? KKT_KERNEL_TC : -KKT_ERR_UNSUPPORTED;
        default: return -KKT_ERR_ARG;
    }
}

namespace kkt {

int make_problem(const void *k, const void *v, const float *beta, const float *g, const int32_t *cu_seqlens,
                 int B, int T, int H, int dk, int dv, int C, void *T_out, void *W_out, void *U_out,
                 int io_dtype, int kernel, struct CUstream_st *stream, Problem *p, int *which, bool *empty) {
    *empty = false;
    if (!k || !v || !beta || !W_out || !U_out) return KKT_ERR_ARG;  // T_out may be NULL
    if (B < 1 || T < 0 || H < 1 || H > 65535) return KKT_ERR_ARG;
    const int w = kkt_select_kernel(dk, dv, C, io_dtype, kernel);
    if (w < 0) return -w;
    if (!aligned16(k) || !aligned16(v) || !aligned16(T_out) || !aligned16(W_out) || !aligned16(U_out) ||
        !aligned4(beta) || (g && !aligned4(g)) || (cu_seqlens && !aligned4(cu_seqlens)))
        return KKT_ERR_ALIGN;
    const int64_t ntok = cu_seqlens ? (int64_t)T : (int64_t)B * T;
    if (ntok == 0) {
        *empty = true;
        return KKT_OK;
    }
    // the work-id space and every flat index must fit comfortably in 63 bits / grid limits
    if (ntok / C + B > 0x7fffffffLL) return KKT_ERR_ARG;

    p->k = k; p->v = v; p->beta = beta; p->g = g; p->cu_seqlens = cu_seqlens;
    p->nseq = B; p->T = T; p->ntok = ntok;
    p->H = H; p->dk = dk; p->dv = dv; p->C = C;
    p->T_out = T_out; p->W_out = W_out; p->U_out = U_out;
    p->io = io_dtype & ~KKT_T_OUT_F16;
    p->t_f16 = (io_dtype & KKT_T_OUT_F16) != 0;
    p->stream = reinterpret_cast<cudaStream_t>(stream);
#ifdef KKT_TRACE
    p->trace = g_trace;
#else
    p->trace = nullptr;
#endif
    p->tile_counter = nullptr;
    p->stall_first_tile = 0;
    *which = w;
    return status_ptr(&p->status);
}

}  // namespace kkt

namespace {

// kkt_solve_fwd_ex and kkt_solve_fwd_gated: g == nullptr is the ungated call.
int solve(const void *k, const void *v, const float *beta, const float *g, const int32_t *cu_seqlens,
          int B, int T, int H, int dk, int dv, int C, void *T_out, void *W_out, void *U_out,
          int io_dtype, int kernel, void *workspace, size_t workspace_bytes, struct CUstream_st *stream) {
    if (workspace && workspace_bytes < KKT_WORKSPACE_BYTES) return KKT_ERR_ARG;
    if (workspace && !aligned16(workspace)) return KKT_ERR_ALIGN;
    kkt::Problem p;
    int which = 0;
    bool empty = false;
    const int st = kkt::make_problem(k, v, beta, g, cu_seqlens, B, T, H, dk, dv, C, T_out, W_out, U_out,
                                     io_dtype, kernel, stream, &p, &which, &empty);
    if (st != KKT_OK || empty) return st;
    // the workspace is zero on entry (zero-filled before first use, and left zero by every call)
    if (which == KKT_KERNEL_TC && workspace) p.tile_counter = static_cast<unsigned long long *>(workspace);
    return which == KKT_KERNEL_TC ? kkt::launch_tc(p) : kkt::launch_simt(p);
}

}  // namespace

extern "C" int kkt_solve_fwd_ex(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                                int B, int T, int H, int dk, int dv, int C,
                                void *T_out, void *W_out, void *U_out,
                                int io_dtype, int kernel, void *workspace, size_t workspace_bytes,
                                struct CUstream_st *stream) {
    return solve(k, v, beta, nullptr, cu_seqlens, B, T, H, dk, dv, C, T_out, W_out, U_out, io_dtype, kernel,
                 workspace, workspace_bytes, stream);
}

extern "C" int kkt_solve_fwd_gated(const void *k, const void *v, const float *beta, const float *g,
                                   const int32_t *cu_seqlens, int B, int T, int H, int dk, int dv, int C,
                                   void *T_out, void *W_out, void *U_out,
                                   int io_dtype, int kernel, void *workspace, size_t workspace_bytes,
                                   struct CUstream_st *stream) {
    return solve(k, v, beta, g, cu_seqlens, B, T, H, dk, dv, C, T_out, W_out, U_out, io_dtype, kernel,
                 workspace, workspace_bytes, stream);
}

extern "C" int kkt_solve_fwd(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                             int B, int T, int H, int dk, int dv, int C,
                             float *T_out, void *W_out, void *U_out, struct CUstream_st *stream) {
    return kkt_solve_fwd_ex(k, v, beta, cu_seqlens, B, T, H, dk, dv, C, T_out, W_out, U_out,
                            KKT_IO_BF16, KKT_KERNEL_AUTO, nullptr, 0, stream);
}

extern "C" int kkt_device_status(struct CUstream_st *stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return KKT_ERR_CUDA;
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_kkt_status, sizeof(int)) != cudaSuccess) return KKT_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_kkt_status, &zero, sizeof(int)) != cudaSuccess) return KKT_ERR_CUDA;
    return value;
}

extern "C" const char *kkt_status_string(int status) {
    switch (status) {
        case KKT_OK: return "ok";
        case KKT_ERR_ARG: return "invalid argument";
        case KKT_ERR_UNSUPPORTED: return "unsupported chunk size, head dimension, dtype or kernel";
        case KKT_ERR_ALIGN: return "pointer misaligned (16 B for k, v, T_out, W_out, U_out; 4 B for beta, g, cu_seqlens)";
        case KKT_ERR_CUDA: return "CUDA error";
        case KKT_ERR_SEQLENS: return "malformed cu_seqlens";
        case KKT_ERR_TIMEOUT: return "device-side wait timed out";
        case KKT_ERR_NO_DEVICE: return "no usable CUDA device";
        default: return "unknown status";
    }
}

extern "C" int kkt_version(void) { return (0 << 16) | (1 << 8) | 0; }

extern "C" int kkt_debug_bounds(unsigned long long *first, int *kind) {
    constexpr int kFiles = 5;  // one record per kernel translation unit
    kkt::BoundsRecord rec[kFiles] = {};
    if (kkt::debug_bounds_tc(&rec[0]) < 0 || kkt::debug_bounds_tc_d64(&rec[1]) < 0 ||
        kkt::debug_bounds_tc_k128v64(&rec[2]) < 0 || kkt::debug_bounds_tc_k64v128(&rec[3]) < 0 ||
        kkt::debug_bounds_simt(&rec[4]) < 0)
        return -1;
    unsigned int total = 0;
    const kkt::BoundsRecord *f = nullptr;
    for (int i = 0; i < kFiles; ++i) {
        total += rec[i].count;
        if (!f && rec[i].count) f = &rec[i];
    }
    if (first) *first = f ? f->first : 0ull;
    if (kind) *kind = f ? (int)f->kind : 0;
    return (int)total;
}

#ifdef KKT_TRACE
// Trace builds only: device buffer of kTraceCtas x kTraceTiles x 16 uint64 time stamps
// (see trace.py), or NULL to stop tracing.
extern "C" void kkt_set_trace_buffer(void *buf) { g_trace = buf; }
#endif
