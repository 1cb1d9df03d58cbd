// kkt_noalloc.cu -- kkt_solve for callers that cannot allocate device memory.
//
// The tensor-core kernel hands out work through a tile counter that lives in
// scratch memory.  kkt_solve_fwd_ex takes that scratch from the caller; this
// entry point instead uses a small array compiled into the library, so the
// call needs no buffer beyond the inputs and outputs and allocates nothing.
#include <cstdint>
#include <cuda_runtime.h>

#include "kkt_internal.cuh"

namespace {

// The scratch of kkt_solve_fwd_noalloc: one array per device, held by every GPU
// that loads the library until the process exits.  A call uses its first 16
// bytes (the tile counter and the count of CTAs done claiming): zero when the
// module loads, and left zero by every call's kernel.
__device__ __align__(256) unsigned char g_noalloc_scratch[KKT_NOALLOC_SCRATCH_BYTES];

// Bytes of scratch one call needs: two 64-bit counters, whatever the problem size.
constexpr size_t kNoallocNeed = 2 * sizeof(unsigned long long);
static_assert(kNoallocNeed <= KKT_NOALLOC_SCRATCH_BYTES, "scratch array too small");

constexpr int kMaxDevices = 64;
unsigned long long *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device, with that device current.
int noalloc_scratch(unsigned long long **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KKT_ERR_NO_DEVICE;
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return KKT_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<unsigned long long *>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return KKT_OK;
}

bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int kkt_solve_fwd_noalloc(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                                     int B, int T, int H, int dk, int dv, int C,
                                     float *T_out, void *W_out, void *U_out, struct CUstream_st *stream) {
    if (!k || !v || !beta || !W_out || !U_out) return KKT_ERR_ARG;  // T_out may be NULL
    if (B < 1 || T < 0 || H < 1 || H > 65535) return KKT_ERR_ARG;
    // only the tensor-core kernel uses scratch; shapes it does not cover are rejected
    const int which = kkt_select_kernel(dk, dv, C, KKT_IO_BF16, KKT_KERNEL_TC);
    if (which < 0) return -which;
    if (!aligned_to(k, 16) || !aligned_to(v, 16) || !aligned_to(T_out, 16) || !aligned_to(W_out, 16) ||
        !aligned_to(U_out, 16) || !aligned_to(beta, 4) || (cu_seqlens && !aligned_to(cu_seqlens, 4)))
        return KKT_ERR_ALIGN;
    const int64_t ntok = cu_seqlens ? (int64_t)T : (int64_t)B * T;
    if (ntok == 0) return KKT_OK;
    if (ntok / C + B > 0x7fffffffLL) return KKT_ERR_ARG;
    if (kNoallocNeed > KKT_NOALLOC_SCRATCH_BYTES) return KKT_ERR_ARG;  // the problem would need more scratch

    kkt::Problem p;
    p.k = k; p.v = v; p.beta = beta; p.cu_seqlens = cu_seqlens;
    p.nseq = B; p.T = T; p.ntok = ntok;
    p.H = H; p.dk = dk; p.dv = dv; p.C = C;
    p.T_out = T_out; p.W_out = W_out; p.U_out = U_out;
    p.io = KKT_IO_BF16;
    p.stream = reinterpret_cast<cudaStream_t>(stream);
    p.trace = nullptr;
    int st = kkt::status_ptr(&p.status);
    if (st != KKT_OK) return st;
    st = noalloc_scratch(&p.tile_counter);
    if (st != KKT_OK) return st;
    // the counters start at zero: zero-initialised with the module, and cleared by the last CTA of
    // every earlier call
    return kkt::launch_tc(p);
}
