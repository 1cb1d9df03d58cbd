// kkt_noalloc.cu -- kkt_solve for callers that cannot allocate device memory.
//
// The tensor-core kernel hands out work through a tile counter that lives in
// scratch memory.  kkt_solve_fwd_ex takes that scratch from the caller; this
// entry point instead uses a small array compiled into the library, so the
// call needs no buffer beyond the inputs and outputs and allocates nothing.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "kkt_internal.cuh"
#include "kkt_test.h"

namespace {

// The scratch of kkt_solve_fwd_noalloc: one array per device, held by every GPU
// that loads the library until the process exits.  A call uses its first 16
// bytes (the tile counter and the count of CTAs done claiming).
__device__ __align__(256) unsigned char g_noalloc_scratch[KKT_NOALLOC_SCRATCH_BYTES];

// Bytes of scratch one call uses: two 64-bit counters, the same for every problem size.
constexpr size_t kNoallocNeed = 2 * sizeof(unsigned long long);
static_assert(kNoallocNeed <= KKT_NOALLOC_SCRATCH_BYTES, "scratch array too small");

// Device address of the array, per device.  Host threads may fill an entry at the same time;
// they all store the same address, and the atomics make that well defined.  cudaDeviceReset
// invalidates the address, so calls after a reset of the device are not supported.
constexpr int kMaxDevices = 64;
std::atomic<unsigned long long *> g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device, with that device current.
int noalloc_scratch(unsigned long long **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KKT_ERR_NO_DEVICE;
    unsigned long long *cached = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
    if (!cached) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return KKT_ERR_CUDA;
        cached = static_cast<unsigned long long *>(ptr);
        g_noalloc_ptr[dev].store(cached, std::memory_order_relaxed);
    }
    *out = cached;
    return KKT_OK;
}

}  // namespace

extern "C" int kkt_solve_fwd_noalloc(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                                     int B, int T, int H, int dk, int dv, int C,
                                     float *T_out, void *W_out, void *U_out, struct CUstream_st *stream) {
    // only the tensor-core kernel uses scratch; shapes it does not cover are rejected
    kkt::Problem p;
    int which = 0;
    bool empty = false;
    int st = kkt::make_problem(k, v, beta, nullptr, cu_seqlens, B, T, H, dk, dv, C, T_out, W_out, U_out,
                               KKT_IO_BF16, KKT_KERNEL_TC, stream, &p, &which, &empty);
    if (st != KKT_OK || empty) return st;
    st = noalloc_scratch(&p.tile_counter);
    if (st != KKT_OK) return st;
    // Clear the counters on the stream before the launch.  Each kernel's last CTA also leaves them
    // zero, but a call that overlapped another one on the GPU, or whose kernel gave up on a timeout,
    // may not have; the clear keeps such a call from spoiling the calls after it.
    if (cudaMemsetAsync(p.tile_counter, 0, kNoallocNeed, p.stream) != cudaSuccess) return KKT_ERR_CUDA;
    return kkt::launch_tc(p);
}

// Test hook (kkt_test.h): the first two 64-bit words of the scratch array on the current device.
extern "C" int kkt_test_noalloc_scratch(unsigned long long *out2) {
    if (!out2) return KKT_ERR_ARG;
    if (cudaMemcpyFromSymbol(out2, g_noalloc_scratch, kNoallocNeed) != cudaSuccess) return KKT_ERR_CUDA;
    return KKT_OK;
}
