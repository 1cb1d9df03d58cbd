// kkt_debug.cuh -- range checks of the bounds-checked debug build (-DKKT_DEBUG_BOUNDS).
//
// compute-sanitizer is not available where this library is tested, so the debug build checks
// the kernels' own index arithmetic instead.  Every shared-memory access of the tensor-core
// kernel goes through smem_chk (the address range must lie inside the block's dynamic shared
// memory), every array access of the SIMT kernel through arr_at (the index must lie inside its
// array), and every plain global store or load through gmem_chk (the element index must lie
// inside the tensor).  A failed check counts a violation, records the first offending address or
// index, and redirects the access to a scratch location, so the kernel runs to its end without a
// fault or a trap.  kkt_debug_bounds() (kkt_test.h) reads and clears the records.  In the default
// build every helper is the identity and costs nothing.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kkt_internal.cuh"

namespace kkt {

#ifdef KKT_DEBUG_BOUNDS

namespace {

// one record per translation unit (kernel file); read by that file's debug_bounds_* function
__device__ BoundsRecord g_kkt_bounds;
__device__ __align__(16) unsigned char g_kkt_bounds_scratch[64];

// Copies and clears this translation unit's record (host).
int read_bounds_record(BoundsRecord *out) {
    if (cudaMemcpyFromSymbol(out, g_kkt_bounds, sizeof(BoundsRecord)) != cudaSuccess) return -1;
    const BoundsRecord zero = {0u, 0u, 0ull};
    if (cudaMemcpyToSymbol(g_kkt_bounds, &zero, sizeof(BoundsRecord)) != cudaSuccess) return -1;
    return 0;
}

}  // namespace

__device__ __forceinline__ void bounds_violation(unsigned int kind, unsigned long long what) {
    if (atomicAdd(&g_kkt_bounds.count, 1u) == 0u) {
        g_kkt_bounds.kind = kind;
        g_kkt_bounds.first = what;
    }
}

__device__ __forceinline__ uint32_t dyn_smem_size() {
    uint32_t s;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(s));
    return s;
}

// [p, p + sizeof(T)) inside this block's dynamic shared memory, else a scratch slot.
template <typename T>
__device__ __forceinline__ T *smem_chk(T *p) {
    extern __shared__ __align__(16) uint8_t kkt_dyn_smem_base[];
    __shared__ __align__(16) uint8_t scratch[64];
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(kkt_dyn_smem_base));
    if (a < base || a + (uint32_t)sizeof(T) > base + dyn_smem_size()) {
        bounds_violation(1u, a);
        return reinterpret_cast<T *>(scratch);
    }
    return p;
}

// arr[i] with 0 <= i < n, else a scratch slot.
template <typename T>
__device__ __forceinline__ T &arr_at(T *arr, int64_t i, int64_t n) {
    __shared__ __align__(16) uint8_t scratch[64];
    if (i < 0 || i >= n) {
        bounds_violation(2u, (unsigned long long)i);
        return *reinterpret_cast<T *>(scratch);
    }
    return arr[i];
}

// base + i with 0 <= i and i + width <= n (elements), else a global scratch slot.
template <typename T>
__device__ __forceinline__ T *gmem_chk(T *base, int64_t i, int64_t n, int64_t width = 1) {
    if (i < 0 || i + width > n) {
        bounds_violation(3u, (unsigned long long)i);
        return reinterpret_cast<T *>(g_kkt_bounds_scratch);
    }
    return base + i;
}

#else

namespace {
int read_bounds_record(BoundsRecord *) { return -1; }  // not a bounds-checked build
}  // namespace

template <typename T>
__device__ __forceinline__ T *smem_chk(T *p) { return p; }
template <typename T>
__device__ __forceinline__ T &arr_at(T *arr, int64_t i, int64_t) { return arr[i]; }
template <typename T>
__device__ __forceinline__ T *gmem_chk(T *base, int64_t i, int64_t, int64_t = 1) { return base + i; }

#endif

}  // namespace kkt
