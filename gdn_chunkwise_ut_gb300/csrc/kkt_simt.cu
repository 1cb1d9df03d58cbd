// kkt_simt.cu -- one CTA per (chunk, head), fp32 CUDA-core arithmetic.
//
// The straightforward kernel: it serves fp32 I/O, every (C, dk, dv) the
// library accepts, and is the baseline the tcgen05 kernel is measured
// against.  It runs the same blocked schedule as the tensor-core kernel
// ("TileLang 实战：单位下三角矩阵求逆" §2.2): 16 x 16 diagonal blocks inverted
// by forward substitution (§2.1, one thread per column), then the coupling
// levels -L11^-1 L10 L00^-1 at s = 16, 32, ..., C/2 as shared-memory GEMMs.
//
// Shared memory (fp32): K [C][dk+1], V [C][dv+1], A/T [C][C+1], beta [C],
// gate prefix sums [C], coupling scratch [C/2][C/2+1].  The +1 row padding keeps the column walks of
// the Gram and epilogue loops on distinct banks.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kkt_debug.cuh"
#include "kkt_internal.cuh"

namespace kkt {
namespace {

constexpr int kSimtThreads = 256;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

struct SimtParams {
    const void *k, *v;
    const float *beta;
    const float *g;  // per-token log decays (gated variant), or nullptr
    const int32_t *cu;
    int nseq, T;
    int64_t ntok;
    int H, dk, dv;
    void *T_out;  // fp32, or fp16 with t_f16; nullptr: T is not written
    int t_f16;
    void *W_out, *U_out;
    int *status;
};

template <typename TIn, int C>
__global__ void __launch_bounds__(kSimtThreads) kkt_simt_kernel(const SimtParams p) {
    extern __shared__ float smem[];
    const int DK = p.dk, DV = p.dv;
    const int KS = DK + 1, VS = DV + 1;
    constexpr int TS = C + 1;
    float *Ks = smem;            // [C][KS]
    float *Vs = Ks + C * KS;     // [C][VS]
    float *Ts = Vs + C * VS;     // [C][TS]: A, overwritten in place by T, then by T diag(beta)
    float *bs = Ts + C * TS;     // [C]
    float *gs = bs + C;          // [C]: prefix sums G of the chunk's log decays (gated variant)
    float *Ys = gs + C;          // coupling scratch, up to (C/2) x (C/2 + 1)
    // element access of each array (range-checked in the bounds-checked debug build)
    auto K_ = [&](int64_t i) -> float & { return arr_at(Ks, i, (int64_t)C * KS); };
    auto V_ = [&](int64_t i) -> float & { return arr_at(Vs, i, (int64_t)C * VS); };
    auto T_ = [&](int64_t i) -> float & { return arr_at(Ts, i, (int64_t)C * TS); };
    auto B_ = [&](int64_t i) -> float & { return arr_at(bs, i, (int64_t)C); };
    auto G_ = [&](int64_t i) -> float & { return arr_at(gs, i, (int64_t)C); };
    auto Y_ = [&](int64_t i) -> float & { return arr_at(Ys, i, (int64_t)(C / 2) * (C / 2 + 1)); };

    const int64_t id = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    if (h == 0 && id < p.nseq && tid == 0) check_sequence(p.cu, (int)id, p.nseq, p.ntok, p.status);
    Chunk ch;
    if (!map_chunk(id, p.cu, p.nseq, p.T, p.ntok, C, p.status, ch)) return;
    const int Lc = ch.Lc;
    const int64_t t0 = ch.t0;
    const int64_t H = p.H;

    const TIn *kg = static_cast<const TIn *>(p.k);
    const TIn *vg = static_cast<const TIn *>(p.v);
    TIn *wg = static_cast<TIn *>(p.W_out);
    TIn *ug = static_cast<TIn *>(p.U_out);

    // 1. stage K, V, beta; rows >= Lc are zero
    for (int e = tid; e < C * DK; e += kSimtThreads) {
        const int i = e / DK, d = e - (e / DK) * DK;
        K_(i * KS + d) = (i < Lc) ? to_f(*gmem_chk(kg, ((t0 + i) * H + h) * DK + d, p.ntok * H * DK)) : 0.f;
    }
    for (int e = tid; e < C * DV; e += kSimtThreads) {
        const int i = e / DV, d = e - (e / DV) * DV;
        V_(i * VS + d) = (i < Lc) ? to_f(*gmem_chk(vg, ((t0 + i) * H + h) * DV + d, p.ntok * H * DV)) : 0.f;
    }
    for (int i = tid; i < C; i += kSimtThreads) B_(i) = (i < Lc) ? *gmem_chk(p.beta, (t0 + i) * H + h, p.ntok * H) : 0.f;
    if (p.g && tid == 0) {
        // G_i = g_0 + ... + g_i over the chunk's tokens, so that Gamma[i][j] = exp(G_i - G_j)
        float acc = 0.f;
        for (int i = 0; i < C; ++i) {
            acc += (i < Lc) ? *gmem_chk(p.g, (t0 + i) * H + h, p.ntok * H) : 0.f;
            G_(i) = acc;
        }
    }
    __syncthreads();

    // 2. A = I + strictLower(diag(beta) K K^T)   (§1; beta on rows, unit diagonal, §3.2), times
    //    Gamma elementwise in the gated variant (§5 item 12)
    for (int e = tid; e < C * C; e += kSimtThreads) {
        const int i = e / C, j = e % C;
        float a = 0.f;
        if (i == j) {
            a = 1.f;
        } else if (i > j) {
            float s = 0.f;
            for (int d = 0; d < DK; ++d) s = fmaf(K_(i * KS + d), K_(j * KS + d), s);
            a = B_(i) * s;
            if (p.g) a *= expf(G_(i) - G_(j));
        }
        T_(i * TS + j) = a;
    }
    __syncthreads();

    // 3. diagonal 16 x 16 blocks: X = L^-1 column by column (thread = block, column)
    //    X[r][c] = delta_rc - sum_{m<r} L[r][m] X[m][c]   (§2.1)
    constexpr int NB = C / 16;
    const bool sub = tid < NB * 16;
    const int b = tid >> 4, c = tid & 15;
    float x[16];
    const int64_t d0 = (int64_t)(16 * b) * TS + 16 * b;  // the diagonal block's first element
    if (sub) {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float s = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) s = fmaf(-T_(d0 + r * TS + m), x[m], s);
            x[r] = s;
        }
    }
    __syncthreads();  // every read of the block's L is done before it is overwritten
    if (sub) {
#pragma unroll
        for (int r = 1; r < 16; ++r)
            if (r > c) T_(d0 + r * TS + c) = x[r];
    }
    __syncthreads();

    // 4. coupling levels: lower block of each pair = -X11 (L10 X00)   (§2.2)
    for (int s = 16; s < C; s *= 2) {
        const int npairs = C / (2 * s);
        const int YS = s + 1;
        const int n = npairs * s * s;
        for (int e = tid; e < n; e += kSimtThreads) {
            const int pr = e / (s * s), r = (e / s) % s, cc = e % s;
            const int o = 2 * s * pr;
            float acc = 0.f;  // (L10 X00)[r][cc], L10 at rows o + s.., columns o..; X00 at (o, o)
            for (int m = cc; m < s; ++m)
                acc = fmaf(T_((int64_t)(o + s + r) * TS + o + m), T_((int64_t)(o + m) * TS + o + cc), acc);
            Y_(pr * s * YS + r * YS + cc) = acc;
        }
        __syncthreads();
        for (int e = tid; e < n; e += kSimtThreads) {
            const int pr = e / (s * s), r = (e / s) % s, cc = e % s;
            const int o = 2 * s * pr;
            float acc = 0.f;  // (X11 Y)[r][cc], X11 at (o + s, o + s)
            for (int m = 0; m <= r; ++m)
                acc = fmaf(T_((int64_t)(o + s + r) * TS + o + s + m), Y_(pr * s * YS + m * YS + cc), acc);
            T_((int64_t)(o + s + r) * TS + o + cc) = -acc;
        }
        __syncthreads();
    }

    // 5. T_out rows of the chunk (zeros in columns >= Lc); none without T_out (W and U~ only)
    for (int e = tid; p.T_out && e < Lc * C; e += kSimtThreads) {
        const int i = e / C, j = e % C;
        const float x = (j < Lc) ? T_(i * TS + j) : 0.f;
        const int64_t at = ((t0 + i) * H + h) * C + j;
        if (p.t_f16)
            *gmem_chk(static_cast<__half *>(p.T_out), at, p.ntok * H * C) = __float2half_rn(x);
        else
            *gmem_chk(static_cast<float *>(p.T_out), at, p.ntok * H * C) = x;
    }
    __syncthreads();

    // 6. T~ = T diag(beta), in place.  Gated: the keys of W carry the decay from the chunk's start
    //    through their own token, W = T diag(beta) diag(e^G) K, so K's rows are scaled by e^{G_j}
    //    (the Gram no longer needs them)
    for (int e = tid; e < C * C; e += kSimtThreads) {
        const int i = e / C, j = e % C;
        T_(i * TS + j) *= B_(j);
    }
    if (p.g) {
        for (int e = tid; e < C * DK; e += kSimtThreads) {
            const int j = e / DK, d = e - (e / DK) * DK;
            K_(j * KS + d) *= expf(G_(j));
        }
    }
    __syncthreads();

    // 7. W = T~ K, U~ = T~ V   (§1); T~ is lower triangular, so j <= i
    for (int e = tid; e < Lc * DK; e += kSimtThreads) {
        const int i = e / DK, d = e - (e / DK) * DK;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc = fmaf(T_(i * TS + j), K_(j * KS + d), acc);
        *gmem_chk(wg, ((t0 + i) * H + h) * DK + d, p.ntok * H * DK) = from_f<TIn>(acc);
    }
    for (int e = tid; e < Lc * DV; e += kSimtThreads) {
        const int i = e / DV, d = e - (e / DV) * DV;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc = fmaf(T_(i * TS + j), V_(j * VS + d), acc);
        *gmem_chk(ug, ((t0 + i) * H + h) * DV + d, p.ntok * H * DV) = from_f<TIn>(acc);
    }
}

template <typename TIn, int C>
int launch_simt_t(const Problem &pb) {
    const size_t smem = sizeof(float) * ((size_t)C * (pb.dk + 1) + (size_t)C * (pb.dv + 1) +
                                         (size_t)C * (C + 1) + 2 * C + (size_t)(C / 2) * (C / 2 + 1));
    auto kern = kkt_simt_kernel<TIn, C>;
    // the limit is raised once, to the size at d_k = d_v = 128, the largest head dimension
    constexpr size_t kMaxSmem = sizeof(float) * ((size_t)C * 129 * 2 + (size_t)C * (C + 1) + 2 * C +
                                                 (size_t)(C / 2) * (C / 2 + 1));
    static_assert(kMaxSmem <= 232448, "SIMT shared memory over the per-block limit");
    if (smem > kMaxSmem || !ensure_max_smem<kkt_simt_kernel<TIn, C>>((int)kMaxSmem)) return KKT_ERR_CUDA;
    SimtParams p;
    p.k = pb.k; p.v = pb.v; p.beta = pb.beta; p.g = pb.g; p.cu = pb.cu_seqlens;
    p.nseq = pb.nseq; p.T = pb.T; p.ntok = pb.ntok;
    p.H = pb.H; p.dk = pb.dk; p.dv = pb.dv;
    p.T_out = pb.T_out; p.t_f16 = pb.t_f16; p.W_out = pb.W_out; p.U_out = pb.U_out; p.status = pb.status;
    const int64_t ids = total_work_ids(pb.ntok, C, pb.nseq);
    dim3 grid((unsigned)ids, (unsigned)pb.H);
    kern<<<grid, kSimtThreads, smem, pb.stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? KKT_OK : KKT_ERR_CUDA;
}

template <typename TIn>
int dispatch_c(const Problem &p) {
    switch (p.C) {
        case 32: return launch_simt_t<TIn, 32>(p);
        case 64: return launch_simt_t<TIn, 64>(p);
        case 128: return launch_simt_t<TIn, 128>(p);
        default: return KKT_ERR_UNSUPPORTED;
    }
}

}  // namespace

int debug_bounds_simt(BoundsRecord *out) { return read_bounds_record(out); }

int launch_simt(const Problem &p) {
    return p.io == KKT_IO_F32 ? dispatch_c<float>(p) : dispatch_c<__nv_bfloat16>(p);
}

}  // namespace kkt
