// gdn_chunk.cu -- the chunk state recurrence and output of Gated DeltaNet chunked prefill: the
// computation that consumes kkt_solve's W and U~ (the FlashQLA page, "Tilelang Warp-Specialized
// Kernel", forward: V', S and O per chunk).  Entry point gdn_chunk_state_fwd (include/kkt.h).
//
// Per sequence and head the state S (d_k x d_v, fp32) runs over the sequence's chunks of C tokens
// (the chunks of kkt_solve), with G_i the gate's decay from the chunk's start through token i (log
// units; 0 without a gate) and Gamma[i][j] = e^{G_i - G_j}:
//     V' = U~ - W S
//     O  = scale (diag(e^G) Q S + (Gamma o tril(Q K^T)) V')          (the diagonal included)
//     S <- e^{G_last} S + (diag(e^{G_last - G}) K)^T V'
// W carries the decay e^{G_j} in its keys (kkt_solve's gated W), so V' row i is beta_i times token
// i's correction v_i - alpha_i S_{i-1}^T k_i of the delta rule.
//
// One CTA per (sequence, head); C = 64, d_k = d_v = 128.  Warps 0-3 ("math") own tensor-memory
// lanes 0-127, thread t holding row t of every tensor-memory matrix; warp 4 loads.
//   tensor memory (512 columns): S^T [128 x 128] fp32 (row e of S^T, i.e. column e of S, in lane e);
//   two D buffers [128 x 192] fp32.
//   shared memory: a two-deep ring of stages, each holding [Q; W] (per 64-column box: the 64 rows of
//   Q, then the 64 rows of W, so that the pair is one 128-row operand) and [S^T_b; K] (per box: the
//   128 rows of the bf16 copy of S^T, written by the math threads, then the 64 rows of K), Q, W and K
//   loaded by TMA with the 128-byte swizzle; the bf16 copies P_b of the masked P (rows 64..127
//   zero), V'_b of V' and, gated, VF_b of diag(e^{G_last - G}) V'; a one-chunk buffer of U~ (TMA,
//   prefetched into L2 a chunk earlier), refilled as soon as the V' warps have read it.
// Per chunk, every tcgen05.mma M = 128:
//   D   = [Q; W] [S^T_b; K]^T   (N = 192: columns 0..127 are [Q S; W S], 128..191 [Q K^T; W K^T])
//   S^T += V'(F)_b^T K          (A = V'^T and B = K both read MN-major, N = 128, K = 64 tokens)
//   D  += [P_b; 0] V'_b         (columns 0..127, rows 0..63 become O / scale)
// The first two are issued by thread 64, whose warps wait for D anyway, the third by thread 0, so that
// the state's chain (S^T -> S^T_b, D, V', the S^T update) does not wait for the output side's
// instructions (P, P V', the drain of O), which run on warps 0-1 and hold their lanes for the next
// S^T readback.
// The math threads between the products: S^T row -> S^T_b (and, gated, S^T <- e^{G_last} S^T in
// place); rows 64..127: W S row -> V' = U~ - W S -> V'_b (and VF_b); rows 0..63: P row -> causal mask
// (times Gamma when gated) -> P_b, gated Q S row -> e^{G_i} Q S, and O row -> scale -> bf16 -> global.
// The two D buffers let the O of one chunk drain while the next chunk's products run.
//
// Every wait is bounded (2 s); on expiry the kernel records KKT_ERR_TIMEOUT, stops, waits for its
// own copies and tensor-core work, frees tensor memory and returns.  Group syncs are mbarrier-based.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kkt_internal.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace kkt {
namespace {

using namespace ptx;

constexpr int kGcC = 64;
constexpr int kGcD = 128;                 // d_k = d_v
constexpr int kGcThreads = 320;           // warps 0-7 math, warp 8 loads, warp 9 issues the MMAs
constexpr uint32_t kGcTmemCols = 512;
constexpr uint32_t kColS = 0;             // S^T: 128 columns
constexpr uint32_t kColD0 = 128;          // D buffers: 192 columns each
constexpr uint32_t kColD1 = 320;
constexpr uint32_t kColDP = 128;          // the P columns inside a D buffer
constexpr uint64_t kGcWaitNs = 2000000000ull;

// shared memory, from a 1024-byte-aligned base
constexpr int kStageBytes = 81920;        // [Q; W] 32 KB, [S^T_b; K] 48 KB
constexpr int kOffQW = 0;                 // 2 boxes x [128 rows][128 B]
constexpr int kOffSK = 32768;             // 2 boxes x [192 rows][128 B]: S^T_b rows 0..127, K rows 128..191
constexpr int kBoxSK = 24576;
constexpr int kOffKInBox = 16384;
constexpr int kOffPb = 2 * kStageBytes;   // [128 rows][128 B]
constexpr int kOffVb = kOffPb + 16384;    // 2 boxes x [64 rows][128 B]
constexpr int kOffVf = kOffVb + 16384;
constexpr int kOffU = kOffVf + 16384;     // U~ of one chunk: 2 boxes x [64 rows][128 B]
constexpr int kOffMeta = kOffU + 16384;   // per stage 512 B: G[64] (log2 units), then the chunk info
constexpr int kOffBar = kOffMeta + 1024;
constexpr int kGcSmem = kOffBar + 256 + 1024;  // + alignment slack
static_assert(kGcSmem <= 232448, "shared memory over the per-block limit");
constexpr uint32_t kStageTx = 49152;      // Q, W and K boxes of one stage

struct GcInfo {
    int64_t t0;
    int Lc;
    int pad;
};

struct GcBars {
    uint64_t full[2], empty[2];
    uint64_t bar_d, bar_s, bar_o;
    uint64_t sb_ready, v_ready, p_ready;  // the math warps' operands are in shared memory
    uint64_t u_full, u_empty;             // the U~ buffer (one chunk)
    uint64_t grp128, fin;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(GcBars) <= 256, "barrier block");

struct GcParams {
    const float *g;        // per-token log decays, or nullptr
    const float *h0;       // [nseq][H][128][128] initial state, or nullptr (zero)
    float *ht;             // [nseq][H][128][128] final state, or nullptr
    const int32_t *cu;     // nullptr: nseq sequences of T tokens
    int nseq, T;
    int64_t ntok;
    int H;
    float scale;
    const __nv_bfloat16 *u;
    __nv_bfloat16 *o;
    int *status;
    unsigned long long *trace;  // KKT_TRACE builds: per-chunk time stamps of the first CTAs, else nullptr
};

// Pipeline trace (builds with -DKKT_TRACE only): SM cycle counter at each event of the first chunks of the
// first CTAs, [cta][chunk][event].
#ifdef KKT_TRACE
constexpr int kGcTraceCtas = 4, kGcTraceChunks = 64, kGcTraceEvents = 16;
#define GC_TRACE(ev, c)                                                                                   \
    do {                                                                                                  \
        if (p.trace && blockIdx.x < kGcTraceCtas && (c) < kGcTraceChunks)                                 \
            p.trace[((size_t)blockIdx.x * kGcTraceChunks + (c)) * kGcTraceEvents + (ev)] = clock64();     \
    } while (0)
#else
#define GC_TRACE(ev, c) \
    do {                \
    } while (0)
#endif

__device__ __forceinline__ uint8_t *align1024_gc(uint8_t *p) {
    const uint32_t a = smem_u32(p);
    return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack2_bf16(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}

// 16-byte chunk e (0..7) of row r of a 128-byte-swizzled box (TMA and UMMA layout).
__device__ __forceinline__ uint4 *sw_chunk(uint8_t *box, int r, int e) {
    return reinterpret_cast<uint4 *>(box + r * 128 + ((e ^ (r & 7)) << 4));
}

// 2^x by the hardware's approximation (about 22 correct bits): enough for factors that multiply values
// rounded to bf16 right after.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ bool gc_wait(uint64_t *bar, uint32_t parity, GcBars *bars, int *status) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, &bars->abort_flag, kGcWaitNs));
    if (!ok && atomicExch(&bars->abort_flag, 1) == 0) record_error(status, KKT_ERR_TIMEOUT);
    return ok;
}

// Bounded group barrier of `warps` whole warps: lane 0 of each arrives, then all wait for the phase.
__device__ __forceinline__ bool gc_group(uint64_t *bar, uint32_t &uses, GcBars *bars, int *status) {
    __syncwarp();
    if ((threadIdx.x & 31u) == 0u) mbar_arrive(bar);
    const bool ok = gc_wait(bar, uses & 1u, bars, status);
    ++uses;
    return ok;
}

// Loads 32 x N consecutive tensor-memory columns of the calling warp's lanes with N loads in flight, then
// waits once.
template <int N>
__device__ __forceinline__ void tmem_ld32xN(uint32_t taddr, uint32_t (&v)[N][32]) {
#pragma unroll
    for (int i = 0; i < N; ++i) tmem_ld32(taddr + 32 * i, v[i]);
    tmem_wait_ld();
}

template <bool GATED>
__global__ void __launch_bounds__(kGcThreads, 1)
    gdn_chunk_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_u,
                     const GcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024_gc(smem_raw);
    GcBars *bars = reinterpret_cast<GcBars *>(smem + kOffBar);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const int seq = blockIdx.x / p.H;
    const int h = blockIdx.x % p.H;

    auto stage = [&](int s) { return smem + s * kStageBytes; };
    auto stage_G = [&](int s) { return reinterpret_cast<float *>(smem + kOffMeta + s * 512); };
    auto stage_info = [&](int s) { return reinterpret_cast<GcInfo *>(smem + kOffMeta + s * 512 + 256); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->full[s], 2);  // the TMA transaction arrival, then one after the gate data
            // free again once the S^T update has read K (a tensor-core commit) and the four output warps
            // have read the gate data: the two sides run a chunk apart
            mbar_init(&bars->empty[s], 5);
        }
        mbar_init(&bars->bar_d, 1);
        mbar_init(&bars->bar_s, 1);
        mbar_init(&bars->bar_o, 1);
        mbar_init(&bars->sb_ready, 8);
        mbar_init(&bars->v_ready, 4);
        mbar_init(&bars->p_ready, 4);
        mbar_init(&bars->grp128, 8);
        mbar_init(&bars->u_full, 1);
        mbar_init(&bars->u_empty, 4);
        mbar_init(&bars->fin, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem_base, kGcTmemCols);
        tmem_relinquish();
    }
    // rows 64..127 of P_b: the lower half of the A operand [P; 0] of the PV product
    for (int e = threadIdx.x; e < 64 * 8; e += kGcThreads)
        *reinterpret_cast<uint4 *>(smem + kOffPb + 8192 + 16 * e) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    griddep_launch_dependents();
    griddep_wait();

    // this CTA's sequence
    const int64_t a = p.cu ? (int64_t)__ldg(p.cu + seq) : (int64_t)seq * p.T;
    const int64_t b = p.cu ? (int64_t)__ldg(p.cu + seq + 1) : (int64_t)(seq + 1) * p.T;
    bool seq_ok = a >= 0 && b >= a && b <= p.ntok;
    if (p.cu && ((seq == 0 && a != 0) || (seq == p.nseq - 1 && b != p.ntok))) seq_ok = false;
    if (!seq_ok && threadIdx.x == 0 && h == 0) record_error(p.status, KKT_ERR_SEQLENS);
    const int nchunks = seq_ok ? (int)((b - a + kGcC - 1) / kGcC) : 0;

    if (warp == 8) {
        // ------------------------------------------------------------------ loads
        if (lane == 0) {
            prefetch_tmap(&map_q);
            prefetch_tmap(&map_k);
            prefetch_tmap(&map_w);
            prefetch_tmap(&map_u);
            if (nchunks > 0) {  // U~ rows of the first chunk into L2
                tma_prefetch_3d(&map_u, 0, h, (int)a);
                tma_prefetch_3d(&map_u, 64, h, (int)a);
            }
        }
        int c = 0;
        bool ok = true;
        for (; c < nchunks; ++c) {
            const int s = c & 1;
            const int64_t t0 = a + (int64_t)kGcC * c;
            const int Lc = (int)((b - t0) < kGcC ? (b - t0) : kGcC);
            // the gate's log decays (log2 units), loaded before the wait for the stage
            constexpr float kLog2e = 1.4426950408889634f;
            float g0 = 0.f, g1 = 0.f;
            if constexpr (GATED) {
                if (lane < Lc) g0 = kLog2e * __ldg(p.g + (t0 + lane) * p.H + h);
                if (lane + 32 < Lc) g1 = kLog2e * __ldg(p.g + (t0 + lane + 32) * p.H + h);
            }
            if (!gc_wait(&bars->empty[s], (((uint32_t)c >> 1) & 1u) ^ 1u, bars, p.status)) { ok = false; break; }
            if (lane == 0) {
                GC_TRACE(10, c);
                GcInfo *info = stage_info(s);
                info->t0 = t0;
                info->Lc = Lc;
                uint8_t *st = stage(s);
                mbar_arrive_expect_tx(&bars->full[s], kStageTx);
                for (int c2 = 0; c2 < 2; ++c2) {
                    tma_load_3d(st + kOffQW + c2 * 16384, &map_q, &bars->full[s], 64 * c2, h, (int)t0);
                    tma_load_3d(st + kOffQW + c2 * 16384 + 8192, &map_w, &bars->full[s], 64 * c2, h, (int)t0);
                    tma_load_3d(st + kOffSK + c2 * kBoxSK + kOffKInBox, &map_k, &bars->full[s], 64 * c2, h,
                                (int)t0);
                }
                if (c + 1 < nchunks) {  // the next chunk's U~ rows into L2
                    tma_prefetch_3d(&map_u, 0, h, (int)(t0 + kGcC));
                    tma_prefetch_3d(&map_u, 64, h, (int)(t0 + kGcC));
                }
            }
            // this chunk's U~ into the one-chunk buffer once the V' warps are done with the previous one
            if (c > 0 && !gc_wait(&bars->u_empty, ((uint32_t)c - 1u) & 1u, bars, p.status)) { ok = false; break; }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->u_full, 16384);
                tma_load_3d(smem + kOffU, &map_u, &bars->u_full, 0, h, (int)t0);
                tma_load_3d(smem + kOffU + 8192, &map_u, &bars->u_full, 64, h, (int)t0);
            }
            if constexpr (GATED) {
                // inclusive prefix sums over the chunk: G_i = g_0 + ... + g_i
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y0 = __shfl_up_sync(0xffffffffu, g0, o);
                    const float y1 = __shfl_up_sync(0xffffffffu, g1, o);
                    if (lane >= o) {
                        g0 += y0;
                        g1 += y1;
                    }
                }
                g1 += __shfl_sync(0xffffffffu, g0, 31);
                float *G = stage_G(s);
                G[lane] = g0;
                G[lane + 32] = g1;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full[s]);
            __syncwarp();
        }
        // after a timeout: the loads already issued must land before shared memory is released
        if (!ok && lane == 0) {
            volatile int never = 0;
            for (int back = 1; back <= 2 && back <= c; ++back) {
                const int j = c - back;
                mbar_wait(&bars->full[j & 1], ((uint32_t)j >> 1) & 1u, &never, kGcWaitNs);
            }
            if (c > 0) mbar_wait(&bars->u_full, ((uint32_t)c - 1u) & 1u, &never, kGcWaitNs);  // the last U~ load
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------------ MMA issuer
        // One thread issues every product, in chunk order, each once the math warps have put its
        // operands in shared memory: an issue waits while the tensor pipe is busy, and no math warp
        // should wait there.
        if (lane == 0) {
            volatile int *abort = &bars->abort_flag;
            auto wait = [&](uint64_t *bar, uint32_t parity) {
                if (mbar_wait(bar, parity, abort, kGcWaitNs)) return true;
                if (atomicExch(&bars->abort_flag, 1) == 0) record_error(p.status, KKT_ERR_TIMEOUT);
                return false;
            };
            const uint32_t idesc_d = idesc_bf16_f32(128, kGcD + kGcC, 0, 0);
            const uint32_t idesc_s = idesc_bf16_f32(128, kGcD, 1, 1);
            const uint32_t idesc_o = idesc_bf16_f32(128, kGcD, 0, 1);
            const uint32_t p0 = smem_u32(smem + kOffPb), v0 = smem_u32(smem + kOffVb);
            const uint32_t vs = smem_u32(smem + (GATED ? kOffVf : kOffVb));
            for (int c = 0; c < nchunks; ++c) {
                const int s = c & 1;
                const uint32_t ph = (uint32_t)c & 1u;
                const uint32_t dcol = (c & 1) ? kColD1 : kColD0;
                const uint32_t qw = smem_u32(stage(s) + kOffQW), sk0 = smem_u32(stage(s) + kOffSK);
                // D = [Q; W] [S^T_b; K]^T.  Its buffer was drained: the output warps drain the O of chunk
                // c - 2 before they make P_b of chunk c - 1 ready, and the P V' of chunk c - 1 was issued
                // after that.
                if (!wait(&bars->sb_ready, ph)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + dcol, sw128_desc(qw + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                           sw128_desc(sk0 + (kk >> 2) * kBoxSK + (kk & 3) * 32, 16, 1024), idesc_d, kk > 0 ? 1u : 0u);
                mma_commit(&bars->bar_d);
                GC_TRACE(2, c);
                // S^T += V'(F)_b^T K
                if (!wait(&bars->v_ready, ph)) break;
                tc_fence_after();
                GC_TRACE(5, c);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + kColS, sw128_desc(vs + kk * 2048, 8192, 1024),
                           sw128_desc(sk0 + kOffKInBox + kk * 2048, kBoxSK, 1024), idesc_s, 1u);
                mma_commit(&bars->bar_s);
                mma_commit(&bars->empty[s]);
                // D += [P_b; 0] V'_b
                if (!wait(&bars->p_ready, ph)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + dcol, sw128_desc(p0 + kk * 32, 16, 1024), sw128_desc(v0 + kk * 2048, 8192, 1024),
                           idesc_o, 1u);
                mma_commit(&bars->bar_o);
                GC_TRACE(9, c);
            }
            // every MMA issued here has completed before tensor memory is released
            mma_commit(&bars->fin);
            volatile int never = 0;
            mbar_wait(&bars->fin, 0u, &never, kGcWaitNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ math warps (0-7)
        // Warp w reads tensor-memory lanes 32 (w & 3) .. + 31 and the half hc = w >> 2 of the columns of
        // each matrix there: 64 columns of S^T, of D's first 128 columns, and 32 of P's 64.
        const int q4 = warp & 3;
        const int hc = warp >> 2;
        const int row = 32 * q4 + lane;                   // tensor-memory lane = matrix row
        const bool out_side = row < 64;                   // rows 0..63: P, O; rows 64..127: W S, V'
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        uint8_t *pb = smem + kOffPb;
        uint8_t *vb = smem + kOffVb;
        uint8_t *vf = smem + kOffVf;
        uint32_t u256 = 0;
        bool ok = true;
        const int64_t state_base = ((int64_t)seq * p.H + h) * kGcD * kGcD;

        // the initial state into tensor memory: lane r holds column r of S (row r of S^T); the loads of
        // a warp read 32 consecutive floats of one row of S
#pragma unroll 1
        for (int piece = 0; piece < 4; ++piece) {
            uint32_t v[16];
            const int d0 = 64 * hc + 16 * piece;
#pragma unroll
            for (int e = 0; e < 16; ++e)
                v[e] = p.h0 ? __float_as_uint(__ldg(p.h0 + state_base + (int64_t)(d0 + e) * kGcD + row)) : 0u;
            tmem_st16(tmem + lane_base + kColS + d0, v);
        }
        tmem_wait_st();
        tc_fence_before();

        // O of chunk cp (buffer cp & 1), this warp's 64 columns of rows 0..63: scale, bf16, plain stores
        auto drain_o = [&](int cp, int64_t t0p, int Lcp) -> bool {
            if (!gc_wait(&bars->bar_o, (uint32_t)cp & 1u, bars, p.status)) return false;
            tc_fence_after();
            const uint32_t dcol = (cp & 1) ? kColD1 : kColD0;
            uint32_t v[2][32];
            tmem_ld32xN<2>(tmem + lane_base + dcol + 64 * hc, v);
            if (row < Lcp) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((t0p + row) * p.H + h) * kGcD + 64 * hc);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t *x = &v[j >> 2][8 * (j & 3)];
                    dst[j] = make_uint4(
                        pack2_bf16(p.scale * __uint_as_float(x[0]), p.scale * __uint_as_float(x[1])),
                        pack2_bf16(p.scale * __uint_as_float(x[2]), p.scale * __uint_as_float(x[3])),
                        pack2_bf16(p.scale * __uint_as_float(x[4]), p.scale * __uint_as_float(x[5])),
                        pack2_bf16(p.scale * __uint_as_float(x[6]), p.scale * __uint_as_float(x[7])));
                }
            }
            tc_fence_before();
            return true;
        };

        if (!gc_group(&bars->grp128, u256, bars, p.status)) ok = false;
        int64_t prev_t0 = 0;
        int prev_Lc = 0;
        int c = 0;
        for (; ok && c < nchunks; ++c) {
            const int s = c & 1;
            uint8_t *st = stage(s);
            uint8_t *sk = st + kOffSK;
            if (!gc_wait(&bars->full[s], ((uint32_t)c >> 1) & 1u, bars, p.status)) { ok = false; break; }
            if (threadIdx.x == 0) GC_TRACE(0, c);
            const GcInfo info = *stage_info(s);
            const int Lc = info.Lc;
            const float *G = stage_G(s);
            const int i = row - 64;
            // rows of a short chunk past its end: K's rows enter V'^T K (times zero rows of V') and
            // the masked columns of P, so they are zeroed (a row of the next sequence, or the fill
            // past the tensor, stays out)
            if (Lc < kGcC) {
                const int per = (kGcC - Lc) * 8;
                for (int e = threadIdx.x; e < 2 * per; e += 256) {
                    const int box = e / per, w = e % per;
                    *reinterpret_cast<uint4 *>(sk + box * kBoxSK + kOffKInBox + (Lc + w / 8) * 128 + (w % 8) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            // S^T row -> S^T_b (the state this chunk starts from), and, gated, S^T <- e^{G_last} S^T
            if (c > 0 && !gc_wait(&bars->bar_s, (uint32_t)(c - 1) & 1u, bars, p.status)) { ok = false; break; }
            tc_fence_after();
            if (threadIdx.x == 0) GC_TRACE(1, c);
            const float glast = GATED ? exp2f(G[Lc - 1]) : 1.f;
            {
                uint32_t v[2][32];
                tmem_ld32xN<2>(tmem + lane_base + kColS + 64 * hc, v);
                if (threadIdx.x == 0) GC_TRACE(15, c);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t *x = &v[j >> 2][8 * (j & 3)];
                    *sw_chunk(sk + hc * kBoxSK, row, j) =
                        make_uint4(pack2_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                   pack2_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                   pack2_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                   pack2_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
                }
                if constexpr (GATED) {
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        uint32_t w0[16], w1[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            w0[e] = __float_as_uint(glast * __uint_as_float(v[q2][e]));
                            w1[e] = __float_as_uint(glast * __uint_as_float(v[q2][16 + e]));
                        }
                        tmem_st16(tmem + lane_base + kColS + 64 * hc + 32 * q2, w0);
                        tmem_st16(tmem + lane_base + kColS + 64 * hc + 32 * q2 + 16, w1);
                    }
                    tmem_wait_st();
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->sb_ready);  // S^T_b (and the zeroed K rows) are written
            if (threadIdx.x == 0) GC_TRACE(11, c);
            const uint32_t dcol = (c & 1) ? kColD1 : kColD0;
            if (!out_side) {
                // W S row -> V' = U~ - W S (zero past the chunk's end) -> V'_b (and VF_b), this warp's
                // 64 columns.  D is in tensor memory; the P V' product of chunk c - 1, the last reader of
                // V'_b, was issued before D by the same thread, so it has completed too.
                if (!gc_wait(&bars->bar_d, (uint32_t)c & 1u, bars, p.status)) { ok = false; break; }
                if (!gc_wait(&bars->u_full, (uint32_t)c & 1u, bars, p.status)) { ok = false; break; }
                tc_fence_after();
                if (threadIdx.x == 64) GC_TRACE(3, c);
                const float fi = (GATED && i < Lc) ? exp2f(G[Lc - 1] - G[i]) : 1.f;
                // the row's U~ chunks into registers before any store: the compiler cannot tell the
                // V'_b stores from the U~ buffer, and would otherwise wait for each store before the
                // next load
                uint4 ur[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) ur[j] = *sw_chunk(smem + kOffU + hc * 8192, i, j);
                uint32_t vv[2][32];
                tmem_ld32xN<2>(tmem + lane_base + dcol + 64 * hc, vv);
                if (threadIdx.x == 64) GC_TRACE(12, c);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t *x = &vv[j >> 2][8 * (j & 3)];
                    const uint4 uu = ur[j];
                    const uint32_t uw[4] = {uu.x, uu.y, uu.z, uu.w};
                    uint32_t o1[4], o2[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 uf = unpack2_bf16(uw[e]);
                        float y0 = uf.x - __uint_as_float(x[2 * e]);
                        float y1 = uf.y - __uint_as_float(x[2 * e + 1]);
                        if (i >= Lc) y0 = y1 = 0.f;
                        o1[e] = pack2_bf16(y0, y1);
                        o2[e] = pack2_bf16(fi * y0, fi * y1);
                    }
                    *sw_chunk(vb + hc * 8192, i, j) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                    if constexpr (GATED)
                        *sw_chunk(vf + hc * 8192, i, j) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
                }
                if (threadIdx.x == 64) GC_TRACE(13, c);
                fence_proxy_async_smem();
                if (threadIdx.x == 64) GC_TRACE(14, c);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars->v_ready);  // this warp's part of V'_b (and VF_b)
                    mbar_arrive(&bars->u_empty);  // and its reads of the U~ buffer are done
                }
                if (threadIdx.x == 64) GC_TRACE(4, c);
            } else {
                // the previous chunk's O, while this chunk's products run
                if (c > 0 && !drain_o(c - 1, prev_t0, prev_Lc)) { ok = false; break; }
                if (threadIdx.x == 0) GC_TRACE(6, c);
                // P row -> causal mask (times Gamma when gated) -> P_b, this warp's 32 columns
                if (!gc_wait(&bars->bar_d, (uint32_t)c & 1u, bars, p.status)) { ok = false; break; }
                tc_fence_after();
                if (threadIdx.x == 0) GC_TRACE(7, c);
                const float gi = GATED ? G[row] : 0.f;
                {
                    // gated: the 32 columns' prefix sums into registers before the P_b stores
                    float gc[32];
                    if constexpr (GATED) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float4 g4 = *reinterpret_cast<const float4 *>(G + 32 * hc + 4 * e);
                            gc[4 * e] = g4.x; gc[4 * e + 1] = g4.y; gc[4 * e + 2] = g4.z; gc[4 * e + 3] = g4.w;
                        }
                    }
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + dcol + kColDP + 32 * hc, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float y[2];
#pragma unroll
                            for (int u2 = 0; u2 < 2; ++u2) {
                                const int col = 32 * hc + 8 * j + 2 * e + u2;
                                float z = (col <= row && row < Lc) ? __uint_as_float(v[8 * j + 2 * e + u2]) : 0.f;
                                if constexpr (GATED)
                                    z = (col <= row && row < Lc) ? z * fast_exp2(gi - gc[8 * j + 2 * e + u2]) : 0.f;
                                y[u2] = z;
                            }
                            w[e] = pack2_bf16(y[0], y[1]);
                        }
                        *sw_chunk(pb, row, 4 * hc + j) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                if constexpr (GATED) {
                    // Q S row -> e^{G_row} Q S (the state term's decay), in place, this warp's 64 columns
                    const float ri = exp2f(gi);
                    uint32_t v[2][32];
                    tmem_ld32xN<2>(tmem + lane_base + dcol + 64 * hc, v);
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        uint32_t w0[16], w1[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            w0[e] = __float_as_uint(ri * __uint_as_float(v[q2][e]));
                            w1[e] = __float_as_uint(ri * __uint_as_float(v[q2][16 + e]));
                        }
                        tmem_st16(tmem + lane_base + dcol + 64 * hc + 32 * q2, w0);
                        tmem_st16(tmem + lane_base + dcol + 64 * hc + 32 * q2 + 16, w1);
                    }
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                // P_b (and the decayed Q S) are ready, and this warp is done with the stage's gate data
                if (lane == 0) {
                    mbar_arrive(&bars->p_ready);
                    mbar_arrive(&bars->empty[s]);
                }
                if (threadIdx.x == 0) GC_TRACE(8, c);
            }
            prev_t0 = info.t0;
            prev_Lc = Lc;
        }
        // the last chunk's O, and the final state (lane r holds column r of S)
        if (ok && nchunks > 0 && out_side && !drain_o(nchunks - 1, prev_t0, prev_Lc)) ok = false;
        if (ok && p.ht) {
            if (nchunks > 0 && !gc_wait(&bars->bar_s, (uint32_t)(nchunks - 1) & 1u, bars, p.status)) ok = false;
            if (ok) {
                tc_fence_after();
                uint32_t v[2][32];
                tmem_ld32xN<2>(tmem + lane_base + kColS + 64 * hc, v);
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    p.ht[state_base + (int64_t)(64 * hc + e) * kGcD + row] = __uint_as_float(v[e >> 5][e & 31]);
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kGcTmemCols);
}

template <bool GATED>
bool gc_ensure_smem() {
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(gdn_chunk_kernel<GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGcSmem) !=
        cudaSuccess)
        return false;
    done[dev] = true;
    return true;
}

bool aligned_to(const void *ptr, uintptr_t n) { return (reinterpret_cast<uintptr_t>(ptr) & (n - 1)) == 0; }

#ifdef KKT_TRACE
void *g_gc_trace = nullptr;
#endif

}  // namespace
}  // namespace kkt

#ifdef KKT_TRACE
// Trace builds only: device buffer of kGcTraceCtas x kGcTraceChunks x kGcTraceEvents uint64 cycle counts of
// the recurrence kernel, or NULL to stop tracing.
extern "C" void gdn_set_trace_buffer(void *buf) { kkt::g_gc_trace = buf; }
#endif

extern "C" int gdn_chunk_state_fwd(const void *q, const void *k, const void *w, const void *u, const float *g,
                                   const float *initial_state, const int32_t *cu_seqlens, int B, int T, int H,
                                   int dk, int dv, int C, float scale, void *o, float *final_state,
                                   struct CUstream_st *stream) {
    using namespace kkt;
    if (B < 1 || T < 0 || H < 1 || H > 65535) return KKT_ERR_ARG;
    const int64_t ntok = cu_seqlens ? (int64_t)T : (int64_t)B * T;
    // the token tensors may be empty (and their pointers null) only when there are no tokens
    if (ntok > 0 && (!q || !k || !w || !u || !o)) return KKT_ERR_ARG;
    if (dk != kGcD || dv != kGcD || C != kGcC) return KKT_ERR_UNSUPPORTED;
    if (!aligned_to(q, 16) || !aligned_to(k, 16) || !aligned_to(w, 16) || !aligned_to(u, 16) || !aligned_to(o, 16) ||
        !aligned_to(initial_state, 16) || !aligned_to(final_state, 16) || !aligned_to(g, 4) ||
        !aligned_to(cu_seqlens, 4))
        return KKT_ERR_ALIGN;
    if ((int64_t)B * H > 0x7fffffffLL || ntok > 0x7fffffffLL) return KKT_ERR_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t state_bytes = (size_t)B * H * kGcD * kGcD * sizeof(float);
    if (ntok == 0) {
        // no tokens: the final state is the initial one
        if (!final_state) return KKT_OK;
        const cudaError_t e = initial_state
                                  ? cudaMemcpyAsync(final_state, initial_state, state_bytes, cudaMemcpyDeviceToDevice, st)
                                  : cudaMemsetAsync(final_state, 0, state_bytes, st);
        return e == cudaSuccess ? KKT_OK : KKT_ERR_CUDA;
    }
    GcParams p;
    p.g = g;
    p.h0 = initial_state;
    p.ht = final_state;
    p.cu = cu_seqlens;
    p.nseq = B;
    p.T = T;
    p.ntok = ntok;
    p.H = H;
    p.scale = scale;
    p.u = static_cast<const __nv_bfloat16 *>(u);
    p.o = static_cast<__nv_bfloat16 *>(o);
#ifdef KKT_TRACE
    p.trace = static_cast<unsigned long long *>(g_gc_trace);
#else
    p.trace = nullptr;
#endif
    int rc = status_ptr(&p.status);
    if (rc != KKT_OK) return rc;
    CUtensorMap mq, mk, mw, mu;
    if (!make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, ntok, H, kGcD, 64, kGcC) ||
        !make_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, ntok, H, kGcD, 64, kGcC) ||
        !make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, ntok, H, kGcD, 64, kGcC) ||
        !make_map(&mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, u, ntok, H, kGcD, 64, kGcC))
        return KKT_ERR_CUDA;
    auto kern = g ? gdn_chunk_kernel<true> : gdn_chunk_kernel<false>;
    if (!(g ? gc_ensure_smem<true>() : gc_ensure_smem<false>())) return KKT_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)B * H));
    cfg.blockDim = dim3(kGcThreads);
    cfg.dynamicSmemBytes = kGcSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mq, mk, mw, mu, p) != cudaSuccess) return KKT_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KKT_OK : KKT_ERR_CUDA;
}
