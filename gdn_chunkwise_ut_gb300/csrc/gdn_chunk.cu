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
//   tensor memory (512 columns): S [128 x 128] fp32 (row d of S in lane d); two D buffers
//   [128 x 128] fp32; P [128 x 64] fp32.
//   shared memory: a two-deep ring of stages, each with [Q; W] (per 64-column box: the 64 rows of
//   Q, then the 64 rows of W, so that the pair is one 128-row operand), K and U~, all loaded by TMA
//   with the 128-byte swizzle; the bf16 copies S_b of S, P_b of the masked P (rows 64..127 zero),
//   V'_b of V' (and, gated, VF_b of diag(e^{G_last - G}) V'), and the staging of O.
// Per chunk, every tcgen05.mma M = 128, one thread issuing:
//   P  = [Q; W] K^T           (N = 64; rows 0..63 are Q K^T, rows 64..127 unused)
//   D  = [Q; W] S_b           (N = 128; rows 0..63 Q S, rows 64..127 W S: one product for both)
//   S += K^T V'(F)_b          (A = K^T read MN-major from the stage, N = 128, K = 64 tokens)
//   D += [P_b; 0] V'_b        (rows 0..63 become O / scale, before the gate's row factor when gated)
// and the math threads between them: S -> S_b (and, gated, S <- e^{G_last} S in place); P row ->
// causal mask (times Gamma) -> P_b; W S row -> V' = U~ - W S -> V'_b; gated, Q S row -> e^{G_i} Q S;
// O row -> scale -> bf16 -> staging -> TMA store (plain stores for a short last chunk).  The two D
// buffers let the O of one chunk drain while the next chunk's products run.
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
constexpr int kGcThreads = 160;           // warps 0-3 math, warp 4 loads
constexpr uint32_t kGcTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColD0 = 128;
constexpr uint32_t kColD1 = 256;
constexpr uint32_t kColP = 384;
constexpr uint64_t kGcWaitNs = 2000000000ull;

// shared memory, from a 1024-byte-aligned base
constexpr int kStageBytes = 65536;        // [Q; W] 32 KB, K 16 KB, U~ 16 KB
constexpr int kOffQW = 0;
constexpr int kOffK = 32768;
constexpr int kOffU = 49152;
constexpr int kOffSb = 2 * kStageBytes;   // 2 boxes x [128 rows][128 B]
constexpr int kOffPb = kOffSb + 32768;    // [128 rows][128 B]
constexpr int kOffVb = kOffPb + 16384;    // 2 boxes x [64 rows][128 B]
constexpr int kOffVf = kOffVb + 16384;
constexpr int kOffOb = kOffVf + 16384;
constexpr int kOffMeta = kOffOb + 16384;  // per stage 512 B: G[64] (log2 units), then the chunk info
constexpr int kOffBar = kOffMeta + 1024;
constexpr int kGcSmem = kOffBar + 256 + 1024;  // + alignment slack
static_assert(kGcSmem <= 232448, "shared memory over the per-block limit");
constexpr uint32_t kStageTx = 65536;

struct GcInfo {
    int64_t t0;
    int Lc;
    int pad;
};

struct GcBars {
    uint64_t full[2], empty[2];
    uint64_t bar_p, bar_d, bar_s, bar_o;
    uint64_t grp128, grp64, fin;
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
    __nv_bfloat16 *o;
    int *status;
};

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

template <bool GATED>
__global__ void __launch_bounds__(kGcThreads, 1)
    gdn_chunk_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_u,
                     const __grid_constant__ CUtensorMap map_o, const GcParams p) {
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
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->bar_p, 1);
        mbar_init(&bars->bar_d, 1);
        mbar_init(&bars->bar_s, 1);
        mbar_init(&bars->bar_o, 1);
        mbar_init(&bars->grp128, 4);
        mbar_init(&bars->grp64, 2);
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

    if (warp == 4) {
        // ------------------------------------------------------------------ loads
        if (lane == 0) {
            prefetch_tmap(&map_q);
            prefetch_tmap(&map_k);
            prefetch_tmap(&map_w);
            prefetch_tmap(&map_u);
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
                GcInfo *info = stage_info(s);
                info->t0 = t0;
                info->Lc = Lc;
                uint8_t *st = stage(s);
                mbar_arrive_expect_tx(&bars->full[s], kStageTx);
                for (int c2 = 0; c2 < 2; ++c2) {
                    tma_load_3d(st + kOffQW + c2 * 16384, &map_q, &bars->full[s], 64 * c2, h, (int)t0);
                    tma_load_3d(st + kOffQW + c2 * 16384 + 8192, &map_w, &bars->full[s], 64 * c2, h, (int)t0);
                    tma_load_3d(st + kOffK + c2 * 8192, &map_k, &bars->full[s], 64 * c2, h, (int)t0);
                    tma_load_3d(st + kOffU + c2 * 8192, &map_u, &bars->full[s], 64 * c2, h, (int)t0);
                }
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
            for (int back = 1; back <= 2 && back <= c; ++back) {
                const int j = c - back;
                volatile int never = 0;
                mbar_wait(&bars->full[j & 1], ((uint32_t)j >> 1) & 1u, &never, kGcWaitNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ math warps
        const int t = threadIdx.x;                        // tensor-memory lane = row
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        uint8_t *sb = smem + kOffSb;
        uint8_t *pb = smem + kOffPb;
        uint8_t *vb = smem + kOffVb;
        uint8_t *vf = smem + kOffVf;
        uint8_t *ob = smem + kOffOb;
        uint32_t u128 = 0, u64 = 0;
        bool ok = true;
        const int64_t state_off = ((int64_t)seq * p.H + h) * kGcD * kGcD + (int64_t)t * kGcD;

        // the initial state into tensor memory, row t of S in lane t
#pragma unroll 1
        for (int piece = 0; piece < 8; ++piece) {
            uint32_t v[16];
            if (p.h0) {
                const float4 *src = reinterpret_cast<const float4 *>(p.h0 + state_off + 16 * piece);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 x = __ldg(src + e);
                    v[4 * e] = __float_as_uint(x.x);
                    v[4 * e + 1] = __float_as_uint(x.y);
                    v[4 * e + 2] = __float_as_uint(x.z);
                    v[4 * e + 3] = __float_as_uint(x.w);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = 0u;
            }
            tmem_st16(tmem + lane_base + kColS + 16 * piece, v);
        }
        tmem_wait_st();
        tc_fence_before();

        // O of chunk cp (buffer cp & 1): rows 0..63, threads 0..63
        auto drain_o = [&](int cp, int64_t t0p, int Lcp) -> bool {
            if (!gc_wait(&bars->bar_o, (uint32_t)cp & 1u, bars, p.status)) return false;
            tc_fence_after();
            const uint32_t dcol = (cp & 1) ? kColD1 : kColD0;
            const bool full = Lcp == kGcC;
            if (full) {
                if (t == 0) bulk_wait_read<0>();  // the previous store has read the staging
                if (!gc_group(&bars->grp64, u64, bars, p.status)) return false;
            }
#pragma unroll 1
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + dcol + 32 * piece, v);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack2_bf16(p.scale * __uint_as_float(v[2 * e]), p.scale * __uint_as_float(v[2 * e + 1]));
                if (full) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *sw_chunk(ob + (piece >> 1) * 8192, t, (piece & 1) * 4 + j) =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                } else if (t < Lcp) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((t0p + t) * p.H + h) * kGcD + 32 * piece);
#pragma unroll
                    for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                }
            }
            tc_fence_before();
            if (full) {
                fence_proxy_async_smem();
                if (!gc_group(&bars->grp64, u64, bars, p.status)) return false;
                if (t == 0) {
                    tma_store_3d(&map_o, ob, 0, h, (int)t0p);
                    tma_store_3d(&map_o, ob + 8192, 64, h, (int)t0p);
                    bulk_commit();
                }
            }
            return true;
        };

        if (!gc_group(&bars->grp128, u128, bars, p.status)) ok = false;
        int64_t prev_t0 = 0;
        int prev_Lc = 0;
        int c = 0;
        for (; ok && c < nchunks; ++c) {
            const int s = c & 1;
            uint8_t *st = stage(s);
            if (!gc_wait(&bars->full[s], ((uint32_t)c >> 1) & 1u, bars, p.status)) { ok = false; break; }
            const GcInfo info = *stage_info(s);
            const int Lc = info.Lc;
            const float *G = stage_G(s);
            // rows of a short chunk past its end: K's rows enter K^T V' (times zero rows of V'), so
            // they are zeroed (a row of the next sequence, or the fill past the tensor, stays out)
            if (Lc < kGcC) {
                const int per = (kGcC - Lc) * 8;
                for (int e = t; e < 2 * per; e += 128) {
                    const int box = e / per, w = e % per;
                    *reinterpret_cast<uint4 *>(st + kOffK + box * 8192 + (Lc + w / 8) * 128 + (w % 8) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            if (!gc_group(&bars->grp128, u128, bars, p.status)) { ok = false; break; }
            // P = [Q; W] K^T
            if (t == 0) {
                tc_fence_after();
                const uint32_t idesc_p = idesc_bf16_f32(128, kGcC, 0, 0);
                const uint32_t qw = smem_u32(st + kOffQW), kk0 = smem_u32(st + kOffK);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + kColP, sw128_desc(qw + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                           sw128_desc(kk0 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), idesc_p, kk > 0 ? 1u : 0u);
                mma_commit(&bars->bar_p);
            }
            // S -> S_b (the state this chunk starts from), and, gated, S <- e^{G_last} S in place
            if (c > 0 && !gc_wait(&bars->bar_s, (uint32_t)(c - 1) & 1u, bars, p.status)) { ok = false; break; }
            tc_fence_after();
            const float glast = GATED ? exp2f(G[Lc - 1]) : 1.f;
#pragma unroll 1
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kColS + 32 * piece, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *sw_chunk(sb + (piece >> 1) * 16384, t, (piece & 1) * 4 + j) = make_uint4(
                        pack2_bf16(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                        pack2_bf16(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                        pack2_bf16(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                        pack2_bf16(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
                if constexpr (GATED) {
                    uint32_t w0[16], w1[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        w0[e] = __float_as_uint(glast * __uint_as_float(v[e]));
                        w1[e] = __float_as_uint(glast * __uint_as_float(v[16 + e]));
                    }
                    tmem_st16(tmem + lane_base + kColS + 32 * piece, w0);
                    tmem_st16(tmem + lane_base + kColS + 32 * piece + 16, w1);
                }
            }
            if constexpr (GATED) tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            if (!gc_group(&bars->grp128, u128, bars, p.status)) { ok = false; break; }
            // D = [Q; W] S_b
            const uint32_t dcol = (c & 1) ? kColD1 : kColD0;
            if (t == 0) {
                tc_fence_after();
                const uint32_t idesc_d = idesc_bf16_f32(128, kGcD, 0, 1);
                const uint32_t qw = smem_u32(st + kOffQW), s0 = smem_u32(sb);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tmem + dcol, sw128_desc(qw + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                           sw128_desc(s0 + kk * 2048, 16384, 1024), idesc_d, kk > 0 ? 1u : 0u);
                mma_commit(&bars->bar_d);
            }
            if (t < 64) {
                // the previous chunk's O, while this chunk's products run
                if (c > 0 && !drain_o(c - 1, prev_t0, prev_Lc)) { ok = false; break; }
                // P row t -> causal mask (times Gamma when gated) -> P_b row t
                if (!gc_wait(&bars->bar_p, (uint32_t)c & 1u, bars, p.status)) { ok = false; break; }
                tc_fence_after();
                const float gi = GATED ? G[t] : 0.f;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + kColP + 32 * half, v);
                    tmem_wait_ld();
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int j = 32 * half + e;
                        float y = (j <= t && t < Lc) ? __uint_as_float(v[e]) : 0.f;
                        if constexpr (GATED) y = (j <= t && t < Lc) ? y * exp2f(gi - G[j]) : 0.f;
                        x[e] = y;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *sw_chunk(pb, t, 4 * half + j) =
                            make_uint4(pack2_bf16(x[8 * j], x[8 * j + 1]), pack2_bf16(x[8 * j + 2], x[8 * j + 3]),
                                       pack2_bf16(x[8 * j + 4], x[8 * j + 5]), pack2_bf16(x[8 * j + 6], x[8 * j + 7]));
                }
                if constexpr (GATED) {
                    // Q S row t -> e^{G_t} Q S (the state term's decay), in place
                    if (!gc_wait(&bars->bar_d, (uint32_t)c & 1u, bars, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const float ri = exp2f(gi);
#pragma unroll 1
                    for (int piece = 0; piece < 8; ++piece) {
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_base + dcol + 16 * piece, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(ri * __uint_as_float(v[e]));
                        tmem_st16(tmem + lane_base + dcol + 16 * piece, v);
                    }
                    tmem_wait_st();
                }
            } else {
                // W S row t -> V' = U~ - W S (zero past the chunk's end) -> V'_b (and VF_b) row t - 64
                const int i = t - 64;
                if (!gc_wait(&bars->bar_d, (uint32_t)c & 1u, bars, p.status)) { ok = false; break; }
                tc_fence_after();
                const float fi = (GATED && i < Lc) ? exp2f(G[Lc - 1] - G[i]) : 1.f;
#pragma unroll 1
                for (int piece = 0; piece < 4; ++piece) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + dcol + 32 * piece, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int ch = (piece & 1) * 4 + j;
                        const uint4 uu = *sw_chunk(st + kOffU + (piece >> 1) * 8192, i, ch);
                        const uint32_t uw[4] = {uu.x, uu.y, uu.z, uu.w};
                        uint32_t o1[4], o2[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 uf = unpack2_bf16(uw[e]);
                            float y0 = uf.x - __uint_as_float(v[8 * j + 2 * e]);
                            float y1 = uf.y - __uint_as_float(v[8 * j + 2 * e + 1]);
                            if (i >= Lc) y0 = y1 = 0.f;
                            o1[e] = pack2_bf16(y0, y1);
                            o2[e] = pack2_bf16(fi * y0, fi * y1);
                        }
                        *sw_chunk(vb + (piece >> 1) * 8192, i, ch) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                        if constexpr (GATED)
                            *sw_chunk(vf + (piece >> 1) * 8192, i, ch) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (!gc_group(&bars->grp128, u128, bars, p.status)) { ok = false; break; }
            // S += K^T V'(F)_b, then D += [P_b; 0] V'_b
            if (t == 0) {
                tc_fence_after();
                const uint32_t idesc_s = idesc_bf16_f32(128, kGcD, 1, 1);
                const uint32_t idesc_o = idesc_bf16_f32(128, kGcD, 0, 1);
                const uint32_t kk0 = smem_u32(st + kOffK), vs = smem_u32(GATED ? vf : vb), v0 = smem_u32(vb);
                const uint32_t p0 = smem_u32(pb);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + kColS, sw128_desc(kk0 + kk * 2048, 8192, 1024), sw128_desc(vs + kk * 2048, 8192, 1024),
                           idesc_s, 1u);
                mma_commit(&bars->bar_s);
                mma_commit(&bars->empty[s]);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + dcol, sw128_desc(p0 + kk * 32, 16, 1024), sw128_desc(v0 + kk * 2048, 8192, 1024),
                           idesc_o, 1u);
                mma_commit(&bars->bar_o);
            }
            prev_t0 = info.t0;
            prev_Lc = Lc;
        }
        // the last chunk's O, and the final state
        if (ok && nchunks > 0 && t < 64 && !drain_o(nchunks - 1, prev_t0, prev_Lc)) ok = false;
        if (ok && p.ht) {
            if (nchunks > 0 && !gc_wait(&bars->bar_s, (uint32_t)(nchunks - 1) & 1u, bars, p.status)) ok = false;
            if (ok) {
                tc_fence_after();
                float4 *dst = reinterpret_cast<float4 *>(p.ht + state_off);
#pragma unroll 1
                for (int piece = 0; piece < 4; ++piece) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + kColS + 32 * piece, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[8 * piece + e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                         __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                }
            }
        }
        // every MMA this CTA issued has completed, and the O stores have left shared memory
        if (t == 0) {
            mma_commit(&bars->fin);
            volatile int never = 0;
            mbar_wait(&bars->fin, 0u, &never, kGcWaitNs);
            bulk_wait<0>();
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

}  // namespace
}  // namespace kkt

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
    p.o = static_cast<__nv_bfloat16 *>(o);
    int rc = status_ptr(&p.status);
    if (rc != KKT_OK) return rc;
    CUtensorMap mq, mk, mw, mu, mo;
    if (!make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, ntok, H, kGcD, 64, kGcC) ||
        !make_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, ntok, H, kGcD, 64, kGcC) ||
        !make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, ntok, H, kGcD, 64, kGcC) ||
        !make_map(&mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, u, ntok, H, kGcD, 64, kGcC) ||
        !make_map(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o, ntok, H, kGcD, 64, kGcC))
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
    if (cudaLaunchKernelEx(&cfg, kern, mq, mk, mw, mu, mo, p) != cudaSuccess) return KKT_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KKT_OK : KKT_ERR_CUDA;
}
