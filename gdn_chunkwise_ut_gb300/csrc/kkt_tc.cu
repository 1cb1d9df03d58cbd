// kkt_tc.cu -- persistent, warp-specialised tcgen05 + TMA kernel for kkt_solve (bf16 I/O).
//
// One CTA per SM walks "tiles" of 128 rows: G = 128 / C heads of one chunk,
// row m = g * C + r (head g, token r of the chunk).  For each tile
// ("TileLang 实战：单位下三角矩阵求逆" §1, §2.2, §3):
//
//   producer warp   TMA: K and V boxes {64 cols, 1 head, C rows} (128-byte
//                   swizzle) into a stage of the shared-memory ring; beta with
//                   plain loads.
//   MMA warp        tcgen05.mma S = K K^T  (M = N = 128, K = 128, bf16 -> fp32
//                   in tensor memory); later D = T~ [K | V] with T~ = T diag(beta)
//                   taken from tensor memory as a bf16 hi + lo pair (two
//                   accumulating passes, M = 128, N = 256, K = 128; T~ is block
//                   diagonal over the G heads).
//   inverse warps   one thread per row: tcgen05.ld of its Gram row, beta row
//                   scale, strict-lower mask and unit diagonal (§3.2); 16 x 16
//                   diagonal blocks by forward substitution with warp shuffles
//                   (§2.1, §3.4; the original row lives in registers, so the
//                   in-place update needs no backup copy); coupling
//                   -L11^-1 L10 L00^-1 at s = 16 (shuffles) and s = 32 (shared
//                   memory between the two warps of a head) (§2.2, §3.5);
//                   T rows to a swizzled staging buffer + TMA store; T~ hi / lo
//                   to tensor memory with tcgen05.st.
//   epilogue warps  tcgen05.ld of D, bf16 conversion, swizzled staging in the
//                   stage's K/V buffers (free once the MMA has read them), TMA
//                   stores of W and U~; then the stage goes back to the producer.
//
// Short last chunks (Lc < C) are zero-padded in shared memory before the Gram
// MMA and written back with plain stores of the Lc valid rows.  Every wait is
// bounded: on expiry the kernel records KKT_ERR_TIMEOUT, stops all roles,
// drains its own copies and MMAs, frees tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kkt_internal.cuh"
#include "sm100_ptx.cuh"

namespace kkt {
namespace {

using namespace ptx;

constexpr int kThreads = 384;            // 12 warps
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpInv0 = 4;             // warps 4..7
constexpr int kWarpEpi0 = 8;             // warps 8..11
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColGram = 0;         // 128 fp32 columns
constexpr uint32_t kColD = 128;          // 256 fp32 columns: W | U~
constexpr uint32_t kColTT = 384;         // 64 packed bf16x2 hi + 64 lo
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait


struct TileInfo {
    int64_t t0;
    int Lc;
    int h0;
    int done;
    int pad;
};

template <int C>
struct Cfg {
    static constexpr int G = 128 / C;             // heads per tile
    static constexpr int NS = 2;                  // stages
    static constexpr int KV_BYTES = 65536;        // K 32 KB + V 32 KB, [colhalf][row][128 B]
    static constexpr int STAGE_BYTES = KV_BYTES + 1024;  // + beta[128] + info, 1 KB aligned
    static constexpr int OFF_BETA = KV_BYTES;
    static constexpr int OFF_INFO = KV_BYTES + 512;
    static constexpr int T_HALVES = C / 32;       // 128-byte column blocks of a T row
    static constexpr int T_STAGE_BYTES = T_HALVES * 16384;
    static constexpr int XCH_BYTES = (C >= 64) ? G * (2 * 4096 + 4096) : 0;  // level-32 exchange
    static constexpr int OFF_T = NS * STAGE_BYTES;
    static constexpr int OFF_XCH = OFF_T + T_STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_XCH + XCH_BYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TX_BYTES = G * 4 * C * 128;           // K + V boxes of one stage
};

struct Barriers {
    uint64_t full[2];
    uint64_t empty[2];
    uint64_t gram_full, gram_empty;
    uint64_t tt_full, tt_empty;
    uint64_t d_full, d_empty;
    uint64_t mma_final;
    uint64_t inv_sync;       // 128 inverse threads
    uint64_t epi_sync;       // 128 epilogue threads
    uint64_t pair_sync[2];   // the two warps of one head (C = 64)
    uint32_t tmem_base;
    int abort_flag;
};

struct TcParams {
    const float *beta;
    const int32_t *cu;
    int nseq, T;
    int64_t ntok;
    int H;
    int64_t tiles;   // work ids x head groups
    int HG;          // head groups
    float *T_out;
    __nv_bfloat16 *W_out, *U_out;
    int *status;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void fail(Barriers *bars, int *status) {
    if (atomicExch(&bars->abort_flag, 1) == 0) record_error(status, KKT_ERR_TIMEOUT);
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Barriers *bars, int *status) {
    if (mbar_wait(bar, parity, &bars->abort_flag, kWaitLimitNs)) return true;
    fail(bars, status);
    return false;
}

// Group barrier on an mbarrier (every member arrives, then waits for the phase):
// unlike bar.sync it is bounded, so a member that gave up cannot hang the others.
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &uses, Barriers *bars, int *status) {
    mbar_arrive(bar);
    const bool ok = wait_bar(bar, uses & 1u, bars, status);
    ++uses;
    return ok;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// ---------------------------------------------------------------------------------------------
// Inverse of one 16 x 16 unit lower-triangular block, one row per lane of a half warp:
// lb[c] = L[k][c] (zero for c >= k), x[c] <- (L^-1)[k][c].  Right-looking substitution:
// once row m is final, every later row subtracts L[k][m] * row m (§2.1).
__device__ __forceinline__ void diag16(const float (&lb)[16], float (&x)[16], int lane) {
    const int k = lane & 15;
    const int base = lane & 16;
#pragma unroll
    for (int c = 0; c < 16; ++c) x[c] = (c == k) ? 1.f : 0.f;
#pragma unroll
    for (int m = 0; m < 15; ++m) {
        const float lm = lb[m];
        x[m] -= lm;
#pragma unroll
        for (int c = 0; c < m; ++c) {
            const float xm = __shfl_sync(0xffffffffu, x[c], base + m);
            x[c] = fmaf(-lm, xm, x[c]);
        }
    }
}

// Level-16 coupling inside one warp: lanes 16..31 (block 1) get
// T10[k][:] = -X11[k][:] (L10 X00), with X00 rows on lanes 0..15.
// l10[j] = L[row][first column of block 0 + j].  Returns m32: the lane's row of the
// warp's 32 x 32 inverse (columns of block 0 then block 1).
__device__ __forceinline__ void couple16(const float (&l10)[16], const float (&x)[16], int lane,
                                         float (&m32)[32]) {
    float y[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) y[c] = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
#pragma unroll
        for (int c = 0; c <= j; ++c) {
            const float xjc = __shfl_sync(0xffffffffu, x[c], j);
            y[c] = fmaf(l10[j], xjc, y[c]);
        }
    }
    float z[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) z[c] = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const float yic = __shfl_sync(0xffffffffu, y[c], 16 + i);
            z[c] = fmaf(x[i], yic, z[c]);
        }
    }
    const bool upper = lane >= 16;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        m32[c] = upper ? -z[c] : x[c];
        m32[16 + c] = upper ? x[c] : 0.f;
    }
}

// ---------------------------------------------------------------------------------------------
template <int C>
__global__ void __launch_bounds__(kThreads, 1)
    kkt_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                  const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_u,
                  const __grid_constant__ CUtensorMap map_t, const TcParams p) {
    using CF = Cfg<C>;
    constexpr int G = CF::G;
    constexpr int NS = CF::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    Barriers *bars = reinterpret_cast<Barriers *>(smem + CF::OFF_BAR);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto stage_ptr = [&](int s) { return smem + s * CF::STAGE_BYTES; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->gram_full, 1);
        mbar_init(&bars->gram_empty, 4);
        mbar_init(&bars->tt_full, 4);
        mbar_init(&bars->tt_empty, 1);
        mbar_init(&bars->d_full, 1);
        mbar_init(&bars->d_empty, 4);
        mbar_init(&bars->mma_final, 1);
        mbar_init(&bars->inv_sync, 128);
        mbar_init(&bars->epi_sync, 128);
        mbar_init(&bars->pair_sync[0], 64);
        mbar_init(&bars->pair_sync[1], 64);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == kWarpProducer) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&map_k);
            prefetch_tmap(&map_v);
        }
        int i = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
            const int64_t id = t / p.HG;
            const int h0 = (int)(t % p.HG) * G;
            if (h0 == 0 && id < p.nseq && lane == 0) check_sequence(p.cu, (int)id, p.nseq, p.ntok, p.status);
            Chunk ch;
            if (!map_chunk(id, p.cu, p.nseq, p.T, p.ntok, C, p.status, ch)) continue;
            const int s = i % NS;
            const uint32_t u = (uint32_t)(i / NS);
            if (!wait_bar(&bars->empty[s], (u & 1u) ^ 1u, bars, p.status)) { ok = false; break; }
            uint8_t *st = stage_ptr(s);
            float *sb = reinterpret_cast<float *>(st + CF::OFF_BETA);
            for (int idx = lane; idx < G * C; idx += 32) {
                const int g = idx / C, r = idx % C;
                float b = 0.f;
                if (r < ch.Lc && h0 + g < p.H) b = __ldg(p.beta + (ch.t0 + r) * p.H + h0 + g);
                sb[idx] = b;
            }
            if (lane == 0) {
                TileInfo *info = reinterpret_cast<TileInfo *>(st + CF::OFF_INFO);
                info->t0 = ch.t0;
                info->Lc = ch.Lc;
                info->h0 = h0;
                info->done = 0;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->full[s], CF::TX_BYTES);
                for (int g = 0; g < G; ++g)
                    for (int c2 = 0; c2 < 2; ++c2) {
                        tma_load_3d(st + c2 * 16384 + g * C * 128, &map_k, &bars->full[s], c2 * 64, h0 + g,
                                    (int)ch.t0);
                        tma_load_3d(st + 32768 + c2 * 16384 + g * C * 128, &map_v, &bars->full[s], c2 * 64,
                                    h0 + g, (int)ch.t0);
                    }
            }
            __syncwarp();
            ++i;
        }
        if (ok) {
            const int s = i % NS;
            const uint32_t u = (uint32_t)(i / NS);
            if (wait_bar(&bars->empty[s], (u & 1u) ^ 1u, bars, p.status)) {
                if (lane == 0) {
                    reinterpret_cast<TileInfo *>(stage_ptr(s) + CF::OFF_INFO)->done = 1;
                    mbar_arrive(&bars->full[s]);
                }
            } else {
                ok = false;
            }
        }
        // after a timeout: our last TMA loads must land before shared memory is released
        // (on the normal path every load was consumed through its full barrier)
        if (!ok && lane == 0) {
            for (int back = 1; back <= NS && back <= i; ++back) {
                const int j = i - back;
                volatile int never = 0;
                mbar_wait(&bars->full[j % NS], (uint32_t)(j / NS) & 1u, &never, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ MMA issuer
        const uint32_t idesc_gram = idesc_bf16_f32(128, 128, 0, 0);
        const uint32_t idesc_epi = idesc_bf16_f32(128, 256, 0, 1);
        auto zero_tail = [&](uint8_t *st, int Lc) {
            // rows Lc..C-1 of every head's K and V boxes
            const int rows = C - Lc;
            const int per_box = rows * 8;  // 16-byte chunks
            for (int e = lane; e < G * 4 * per_box; e += 32) {
                const int box = e / per_box, w = e % per_box;
                const int g = box % G, kvh = box / G;  // kvh: 0,1 = K halves, 2,3 = V halves
                uint8_t *b = st + kvh * 16384 + g * C * 128;
                *reinterpret_cast<uint4 *>(b + (Lc + w / 8) * 128 + (w % 8) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
        };
        auto issue_gram = [&](uint8_t *st) {
            if (lane == 0) {
                tc_fence_after();
                const uint32_t a0 = smem_u32(st);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t d = sw128_desc(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    mma_ss(tmem + kColGram, d, d, idesc_gram, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars->gram_full);
            }
            __syncwarp();
        };
        auto issue_epi = [&](uint8_t *st) {
            if (lane == 0) {
                tc_fence_after();
                const uint32_t b0 = smem_u32(st);
#pragma unroll
                for (int pass = 0; pass < 2; ++pass)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t d = sw128_desc(b0 + kk * 2048, 16384, 1024);
                        mma_ts(tmem + kColD, tmem + kColTT + pass * 64 + kk * 8, d, idesc_epi,
                               (pass | kk) ? 1u : 0u);
                    }
                mma_commit(&bars->tt_empty);
                mma_commit(&bars->d_full);
            }
            __syncwarp();
        };
        int i = 0;
        bool ok = wait_bar(&bars->full[0], 0u, bars, p.status);
        const TileInfo *info0 = reinterpret_cast<const TileInfo *>(stage_ptr(0) + CF::OFF_INFO);
        bool have = ok && !info0->done;
        if (have) {
            if (info0->Lc < C) zero_tail(stage_ptr(0), info0->Lc);
            ok = wait_bar(&bars->gram_empty, 1u, bars, p.status);
            if (ok) issue_gram(stage_ptr(0));
        }
        while (ok && have) {
            const int n = i + 1;
            const int sn = n % NS;
            ok = wait_bar(&bars->full[sn], (uint32_t)(n / NS) & 1u, bars, p.status);
            if (!ok) break;
            const TileInfo *infn = reinterpret_cast<const TileInfo *>(stage_ptr(sn) + CF::OFF_INFO);
            const bool has_next = !infn->done;
            if (has_next) {
                if (infn->Lc < C) zero_tail(stage_ptr(sn), infn->Lc);
                ok = wait_bar(&bars->gram_empty, ((uint32_t)n & 1u) ^ 1u, bars, p.status);
                if (!ok) break;
                issue_gram(stage_ptr(sn));
            }
            ok = wait_bar(&bars->tt_full, (uint32_t)i & 1u, bars, p.status) &&
                 wait_bar(&bars->d_empty, ((uint32_t)i & 1u) ^ 1u, bars, p.status);
            if (!ok) break;
            issue_epi(stage_ptr(i % NS));
            i = n;
            have = has_next;
        }
        // every MMA issued by this thread has completed before tensor memory is freed
        if (lane == 0) {
            mma_commit(&bars->mma_final);
            volatile int never = 0;
            mbar_wait(&bars->mma_final, 0u, &never, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= kWarpInv0 && warp < kWarpInv0 + 4) {
        // ------------------------------------------------------------------ inverse warps
        const int q = warp & 3;             // tensor-memory lane quarter
        const int m = 32 * q + lane;        // tile row
        const int g = m / C;                // head within the tile
        const int r = m % C;                // row within the chunk
        const int wp = r / 32;              // warp position within the head (0 for C = 32)
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        uint8_t *tstage = smem + CF::OFF_T;
        // zero this lane's T~ columns (other heads' blocks and the upper triangle stay zero)
        {
            uint32_t zz[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) zz[c] = 0u;
#pragma unroll
            for (int c = 0; c < 128; c += 16) tmem_st16(tmem + lane_base + kColTT + c, zz);
            tmem_wait_st();
            for (int h = 0; h < CF::T_HALVES; ++h)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(tstage + h * 16384 + m * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
        int i = 0;
        uint32_t inv_uses = 0, pair_uses = 0;
        while (true) {
            const int s = i % NS;
            if (!wait_bar(&bars->full[s], (uint32_t)(i / NS) & 1u, bars, p.status)) break;
            const uint8_t *st = stage_ptr(s);
            const TileInfo info = *reinterpret_cast<const TileInfo *>(st + CF::OFF_INFO);
            if (info.done) break;
            const float *sb = reinterpret_cast<const float *>(st + CF::OFF_BETA) + g * C;
            const float beta_r = sb[r];

            if (!wait_bar(&bars->gram_full, (uint32_t)i & 1u, bars, p.status)) break;
            tc_fence_after();
            // Gram row -> strictly-lower L row (beta on rows, §3.2); only columns < 32 (wp + 1) matter
            float l[C >= 64 ? 64 : 32];
            {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kColGram + g * C, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) l[j] = (j < r) ? beta_r * __uint_as_float(v[j]) : 0.f;
                if constexpr (C >= 64) {
                    tmem_ld32(tmem + lane_base + kColGram + g * C + 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) l[32 + j] = (32 + j < r) ? beta_r * __uint_as_float(v[j]) : 0.f;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->gram_empty);

            // this warp's 32-column slab of L: columns 32 wp .. 32 wp + 31
            float slab[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if constexpr (C >= 64) slab[j] = wp ? l[32 + j] : l[j];
                else slab[j] = l[j];
            }
            // diagonal 16 x 16 block of this half warp
            const bool upper = lane >= 16;
            float lb[16], x[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) lb[c] = upper ? slab[16 + c] : slab[c];
            diag16(lb, x, lane);
            // level 16: couple the warp's two diagonal blocks
            float l10[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) l10[c] = slab[c];
            float m32[32];
            couple16(l10, x, lane, m32);

            // the lane's row of T over columns 0 .. C-1 (zero above the diagonal)
            float trow[C >= 64 ? 64 : 32];
            if constexpr (C >= 64) {
                // level 32: rows 32..63 of the head get -M11^-1 M10 M00^-1, with M00^-1 rows
                // shared by the lower warp through shared memory
                float *xbuf = reinterpret_cast<float *>(smem + CF::OFF_XCH) + g * 3072 + (i & 1) * 1024;
                float *ybuf = reinterpret_cast<float *>(smem + CF::OFF_XCH) + g * 3072 + 2048;
                if (wp == 0) {
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4 *>(xbuf + lane * 32 + c) =
                            make_float4(m32[c], m32[c + 1], m32[c + 2], m32[c + 3]);
                }
                if (!group_sync(&bars->pair_sync[g], pair_uses, bars, p.status)) break;
                if (wp == 1) {
                    float y[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) y[c] = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float lj = l[j];
#pragma unroll
                        for (int c = 0; c <= (j | 3); c += 4) {
                            const float4 xv = *reinterpret_cast<const float4 *>(xbuf + j * 32 + c);
                            y[c] = fmaf(lj, xv.x, y[c]);
                            y[c + 1] = fmaf(lj, xv.y, y[c + 1]);
                            y[c + 2] = fmaf(lj, xv.z, y[c + 2]);
                            y[c + 3] = fmaf(lj, xv.w, y[c + 3]);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4 *>(ybuf + lane * 32 + c) = make_float4(y[c], y[c + 1], y[c + 2], y[c + 3]);
                    __syncwarp();
                    float z[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) z[c] = 0.f;
#pragma unroll
                    for (int k2 = 0; k2 < 32; ++k2) {
                        const float mk = m32[k2];
#pragma unroll
                        for (int c = 0; c < 32; c += 4) {
                            const float4 yv = *reinterpret_cast<const float4 *>(ybuf + k2 * 32 + c);
                            z[c] = fmaf(mk, yv.x, z[c]);
                            z[c + 1] = fmaf(mk, yv.y, z[c + 1]);
                            z[c + 2] = fmaf(mk, yv.z, z[c + 2]);
                            z[c + 3] = fmaf(mk, yv.w, z[c + 3]);
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        trow[c] = -z[c];
                        trow[32 + c] = m32[c];
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        trow[c] = m32[c];
                        trow[32 + c] = 0.f;
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) trow[c] = m32[c];
            }

            // T rows: staging + TMA store for a full chunk, plain stores for a short one
            const bool full_chunk = info.Lc == C;
            if (full_chunk) {
                if (threadIdx.x == kWarpInv0 * 32) bulk_wait_read<0>();
                if (!group_sync(&bars->inv_sync, inv_uses, bars, p.status)) break;
#pragma unroll
                for (int h = 0; h < CF::T_HALVES; ++h) {
                    if (h <= wp) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint32_t off = sw128((uint32_t)(m * 128 + c * 16));
                            *reinterpret_cast<float4 *>(tstage + h * 16384 + off) =
                                make_float4(trow[32 * h + 4 * c], trow[32 * h + 4 * c + 1], trow[32 * h + 4 * c + 2],
                                            trow[32 * h + 4 * c + 3]);
                        }
                    }
                }
                fence_proxy_async_smem();
                if (!group_sync(&bars->inv_sync, inv_uses, bars, p.status)) break;
                if (threadIdx.x == kWarpInv0 * 32) {
                    for (int gg = 0; gg < G; ++gg)
                        for (int h = 0; h < CF::T_HALVES; ++h)
                            tma_store_3d(&map_t, tstage + h * 16384 + gg * C * 128, 32 * h, info.h0 + gg,
                                         (int)info.t0);
                    bulk_commit();
                }
            } else if (r < info.Lc && info.h0 + g < p.H) {
                float4 *dst = reinterpret_cast<float4 *>(p.T_out + ((info.t0 + r) * p.H + info.h0 + g) * C);
#pragma unroll
                for (int c = 0; c < C / 4; ++c)
                    dst[c] = make_float4(trow[4 * c], trow[4 * c + 1], trow[4 * c + 2], trow[4 * c + 3]);
            }

            // T~ = T diag(beta), split into bf16 hi + lo, into tensor memory (A operand)
            if (!wait_bar(&bars->tt_empty, ((uint32_t)i & 1u) ^ 1u, bars, p.status)) break;
            tc_fence_after();
            {
                constexpr int NJ = C >= 64 ? 64 : 32;
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int blk = 0; blk < NJ / 32; ++blk) {
                    if (blk <= wp) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int j = 32 * blk + 2 * c;
                            const float a = trow[j] * sb[j];
                            const float b = trow[j + 1] * sb[j + 1];
                            const __nv_bfloat16 ah = __float2bfloat16_rn(a), bh = __float2bfloat16_rn(b);
                            hi[c] = (uint32_t)__bfloat16_as_ushort(ah) | ((uint32_t)__bfloat16_as_ushort(bh) << 16);
                            lo[c] = pack_bf16(a - __bfloat162float(ah), b - __bfloat162float(bh));
                        }
                        const uint32_t col = (uint32_t)(g * C + 32 * blk) / 2;
                        tmem_st16(tmem + lane_base + kColTT + col, hi);
                        tmem_st16(tmem + lane_base + kColTT + 64 + col, lo);
                    }
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tt_full);
            ++i;
        }
        if (threadIdx.x == kWarpInv0 * 32) bulk_wait<0>();
        __syncwarp();
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
        // ------------------------------------------------------------------ epilogue warps
        const int q = warp & 3;
        const int m = 32 * q + lane;
        const int g = m / C;
        const int r = m % C;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        int i = 0;
        uint32_t epi_uses = 0;
        while (true) {
            const int s = i % NS;
            if (!wait_bar(&bars->full[s], (uint32_t)(i / NS) & 1u, bars, p.status)) break;
            uint8_t *st = stage_ptr(s);
            const TileInfo info = *reinterpret_cast<const TileInfo *>(st + CF::OFF_INFO);
            if (info.done) break;
            if (!wait_bar(&bars->d_full, (uint32_t)i & 1u, bars, p.status)) break;
            tc_fence_after();
            const bool full_chunk = info.Lc == C;
            const bool row_ok = r < info.Lc && info.h0 + g < p.H;
            const int64_t grow = (info.t0 + r) * p.H + info.h0 + g;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {  // 32 fp32 columns of D at a time: W cols 0..127, U~ 128..255
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kColD + 32 * c, v);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                const int n0 = 32 * c;              // first column in [W | U~]
                const int kv = n0 / 128;            // 0: W, 1: U~
                const int half = (n0 % 128) / 64;   // 64-column box
                const int cb = (n0 % 64) * 2;       // byte offset inside the 128-byte row
                if (full_chunk) {
                    uint8_t *dst = st + kv * 32768 + half * 16384;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        *reinterpret_cast<uint4 *>(dst + sw128((uint32_t)(m * 128 + cb + 16 * e))) =
                            make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                } else if (row_ok) {
                    __nv_bfloat16 *base = (kv == 0 ? p.W_out : p.U_out) + grow * 128 + (n0 % 128);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        reinterpret_cast<uint4 *>(base)[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->d_empty);
            if (full_chunk) fence_proxy_async_smem();
            if (!group_sync(&bars->epi_sync, epi_uses, bars, p.status)) break;
            if (threadIdx.x == kWarpEpi0 * 32) {
                if (full_chunk) {
                    for (int gg = 0; gg < G; ++gg)
                        for (int h = 0; h < 2; ++h) {
                            tma_store_3d(&map_w, st + h * 16384 + gg * C * 128, 64 * h, info.h0 + gg, (int)info.t0);
                            tma_store_3d(&map_u, st + 32768 + h * 16384 + gg * C * 128, 64 * h, info.h0 + gg,
                                         (int)info.t0);
                        }
                    bulk_commit();
                    bulk_wait_read<0>();
                }
                mbar_arrive(&bars->empty[s]);
            }
            ++i;
        }
        if (threadIdx.x == kWarpEpi0 * 32) bulk_wait<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [ntok][H][inner] row-major, box {box_inner, 1, rows}, 128-byte swizzle.
bool make_map(CUtensorMap *map, CUtensorMapDataType dt, int esize, const void *ptr, int64_t ntok, int H, int inner,
              int box_inner, int rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)H, (cuuint64_t)ntok};
    cuuint64_t strides[2] = {(cuuint64_t)inner * esize, (cuuint64_t)H * inner * esize};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, 1u, (cuuint32_t)rows};
    cuuint32_t es[3] = {1u, 1u, 1u};
    return enc(map, dt, 3, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

template <int C>
int launch_tc_t(const Problem &pb) {
    using CF = Cfg<C>;
    CUtensorMap mk, mv, mw, mu, mt;
    if (!make_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pb.k, pb.ntok, pb.H, pb.dk, 64, C) ||
        !make_map(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pb.v, pb.ntok, pb.H, pb.dv, 64, C) ||
        !make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pb.W_out, pb.ntok, pb.H, pb.dk, 64, C) ||
        !make_map(&mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pb.U_out, pb.ntok, pb.H, pb.dv, 64, C) ||
        !make_map(&mt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pb.T_out, pb.ntok, pb.H, C, 32, C))
        return KKT_ERR_CUDA;
    TcParams p;
    p.beta = pb.beta;
    p.cu = pb.cu_seqlens;
    p.nseq = pb.nseq;
    p.T = pb.T;
    p.ntok = pb.ntok;
    p.H = pb.H;
    p.HG = (pb.H + CF::G - 1) / CF::G;
    p.tiles = total_work_ids(pb.ntok, C, pb.nseq) * p.HG;
    p.T_out = pb.T_out;
    p.W_out = static_cast<__nv_bfloat16 *>(pb.W_out);
    p.U_out = static_cast<__nv_bfloat16 *>(pb.U_out);
    p.status = pb.status;
    auto kern = kkt_tc_kernel<C>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_BYTES) != cudaSuccess)
        return KKT_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return KKT_ERR_CUDA;
    const int64_t grid = p.tiles < sms ? p.tiles : sms;
    kern<<<(unsigned)grid, kThreads, CF::SMEM_BYTES, pb.stream>>>(mk, mv, mw, mu, mt, p);
    return cudaGetLastError() == cudaSuccess ? KKT_OK : KKT_ERR_CUDA;
}

}  // namespace

bool tc_supports(int dk, int dv, int C, int io) {
    return io == KKT_IO_BF16 && dk == 128 && dv == 128 && (C == 32 || C == 64);
}

int launch_tc(const Problem &p) {
    switch (p.C) {
        case 32: return launch_tc_t<32>(p);
        case 64: return launch_tc_t<64>(p);
        default: return KKT_ERR_UNSUPPORTED;
    }
}

}  // namespace kkt
