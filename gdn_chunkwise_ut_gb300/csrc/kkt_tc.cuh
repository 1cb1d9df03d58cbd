// kkt_tc.cuh -- persistent, warp-specialised tcgen05 + TMA kernel for kkt_solve (bf16 I/O),
// templated on the chunk size C and the head dimensions d_k and d_v (64 or 128 each).  Included by
// one translation unit per (d_k, d_v) pair (kkt_tc.cu: 128 / 128, kkt_tc_d64.cu: 64 / 64,
// kkt_tc_k128v64.cu and kkt_tc_k64v128.cu: the mixed pairs), which compile in parallel; everything
// here has internal linkage.
//
// One CTA per SM walks "tiles" of 128 rows: G = 128 / C heads of one chunk,
// row m = g * C + r (head g, token r of the chunk).  For each tile
// ("TileLang 实战：单位下三角矩阵求逆" §1, §2.2, §3):
//
//   producer warp   TMA: K and V boxes {64 cols, 1 head, C rows} (128-byte
//                   swizzle) into a stage of a two-deep shared-memory ring;
//                   beta (and the gate's prefix sums, gated kernels) with plain
//                   loads.
//   Gram warp       one lane issuing tcgen05.mma S = K K^T (M = N = 128,
//                   K = d_k, bf16 -> fp32 in tensor memory); zeroes the rows past
//                   a short chunk's end first.
//   W|U warp        one lane issuing D = T~ [K | V] with T~ = T diag(beta) read
//                   from tensor memory as a bf16 hi + lo pair (two accumulating
//                   passes, M = 128, N = d_k + d_v, K = 128; T~ is block diagonal over
//                   the G heads).  The commit after D frees the stage.
//   inverse warps   a thread per row loads its Gram row (tcgen05.ld), applies
//                   the beta row scale, strict-lower mask and unit diagonal
//                   (§3.2) and writes the row of A into the tile's fp32 T
//                   buffer in shared memory (128-byte swizzle, TMA layout),
//                   which is then turned into T = A^-1 in place:
//                   16 x 16 diagonal blocks by right-looking forward
//                   substitution, one column per lane, so the dependency chain
//                   is 15 FMAs (§2.1; in-place, with the L values read before
//                   any column is written back, §3.4); coupling
//                   -L11^-1 L10 L00^-1 at s = 16 (inside a warp) and s = 32 (the
//                   two warps of a 64-row block) as register-tiled shared-memory
//                   GEMMs with L10 consumed before it is overwritten (§2.2,
//                   §3.5); at C = 128, s = 64 as two 3-pass bf16 tcgen05 MMAs
//                   that the W|U warp issues between the tile's conversions of
//                   their operands.  Each warp TMA-stores its 32 rows of T from that
//                   buffer, and writes its rows of T~ = T diag(beta) as a bf16
//                   hi / lo pair into tensor memory (tcgen05.st).
//   epilogue warps  per warp: tcgen05.ld of its 32 rows of D, bf16 conversion,
//                   a swizzled staging (double-buffered at C <= 64) and TMA
//                   stores of W, U~.  Gated, they also scale the stage's K rows
//                   by the decay from the chunk's start; at C = 128 the two of
//                   lanes 64..127 form M10 from the Gram into tensor memory for
//                   the level-64 MMA.
//
// Rows of a short last chunk (Lc < C) past Lc are zeroed in shared memory
// before the Gram MMA; warps whose 32 rows are not all valid write their valid
// rows with plain stores.  Every wait is bounded: on expiry the kernel records
// KKT_ERR_TIMEOUT, stops all roles, drains its own copies and MMAs, frees
// tensor memory and returns.
//
// The warp index is broadcast from lane 0 and every bounded wait votes its result over the warp,
// so the compiler sees the role loops and the per-warp branches as warp-uniform; that alone took
// about 6 % off the bench workload.
//
// Building with -DKKT_TRACE adds time stamps of the pipeline events of the
// first CTAs to a caller-provided buffer (see trace.py); the default build has
// none of it.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kkt_debug.cuh"
#include "kkt_internal.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace kkt {
namespace {

using namespace ptx;

constexpr int kThreads = 384;            // 12 warps
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;              // W|U MMAs
constexpr int kWarpGram = 2;             // Gram MMAs
constexpr int kWarpInv0 = 4;             // warps 4..7
constexpr int kWarpEpi0 = 8;             // warps 8..11
constexpr int kNS = 2;                   // stages
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColGram = 0;         // 128 fp32 columns
constexpr uint32_t kColD = 128;          // 256 fp32 columns: W | U~
constexpr uint32_t kColTT = 384;         // 64 packed bf16x2 hi + 64 lo
// C = 128, level 64 on the tensor core.  The A operands as packed bf16 hi + lo pairs (32 + 32
// columns, lanes 64..127): M10 in T~'s columns (free once the previous tile's W|U MMA has read T~),
// M11^-1 in the Gram's columns 64..127 (in those lanes only read by the warps of rows 64..127 when
// they form A; the next Gram MMA waits for Z); the fp32 products Y, then Z, in the other 64 columns
// of T~'s.
constexpr uint32_t kColL64M10 = kColTT;
constexpr uint32_t kColL64M11 = kColGram + 64;
constexpr uint32_t kColL64D = kColTT + 64;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

struct TileInfo {
    int64_t t0;
    int Lc;
    int h0;
    int done;
    int pad;
};

template <int C, int DK, int DV>
struct Cfg {
    static constexpr int G = 128 / C;                         // heads per tile
    static constexpr int NBK = DK / 64;                        // 64-column TMA boxes per K row
    static constexpr int NBV = DV / 64;                        // and per V row
    static constexpr int NBKV = NBK + NBV;
    static constexpr int KV_BYTES = NBKV * 16384;             // K then V boxes, [box][row][128 B]
    // per stage: beta[128]; gated kernels: the gate's prefix sums G[128] (log2 units), the column
    // factors w[128] and one "factorable" flag per 32-row block (int[4]); then the TileInfo
    static constexpr int META_BYTES = 1584;
    static constexpr int T_HALVES = C / 32;                   // 128-byte column blocks of a T row
    static constexpr int OFF_T = kNS * KV_BYTES;              // T of the tile: [half][128 rows][128 B]
    // W / U~ staging per epilogue warp: two 4 KB buffers, one at C = 128 (whose T takes 64 KB)
    static constexpr int WU_BUFS = C == 128 ? 1 : 2;
    static constexpr int OFF_WU = OFF_T + T_HALVES * 16384;
    static constexpr int OFF_META = OFF_WU + 4 * WU_BUFS * 4096;  // per stage: beta[128] + TileInfo
    static constexpr int OFF_BAR = OFF_META + kNS * META_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TX_BYTES = G * NBKV * C * 128;        // K + V boxes of one stage
    static_assert(SMEM_BYTES <= 232448, "shared memory over the per-block limit");
};

struct Barriers {
    uint64_t full[kNS];
    uint64_t empty[kNS];
    uint64_t gram_full, gram_empty;
    uint64_t tt_full, tt_empty;
    uint64_t d_full, d_empty;
    uint64_t einfo_full[2];
    uint64_t mma_final, gram_final;
    uint64_t pair_sync[2];   // warps 2p and 2p + 1: one 64-row block (C = 64, 128)
    uint64_t l64_ops;        // C = 128: the operands of Y = M10 M00^-1 are in place (inverse warps 0, 1
                             // and epilogue warps 2, 3)
    uint64_t l64_y;          // C = 128: Y is in tensor memory (MMA commit)
    uint64_t l64_yb;         // C = 128: Y, the B operand of Z, is in shared memory (warps 2, 3)
    uint64_t l64_z;          // C = 128: Z = M11^-1 Y is in tensor memory (MMA commit)
    uint64_t kread[kNS];     // gated: the Gram MMA of the stage's tile has read its K
    uint64_t kscaled;        // gated: the epilogue warps have scaled the tile's K rows for W
    TileInfo einfo[2];       // tile info for the epilogue warps, written by the W|U warp
    uint32_t tmem_base;
    int abort_flag;
};

struct TcParams {
    const float *beta;
    const float *g;  // per-token log decays (GATED kernels)
    const int32_t *cu;
    int nseq, T;
    int64_t ntok;
    int H;
    int64_t tiles;   // work ids x head groups
    int HG;          // head groups
    void *T_out;     // fp32, or fp16 in the TF16 kernels; nullptr: T is not written
    __nv_bfloat16 *W_out, *U_out;
    int *status;
    unsigned long long *trace;
    unsigned long long *tile_counter;  // dynamic scheduling when not null: [0] tiles claimed, [1] CTAs done
                                       // claiming; zero at launch, left zero by the last CTA
    int stall_first_tile;              // test hook: every CTA skips the loads of its first tile
};

// ---- optional pipeline trace ------------------------------------------------------------------
enum TraceEvent {
    EV_P_EMPTY = 0, EV_P_ISSUE, EV_M_FULL, EV_M_GRAM, EV_M_EPI, EV_I_GRAM, EV_I_INV, EV_I_TSTORE,
    EV_I_TT, EV_E_DFULL, EV_E_DEMPTY, EV_E_DONE, EV_I_LD, EV_I_DIAG, EV_I_C16, EV_I_PAIR, EV_M_LATE,
    EV_M_READY, EV_I_BW, EV_I_TTW, EV_I_L32,
    // C = 128, level 64: rows 64..127 (warp quarter 3) end level 32, have M11^-1 in tensor memory,
    // see Y, have Y's split in shared memory, see Z, end level 64; rows 0..63 (quarter 1) have split
    // M00^-1; the epilogue warp of quarter 3 has formed M10; the W|U thread issues Y, then Z
    EV_I_L32B, EV_I_M11, EV_I_Y, EV_I_YB, EV_I_Z, EV_I_INVB, EV_I_OPS, EV_E_M10, EV_M_L64Y, EV_M_L64Z,
    // ... and the shared-memory stores of M00^-1's split (quarter 1) and of Y's (quarter 3) are issued
    EV_I_SPLIT, EV_I_YSPL, EV_COUNT
};
constexpr int kTraceCtas = 160;
constexpr int kTraceTiles = 64;  // the last tile row holds the CTA's clock calibration
constexpr int kTraceSlots = 40;
static_assert(EV_COUNT <= kTraceSlots, "trace slots");
#ifdef KKT_TRACE
// SM cycle counter at each event; trace.py maps it to ns with the (globaltimer, clock) pairs that
// thread 0 records at the start and end of the CTA
#define KKT_TRACE_EVENT(ev, tile)                                                                        \
    do {                                                                                               \
        if (p.trace && blockIdx.x < kTraceCtas && (tile) < kTraceTiles - 1)                            \
            p.trace[((size_t)blockIdx.x * kTraceTiles + (tile)) * kTraceSlots + (ev)] = clock64();      \
    } while (0)
// the event row of a tile, for functions that record events without the kernel's parameters
#define KKT_TRACE_ROW(tile)                                                                              \
    ((p.trace && blockIdx.x < kTraceCtas && (tile) < kTraceTiles - 1)                                  \
         ? p.trace + ((size_t)blockIdx.x * kTraceTiles + (tile)) * kTraceSlots                         \
         : nullptr)
#define KKT_TRACE_AT(row, ev)                 \
    do {                                      \
        if (row) (row)[(ev)] = clock64();     \
    } while (0)
#define KKT_TRACE_CALIB(slot)                                                                            \
    do {                                                                                               \
        if (p.trace && blockIdx.x < kTraceCtas && threadIdx.x == 0) {                                  \
            unsigned long long *c = p.trace + ((size_t)blockIdx.x * kTraceTiles + kTraceTiles - 1) * kTraceSlots; \
            c[2 * (slot)] = globaltimer_ns();                                                          \
            c[2 * (slot) + 1] = clock64();                                                             \
        }                                                                                              \
    } while (0)
#else
#define KKT_TRACE_EVENT(ev, tile) \
    do {                          \
    } while (0)
#define KKT_TRACE_ROW(tile) (static_cast<unsigned long long *>(nullptr))
#define KKT_TRACE_AT(row, ev) \
    do {                      \
    } while (0)
#define KKT_TRACE_CALIB(slot) \
    do {                      \
    } while (0)
#endif

// First 1024-byte-aligned byte of the dynamic shared memory.  The offset is
// computed in the shared window and added to the shared pointer itself, so the
// compiler keeps the shared address space (LDS/STS rather than generic loads).
__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    const uint32_t a = smem_u32(p);
    return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ void fail(Barriers *bars, int *status) {
    if (atomicExch(&bars->abort_flag, 1) == 0) record_error(status, KKT_ERR_TIMEOUT);
}

// Called by every lane of a warp (all callers are whole warps).  The result is made warp-uniform,
// so that a timeout seen by one lane is taken by all before the .sync.aligned instructions after it.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, Barriers *bars, int *status) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, &bars->abort_flag, kWaitLimitNs));
    if (!ok) fail(bars, status);
    return ok;
}

// Group barrier on an mbarrier (every member arrives, then waits for the phase):
// unlike bar.sync it is bounded, so a member that gave up cannot hang the others.
__device__ __forceinline__ bool group_sync(uint64_t *bar, uint32_t &uses, Barriers *bars, int *status) {
    mbar_arrive(bar);
    const bool ok = wait_bar(bar, uses & 1u, bars, status);
    ++uses;
    return ok;
}

// Element (row m, column j) of a fp32 matrix stored as 32-column halves of 128-byte rows,
// [half][128 rows][128 B], with the 128-byte swizzle that TMA uses (16-byte chunk index XOR
// row mod 8): rows are conflict-free for a thread per row, and a row is a TMA box row.
__device__ __forceinline__ float *tm_elem(uint8_t *tm, int m, int j) {
    return smem_chk(reinterpret_cast<float *>(tm + (j >> 5) * 16384 + m * 128 + ((((j & 31) >> 2) ^ (m & 7)) << 4) +
                                              (j & 3) * 4));
}
__device__ __forceinline__ float4 *tm_vec(uint8_t *tm, int m, int j) {  // j a multiple of 4
    return smem_chk(reinterpret_cast<float4 *>(tm + (j >> 5) * 16384 + m * 128 + ((((j & 31) >> 2) ^ (m & 7)) << 4)));
}

// Two fp16 (round to nearest even) in the bits of one float: lo in bits 0..15, hi in 16..31.
__device__ __forceinline__ float pack_f16(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return __uint_as_float(*reinterpret_cast<const uint32_t *>(&v));
}

// Two bf16 (round to nearest even) in one register: lo in bits 0..15, hi in 16..31.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Packed fp32 product of a pair (one f32x2 instruction): a * b, elementwise.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// A bf16 pair times a bf16 pair of factors, the products rounded to nearest (one packed multiply).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Packed fp32 FMA on a pair (one f32x2 instruction): a * b + c, elementwise.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// bf16 hi + lo split of a pair, packed as two bf16x2 words: hi = bf16(x), lo = bf16(x - hi)
// (the difference is exact in fp32).
__device__ __forceinline__ void split_bf16(float2 x, uint32_t &hi, uint32_t &lo) {
    const uint32_t h = pack_bf16(x.x, x.y);
    const float2 hf = make_float2(__uint_as_float(h << 16), __uint_as_float(h & 0xffff0000u));
    hi = h;
    const float2 r = ffma2(hf, make_float2(-1.f, -1.f), x);
    lo = pack_bf16(r.x, r.y);
}

// D (4 x 4 tile, as 4 rows x 2 packed pairs) += A B over NKB blocks of 8 k.  A rows: byte pointers to
// the start of the rows' 128-byte lines in the k range's half, with their swizzle phases as XOR
// masks; acol0 is the first k column (a multiple of 8) inside that half.  B rows: base pointer of
// row 0 of the k range (its row index a multiple of 8), bsw[kk] the byte offset of this lane's
// 16-byte column chunk in a row with phase kk.
// A loop over 8-k blocks rather than an unrolled sequence: the kernel is sensitive to its
// instruction-cache footprint, so the code size of this inner product is kept small (UNROLL
// blocks per iteration: 1 at C <= 64, 2 at C = 128).
template <int UNROLL>
__device__ __forceinline__ void tile4x4_fma(float2 (&y)[4][2], const uint8_t *const (&arow)[4],
                                         const uint32_t (&axor)[4], int acol0, const uint8_t *brow0,
                                         const uint32_t (&bsw)[8], int nkb) {
#pragma unroll UNROLL
    for (int kb = 0; kb < nkb; ++kb) {
        float av[4][8];
        const uint32_t ca = (uint32_t)((acol0 >> 2) + 2 * kb) << 4;
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const float4 a0 = *smem_chk(reinterpret_cast<const float4 *>(arow[rr] + (ca ^ axor[rr])));
            const float4 a1 = *smem_chk(reinterpret_cast<const float4 *>(arow[rr] + ((ca + 16u) ^ axor[rr])));
            av[rr][0] = a0.x; av[rr][1] = a0.y; av[rr][2] = a0.z; av[rr][3] = a0.w;
            av[rr][4] = a1.x; av[rr][5] = a1.y; av[rr][6] = a1.z; av[rr][7] = a1.w;
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const float4 b = *smem_chk(reinterpret_cast<const float4 *>(brow0 + (8 * kb + kk) * 128 + bsw[kk]));
            const float2 b01 = make_float2(b.x, b.y), b23 = make_float2(b.z, b.w);
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const float2 ak = make_float2(av[rr][kk], av[rr][kk]);
                y[rr][0] = ffma2(ak, b01, y[rr][0]);
                y[rr][1] = ffma2(ak, b23, y[rr][1]);
            }
        }
    }
}

// Level-32 coupling of one 64 x 64 diagonal block (rows m0 .. m0 + 63, columns c0 .. c0 + 63 of
// the chunk, in the tile's T buffer) for warp WP (0 or 1) of its two warps.  With 16 x 16 blocks
// M00^-1 = [[A, 0], [Cb, D]], M10 = [P, Q], M11^-1 = [[A', 0], [Cb', D']]:
// Y = M10 M00^-1 = [P A + Q Cb, Q D] and Z = M11^-1 Y = [A' Y_top ; Cb' Y_top + D' Y_bot].
// Warp 0 computes Y_left (K = 32) and Z_top (K = 16), warp 1 Y_right (K = 16) and Z_bot (K = 32):
// the zero blocks are skipped and both warps do 384 packed FMAs per lane.  Rows 32..63, columns
// 0..31 of the block receive -Z.  ybuf32 points at row 0 of the block's upper-right 32 x 32 (rows
// 0..31, columns 32..63 of the block, zero in T), which holds Y and is cleared again at the end.
template <int UNROLL>
__device__ __forceinline__ bool level32(const int WP, uint8_t *tm, uint8_t *ybuf32, int m0, int c0, int lane,
                                        uint64_t *pair_bar, uint32_t &pair_uses, Barriers *bars, int *status) {
    uint8_t *th = tm + (c0 >> 5) * 16384;  // the 32-column half holding the block's first columns
    {
        // Y part: rows yr + 8 rr of 32, columns 16 WP + 4 yc .. + 3; k in [16 WP, 32).  A quarter-warp
        // covers 8 rows of one column group: 8 different swizzled chunks, no bank conflict
        const int yr = lane & 7, yc = lane >> 3;
        const uint8_t *arow[4];
        uint32_t axor[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            arow[rr] = th + (m0 + 32 + yr + 8 * rr) * 128;
            axor[rr] = (uint32_t)(yr & 7) << 4;
        }
        uint32_t bsw[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) bsw[kk] = (uint32_t)((4 * WP + yc) ^ kk) << 4;
        float2 y[4][2];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) y[rr][0] = y[rr][1] = make_float2(0.f, 0.f);
        tile4x4_fma<UNROLL>(y, arow, axor, 16 * WP, th + (m0 + 16 * WP) * 128, bsw, 4 - 2 * WP);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
            *tm_vec(ybuf32, yr + 8 * rr, 16 * WP + 4 * yc) = make_float4(y[rr][0].x, y[rr][0].y, y[rr][1].x, y[rr][1].y);
    }
    if (!group_sync(pair_bar, pair_uses, bars, status)) return false;
    {
        // Z part: rows 16 WP + zr + 4 rr (zr = 0..3), columns 4 zc .. + 3 (zc = 0..7); k in [0, 16 + 16 WP)
        const int zr = lane >> 3, zc = lane & 7;
        const uint8_t *arow[4];
        uint32_t axor[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int row = m0 + 32 + 16 * WP + zr + 4 * rr;
            arow[rr] = th + 16384 + row * 128;  // columns 32..63 of the block: the next half
            axor[rr] = (uint32_t)(row & 7) << 4;
        }
        uint32_t bsw[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) bsw[kk] = (uint32_t)(zc ^ kk) << 4;
        float2 z[4][2];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) z[rr][0] = z[rr][1] = make_float2(0.f, 0.f);
        tile4x4_fma<UNROLL>(z, arow, axor, 0, ybuf32, bsw, 2 + 2 * WP);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
            *tm_vec(tm, m0 + 32 + 16 * WP + zr + 4 * rr, c0 + 4 * zc) =
                make_float4(-z[rr][0].x, -z[rr][0].y, -z[rr][1].x, -z[rr][1].y);
    }
    if (!group_sync(pair_bar, pair_uses, bars, status)) return false;
    if (WP == 0) {
        // ybuf32 is the block's upper-right 32 x 32, zero in T: clear it again
#pragma unroll
        for (int j = 0; j < 32; j += 4) *tm_vec(ybuf32, lane, j) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    fence_proxy_async_smem();
    __syncwarp();
    return true;
}

// Gram row -> row m of A = I + strictLower(diag(beta) S) (beta on rows, unit diagonal, §3.2), times
// Gamma elementwise when gated (§5 item 12), into the T buffer: columns 32 h_lo .. 32 h_hi + 31.  r is
// the row's token within the chunk and gram the tensor-memory address of its head's Gram row.  When
// gated and every block of the head is factorable (fac), Gamma[r][j] for columns 32 h + c is
// exp2(G_r - R_h) w_j with R_h = G at the block's first row; otherwise the row is formed without it
// and multiplied by exp2(G_r - G_j) element by element after (a compact loop: such gates are rare,
// and the unrolled code stays small).  One 32-column block at a time, in a loop: the kernel is
// sensitive to its code size, and an unrolled form measured slower (gated) or the same.
template <bool GATED>
__device__ __forceinline__ void form_a_row(uint8_t *tm, uint32_t gram, int m, int r, int h_lo, int h_hi,
                                           float beta_r, bool fac, float g_r, const float *sg, const float *sw) {
#pragma unroll 1
    for (int h = h_lo; h <= h_hi; ++h) {
        uint32_t v[32];
        tmem_ld32(gram + 32 * h, v);
        float bu = beta_r;  // beta_r, times the block's row factor when gated
        float4 wq[8];
        if constexpr (GATED) {
            bu *= fac ? exp2f(g_r - *smem_chk(sg + 32 * h)) : 1.f;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                wq[c8] = fac ? *smem_chk(reinterpret_cast<const float4 *>(sw + 32 * h + 4 * c8)) : make_float4(1.f, 1.f, 1.f, 1.f);
        }
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            float e[4];
            float wj[4] = {1.f, 1.f, 1.f, 1.f};
            if constexpr (GATED) {
                const float4 w4 = wq[c / 4];
                wj[0] = w4.x; wj[1] = w4.y; wj[2] = w4.z; wj[3] = w4.w;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = 32 * h + c + u;
                e[u] = (j < r) ? bu * __uint_as_float(v[c + u]) * wj[u] : (j == r ? 1.f : 0.f);
            }
            *tm_vec(tm, m, 32 * h + c) = make_float4(e[0], e[1], e[2], e[3]);
        }
    }
    if constexpr (GATED) {
        if (!fac) {
            const int j_end = r < 32 * h_hi + 32 ? r : 32 * h_hi + 32;
#pragma unroll 1
            for (int j = 32 * h_lo; j < j_end; ++j) *tm_elem(tm, m, j) *= exp2f(g_r - *smem_chk(sg + j));
        }
    }
}

// Level-64 coupling of a 128-token chunk (C = 128; the tile's rows are the chunk's rows) (§2.2):
// rows 64..127, columns 0..63 receive -Z = -M11^-1 M10 M00^-1 with 64 x 64 blocks M00^-1 =
// T[0..63][0..63], M11^-1 = T[64..][64..] (both final after level 32) and M10 = L[64..][0..63].  The
// two products run on the tensor core as 3-pass bf16 MMAs (hi hi + hi lo + lo hi of a hi + lo split
// of each operand, fp32 accumulation; M = 128, N = 64, K = 64, lanes 0..63 of A and D unused):
//   Y = M10 M00^-1: A = M10 from tensor memory, B = M00^-1 (rows k, MN-major) in shared memory;
//   Z = M11^-1 Y:   A = M11^-1 from tensor memory, B = Y (rows k, MN-major) in shared memory.
// The B operands live in rows 0..63 of the T buffer's columns 64..127 (zero in T): hi in the third
// 32-column half, lo in the fourth, each row one 128-byte swizzled line of 64 bf16.  Warps 0 and 1
// write M00^-1 there and clear it again once Z is done.  The epilogue warps of lanes 64..127 form M10
// from the Gram rows straight into tensor memory as soon as the previous tile's W|U MMA has read T~,
// so that Y runs while warps 2 and 3 finish their level 32 (and those warps form only the diagonal
// half of their rows of A).  Warps 2 and 3 then put M11^-1 into the Gram's columns 64..127 of their
// lanes, turn Y into Z's B operand and write -Z into columns 0..63 of their rows.  The W|U issuer
// issues the MMAs; the next tile's Gram MMA waits for Z.

// bf16 hi + lo split of 8 fp32 values (two float4) into one 16-byte chunk of each.
__device__ __forceinline__ void split8(const float4 a, const float4 b, uint4 &hi, uint4 &lo) {
    split_bf16(make_float2(a.x, a.y), hi.x, lo.x);
    split_bf16(make_float2(a.z, a.w), hi.y, lo.y);
    split_bf16(make_float2(b.x, b.y), hi.z, lo.z);
    split_bf16(make_float2(b.z, b.w), hi.w, lo.w);
}

// Chunk c (columns 8 c .. 8 c + 7) of row k of a level-64 B operand: part 0 = hi, 1 = lo.
__device__ __forceinline__ uint4 *l64_b(uint8_t *tm, int part, int k, int c) {
    return smem_chk(reinterpret_cast<uint4 *>(tm + (2 + part) * 16384 + k * 128 + ((c ^ (k & 7)) << 4)));
}

// Row m of the T buffer, columns c0 .. c0 + 63, as a level-64 A operand in tensor memory: packed
// hi pairs in columns taddr .. + 31, lo pairs in taddr + 32 .. + 63 (this warp's lanes).
__device__ __forceinline__ void l64_row_to_tmem(uint8_t *tm, int m, int c0, uint32_t taddr) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
            const float4 a = *tm_vec(tm, m, c0 + 32 * h + c), b = *tm_vec(tm, m, c0 + 32 * h + c + 4);
            split_bf16(make_float2(a.x, a.y), hi[c / 2], lo[c / 2]);
            split_bf16(make_float2(a.z, a.w), hi[c / 2 + 1], lo[c / 2 + 1]);
            split_bf16(make_float2(b.x, b.y), hi[c / 2 + 2], lo[c / 2 + 2]);
            split_bf16(make_float2(b.z, b.w), hi[c / 2 + 3], lo[c / 2 + 3]);
        }
        tmem_st16(taddr + 16 * h, hi);
        tmem_st16(taddr + 32 + 16 * h, lo);
    }
}

// M10 row r (columns 0..63 of row r >= 64 of A: beta_r S[r][j], times Gamma[r][j] when gated, all
// strictly below the diagonal) from the Gram row in tensor memory straight into a level-64 A operand:
// packed hi pairs at taddr .. + 31, lo pairs at taddr + 32 .. + 63 (see form_a_row for Gamma).
template <bool GATED>
__device__ __forceinline__ void m10_from_gram(uint32_t gram, uint32_t taddr, int r, float beta_r, bool fac, float g_r,
                                              const float *sg, const float *sw) {
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld32(gram + 32 * h, v);
        float uh = beta_r;
        if constexpr (GATED) uh *= fac ? exp2f(g_r - *smem_chk(sg + 32 * h)) : 1.f;
        tmem_wait_ld();
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            float4 w4 = make_float4(1.f, 1.f, 1.f, 1.f);
            if constexpr (GATED) {
                if (fac) {
                    w4 = *smem_chk(reinterpret_cast<const float4 *>(sw + 32 * h + c));
                } else {
                    const float4 g4 = *smem_chk(reinterpret_cast<const float4 *>(sg + 32 * h + c));
                    w4 = make_float4(exp2f(g_r - g4.x), exp2f(g_r - g4.y), exp2f(g_r - g4.z), exp2f(g_r - g4.w));
                }
            }
            const float e0 = uh * __uint_as_float(v[c]) * w4.x, e1 = uh * __uint_as_float(v[c + 1]) * w4.y;
            const float e2 = uh * __uint_as_float(v[c + 2]) * w4.z, e3 = uh * __uint_as_float(v[c + 3]) * w4.w;
            split_bf16(make_float2(e0, e1), hi[c / 2], lo[c / 2]);
            split_bf16(make_float2(e2, e3), hi[c / 2 + 1], lo[c / 2 + 1]);
        }
        tmem_st16(taddr + 16 * h, hi);
        tmem_st16(taddr + 32 + 16 * h, lo);
    }
}

// One level-64 product (issuing thread): D = A B over K = 64 in three accumulating passes.
__device__ __forceinline__ void l64_mma(uint32_t d, uint32_t a, uint32_t b_smem) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 64, 0, 1);  // B MN-major: rows k of 64 bf16
#pragma unroll
    for (int pass = 0; pass < 3; ++pass)      // hi hi, hi lo, lo hi
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {      // K = 64 in steps of 16 (8 packed columns, 16 rows)
            const uint32_t ac = a + (pass == 2 ? 32u : 0u) + 8u * kk;
            const uint64_t bd = sw128_desc(b_smem + (pass == 1 ? 16384u : 0u) + 2048u * kk, 16384, 1024);
            mma_ts(d, ac, bd, idesc, (pass | kk) ? 1u : 0u);
        }
}

// The inverse warps' part of level 64 for tile i (q: the warp's row quarter, m its row).
__device__ __forceinline__ bool level64_tc(int q, int m, int i, uint8_t *tm, uint32_t tmem, uint32_t lane_base,
                                           int lane, Barriers *bars, int *status, unsigned long long *trow) {
    (void)trow;  // the tile's trace row (trace builds only)
    const bool tr = (q == 1 || q == 3) && lane == 0;
    const uint32_t ph = (uint32_t)i & 1u;
    if (q < 2) {
        // M00^-1 row m (= row k of Y's B operand), split into hi + lo
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 hi, lo;
            split8(*tm_vec(tm, m, 8 * c), *tm_vec(tm, m, 8 * c + 4), hi, lo);
            *l64_b(tm, 0, m, c) = hi;
            *l64_b(tm, 1, m, c) = lo;
        }
        if (tr) KKT_TRACE_AT(trow, EV_I_SPLIT);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->l64_ops);
        if (tr) KKT_TRACE_AT(trow, EV_I_OPS);
        // Z done: the B operand area is read, and is cleared again (the upper right of T is zero)
        if (!wait_bar(&bars->l64_z, ph, bars, status)) return false;
#pragma unroll
        for (int j = 64; j < 128; j += 4) *tm_vec(tm, m, j) = make_float4(0.f, 0.f, 0.f, 0.f);
        return true;
    }
    // M11^-1 (columns 64..127) into the Gram's columns 64..127, which this warp read when it formed A
    l64_row_to_tmem(tm, m, 64, tmem + lane_base + kColL64M11);
    if (tr) KKT_TRACE_AT(trow, EV_I_M11);
    // Y row m - 64 -> row k = m - 64 of Z's B operand
    if (!wait_bar(&bars->l64_y, ph, bars, status)) return false;
    tc_fence_after();
    if (tr) KKT_TRACE_AT(trow, EV_I_Y);
    const int k = m - 64;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kColL64D + 32 * h, v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint4 hi, lo;
            split8(make_float4(__uint_as_float(v[8 * c]), __uint_as_float(v[8 * c + 1]), __uint_as_float(v[8 * c + 2]),
                               __uint_as_float(v[8 * c + 3])),
                   make_float4(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5]),
                               __uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])),
                   hi, lo);
            *l64_b(tm, 0, k, 4 * h + c) = hi;
            *l64_b(tm, 1, k, 4 * h + c) = lo;
        }
    }
    if (tr) KKT_TRACE_AT(trow, EV_I_YSPL);
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->l64_yb);
    if (tr) KKT_TRACE_AT(trow, EV_I_YB);
    // -Z into columns 0..63 of the row (M10 was formed straight into tensor memory, not here)
    if (!wait_bar(&bars->l64_z, ph, bars, status)) return false;
    tc_fence_after();
    if (tr) KKT_TRACE_AT(trow, EV_I_Z);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kColL64D + 32 * h, v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 4)
            *tm_vec(tm, m, 32 * h + c) = make_float4(-__uint_as_float(v[c]), -__uint_as_float(v[c + 1]),
                                                     -__uint_as_float(v[c + 2]), -__uint_as_float(v[c + 3]));
    }
    tc_fence_before();
    return true;
}

// ---------------------------------------------------------------------------------------------
// Inclusive prefix sums of x over the C rows of each head of a tile, value e of a lane being row
// (lane + 32 e) % C of head (lane + 32 e) / C: a warp scan of each 32-row segment, then the totals
// of the earlier segments of the same head.
template <int C>
__device__ __forceinline__ void head_prefix_sums(float (&x)[4], int lane) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x[e], o);
            if (lane >= o) x[e] += y;
        }
    float carry = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if ((32 * e) % C == 0) carry = 0.f;  // first segment of a head
        const float total = __shfl_sync(0xffffffffu, x[e], 31);
        x[e] += carry;
        carry += total;
    }
}

template <int C, int DK, int DV, bool TF16, bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
    kkt_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                  const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_u,
                  const __grid_constant__ CUtensorMap map_t, const TcParams p) {
    using CF = Cfg<C, DK, DV>;
    constexpr int G = CF::G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    Barriers *bars = reinterpret_cast<Barriers *>(smem + CF::OFF_BAR);
    // the warp index, broadcast from lane 0 so that the compiler knows it is warp-uniform (as are
    // the role branches and the per-warp constants derived from it)
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    auto stage_kv = [&](int s) { return smem + s * CF::KV_BYTES; };
    auto stage_beta = [&](int s) { return reinterpret_cast<float *>(smem + CF::OFF_META + s * CF::META_BYTES); };
    auto stage_gate = [&](int s) { return reinterpret_cast<float *>(smem + CF::OFF_META + s * CF::META_BYTES + 512); };
    auto stage_gw = [&](int s) { return reinterpret_cast<float *>(smem + CF::OFF_META + s * CF::META_BYTES + 1024); };
    auto stage_gflag = [&](int s) { return reinterpret_cast<int *>(smem + CF::OFF_META + s * CF::META_BYTES + 1536); };
    auto stage_info = [&](int s) {
        return smem_chk(reinterpret_cast<TileInfo *>(smem + CF::OFF_META + s * CF::META_BYTES + 1552));
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            // the TMA transaction arrival, and a second one once beta (and the gate data) are written
            mbar_init(&bars->full[s], 2);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->gram_full, 1);
        mbar_init(&bars->gram_empty, C == 128 ? 6 : 4);  // C = 128: + epilogue warps 2, 3 (M10)
        mbar_init(&bars->tt_full, 4);
        mbar_init(&bars->tt_empty, 1);
        mbar_init(&bars->d_full, 1);
        mbar_init(&bars->d_empty, 4);
        mbar_init(&bars->einfo_full[0], 1);
        mbar_init(&bars->einfo_full[1], 1);
        mbar_init(&bars->mma_final, 1);
        mbar_init(&bars->gram_final, 1);
        mbar_init(&bars->pair_sync[0], 64);
        mbar_init(&bars->pair_sync[1], 64);
        mbar_init(&bars->l64_ops, 4);
        mbar_init(&bars->l64_y, 1);
        mbar_init(&bars->l64_yb, 2);
        mbar_init(&bars->l64_z, 1);
        mbar_init(&bars->kread[0], 1);
        mbar_init(&bars->kread[1], 1);
        mbar_init(&bars->kscaled, 4);
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
    // The next call on the stream may be scheduled now: its CTAs take SMs as this grid's CTAs leave
    // them and run their set-up meanwhile.  This grid's own global-memory work (tile claims, loads
    // of k / v / beta, stores of T / W / U) waits for the previous grid on the stream to complete.
    griddep_launch_dependents();
    griddep_wait();
    KKT_TRACE_CALIB(0);

    if (warp == kWarpProducer) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&map_k);
            prefetch_tmap(&map_v);
        }
        int i = 0;
        bool ok = true;
        // next tile: a fixed round robin, or claimed from the shared counter one tile ahead so
        // that the atomic's round trip overlaps the current tile.  The first tile is blockIdx.x in
        // both schedules (counter value v stands for tile gridDim.x + v), which keeps the launch's
        // burst of atomics on one address off the path to the first load.
        auto claim = [&]() -> int64_t {
            unsigned long long v = 0;
            if (lane == 0) v = atomicAdd(p.tile_counter, 1ull);
            return (int64_t)gridDim.x + (int64_t)__shfl_sync(0xffffffffu, v, 0);
        };
        const bool dyn = p.tile_counter != nullptr;
        int64_t t = (int64_t)blockIdx.x;
        for (; t < p.tiles;) {
            const int64_t t_now = t;
            t = dyn ? claim() : t + gridDim.x;
            const int64_t id = t_now / p.HG;
            const int h0 = (int)(t_now % p.HG) * G;
            if (h0 == 0 && id < p.nseq && lane == 0) check_sequence(p.cu, (int)id, p.nseq, p.ntok, p.status);
            Chunk ch;
            if (!map_chunk(id, p.cu, p.nseq, p.T, p.ntok, C, p.status, ch)) continue;
            if (p.stall_first_tile && i == 0) {
                // test hook: stage 0 is never filled, so every wait on it runs out (failure detection)
                ++i;
                continue;
            }
            // beta of the tile (G x C values, 4 per lane), loaded before waiting for the stage
            float bv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int idx = lane + 32 * e;
                const int g = idx / C, r = idx % C;
                bv[e] = (r < ch.Lc && h0 + g < p.H) ? __ldg(gmem_chk(p.beta, (ch.t0 + r) * p.H + h0 + g, p.ntok * p.H)) : 0.f;
            }
            // gated: prefix sums G of the log decays over each head's chunk, in log2 units, so that
            // Gamma[i][j] = exp2(G_i - G_j).  For a column j of 32-row block b, with R_b = G at the
            // block's first row: Gamma[i][j] = exp2(G_i - R_b) * w_j, w_j = exp2(R_b - G_j), one power
            // per row and block instead of one per element.  That is exact up to rounding while the
            // factors stay in range: |R_b - G_j| <= 96 over the block (a decay of at most 2^-96
            // inside 32 tokens), recorded as the block's flag; other blocks take one power per element.
            // (the loads are issued here and consumed after the stage wait, which hides their latency)
            float gv[4] = {0.f, 0.f, 0.f, 0.f}, wv[4] = {0.f, 0.f, 0.f, 0.f};
            int fv[4] = {0, 0, 0, 0};
            if constexpr (GATED) {
                constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int idx = lane + 32 * e;
                    const int g = idx / C, r = idx % C;
                    gv[e] = (r < ch.Lc && h0 + g < p.H) ? kLog2e * __ldg(gmem_chk(p.g, (ch.t0 + r) * p.H + h0 + g, p.ntok * p.H)) : 0.f;
                }
            }
            const int s = i % kNS;
            const uint32_t u = (uint32_t)(i / kNS);
            if (!wait_bar(&bars->empty[s], (u & 1u) ^ 1u, bars, p.status)) { ok = false; break; }
            if (lane == 0) KKT_TRACE_EVENT(EV_P_EMPTY, i);
            if (lane == 0) {
                TileInfo *info = stage_info(s);
                info->t0 = ch.t0;
                info->Lc = ch.Lc;
                info->h0 = h0;
                info->done = 0;
                uint8_t *st = stage_kv(s);
                mbar_arrive_expect_tx(&bars->full[s], CF::TX_BYTES);
                for (int g = 0; g < G; ++g) {
                    for (int c2 = 0; c2 < CF::NBK; ++c2)
                        tma_load_3d(st + c2 * 16384 + g * C * 128, &map_k, &bars->full[s], c2 * 64, h0 + g,
                                    (int)ch.t0);
                    for (int c2 = 0; c2 < CF::NBV; ++c2)
                        tma_load_3d(st + CF::NBK * 16384 + c2 * 16384 + g * C * 128, &map_v, &bars->full[s],
                                    c2 * 64, h0 + g, (int)ch.t0);
                }
                KKT_TRACE_EVENT(EV_P_ISSUE, i);
            }
            // beta (and, gated, the gate data) while the loads are in flight, so that the first
            // tile's loads do not wait for beta's; the stage completes with a second arrival
            float *sb = stage_beta(s);
#pragma unroll
            for (int e = 0; e < 4; ++e) *smem_chk(sb + lane + 32 * e) = bv[e];
            if constexpr (GATED) {
                head_prefix_sums<C>(gv, lane);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float ref = __shfl_sync(0xffffffffu, gv[e], 0);
                    float dev = fabsf(ref - gv[e]);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) dev = fmaxf(dev, __shfl_xor_sync(0xffffffffu, dev, o));
                    fv[e] = dev <= 96.f;
                    wv[e] = exp2f(ref - gv[e]);
                }
                float *sg = stage_gate(s), *sw = stage_gw(s);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    *smem_chk(sg + lane + 32 * e) = gv[e];
                    *smem_chk(sw + lane + 32 * e) = wv[e];
                }
                if (lane == 0)
                    for (int e = 0; e < 4; ++e) *smem_chk(stage_gflag(s) + e) = fv[e];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full[s]);
            __syncwarp();
            ++i;
        }
        if (ok) {
            const int s = i % kNS;
            const uint32_t u = (uint32_t)(i / kNS);
            if (wait_bar(&bars->empty[s], (u & 1u) ^ 1u, bars, p.status)) {
                if (lane == 0) {
                    stage_info(s)->done = 1;
                    mbar_arrive(&bars->full[s]);
                    mbar_arrive(&bars->full[s]);
                }
            } else {
                ok = false;
            }
        }
        // This CTA claims no more tiles.  The workspace holds the tile counter and a count of CTAs
        // done claiming; the last CTA to finish claiming zeroes both, so the next call on the same
        // workspace starts from zero without a clear of its own (the fence orders this CTA's
        // claims before its count; every other CTA has counted itself, so none claims again).
        if (dyn && lane == 0) {
            __threadfence();
            if (atomicAdd(p.tile_counter + 1, 1ull) == gridDim.x - 1ull) {
                atomicExch(p.tile_counter, 0ull);
                atomicExch(p.tile_counter + 1, 0ull);
            }
        }
        // after a timeout: our last TMA loads must land before shared memory is released
        // (on the normal path every load was consumed through its full barrier)
        if (!ok && lane == 0) {
            for (int back = 1; back <= kNS && back <= i; ++back) {
                const int j = i - back;
                volatile int never = 0;
                mbar_wait(&bars->full[j % kNS], (uint32_t)(j / kNS) & 1u, &never, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == kWarpGram) {
        // ------------------------------------------------------------------ Gram issuer
        // Tile by tile: wait for the stage, zero the rows of a short chunk, wait for the Gram
        // columns of tensor memory, issue S = K K^T.  A thread of its own, so that a Gram is never
        // held up behind the issue of a W|U MMA (whose instructions wait for the tensor pipe).
        const uint32_t idesc_gram = idesc_bf16_f32(128, 128, 0, 0);
        for (int i = 0;; ++i) {
            const int s = i % kNS;
            if (!wait_bar(&bars->full[s], (uint32_t)(i / kNS) & 1u, bars, p.status)) break;
            const TileInfo info = *stage_info(s);
            if (info.done) break;
            if (lane == 0) KKT_TRACE_EVENT(EV_M_FULL, i);
            if (info.Lc < C) {
                // zero rows Lc..C-1 of every head's K and V boxes
                uint8_t *st = stage_kv(s);
                const int per_box = (C - info.Lc) * 8;  // 16-byte chunks
                for (int e = lane; e < G * CF::NBKV * per_box; e += 32) {
                    const int box = e / per_box, w = e % per_box;
                    const int g = box % G, kvh = box / G;  // kvh: the K boxes, then the V boxes
                    *smem_chk(reinterpret_cast<uint4 *>(st + kvh * 16384 + g * C * 128 + (info.Lc + w / 8) * 128 +
                                                        (w % 8) * 16)) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (!wait_bar(&bars->gram_empty, ((uint32_t)i & 1u) ^ 1u, bars, p.status)) break;
            if constexpr (C == 128) {
                // the previous tile's Z has read M11^-1 from the Gram's columns
                if (!wait_bar(&bars->l64_z, ((uint32_t)i & 1u) ^ 1u, bars, p.status)) break;
            }
            if (lane == 0) {
                tc_fence_after();
                const uint32_t a0 = smem_u32(stage_kv(s));
#pragma unroll
                for (int kk = 0; kk < 4 * CF::NBK; ++kk) {  // K = d_k in steps of 16
                    const uint64_t d = sw128_desc(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    mma_ss(tmem + kColGram, d, d, idesc_gram, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars->gram_full);
                if constexpr (GATED) mma_commit(&bars->kread[s]);
                KKT_TRACE_EVENT(EV_M_GRAM, i);
            }
            __syncwarp();
        }
        // every MMA issued by this thread has completed before tensor memory is freed
        if (lane == 0) {
            mma_commit(&bars->gram_final);
            volatile int never = 0;
            mbar_wait(&bars->gram_final, 0u, &never, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ W|U issuer
        // Tile by tile: once T~ is in tensor memory and the epilogue has drained D, hand the tile
        // info to the epilogue and issue D = T~ [K|V] (hi and lo passes); the commit frees T~, the
        // stage, and tells the epilogue that D is ready.  The stage's info marks the end of work.
        const uint32_t idesc_epi = idesc_bf16_f32(128, DK + DV, 0, 1);  // N = d_k columns of K, then d_v of V
        for (int i = 0;; ++i) {
            const int s = i % kNS;
            if (!wait_bar(&bars->full[s], (uint32_t)(i / kNS) & 1u, bars, p.status)) break;
            const TileInfo info = *stage_info(s);
            if (info.done) {
                if (lane == 0) {
                    bars->einfo[i & 1] = info;
                    mbar_arrive(&bars->einfo_full[i & 1]);
                }
                __syncwarp();
                break;
            }
            if constexpr (C == 128) {
                // the tile's level-64 products (see level64_tc); the operands' arrivals imply that the
                // previous W|U MMA has read T~ (Y's columns)
                const uint32_t b_smem = smem_u32(smem + CF::OFF_T + 2 * 16384);
                if (!wait_bar(&bars->l64_ops, (uint32_t)i & 1u, bars, p.status)) break;
                if (lane == 0) {
                    KKT_TRACE_EVENT(EV_M_L64Y, i);
                    tc_fence_after();
                    l64_mma(tmem + kColL64D, tmem + kColL64M10, b_smem);
                    mma_commit(&bars->l64_y);
                }
                __syncwarp();
                if (!wait_bar(&bars->l64_yb, (uint32_t)i & 1u, bars, p.status)) break;
                if (lane == 0) {
                    KKT_TRACE_EVENT(EV_M_L64Z, i);
                    tc_fence_after();
                    l64_mma(tmem + kColL64D, tmem + kColL64M11, b_smem);
                    mma_commit(&bars->l64_z);
                }
                __syncwarp();
            }
            if (!wait_bar(&bars->tt_full, (uint32_t)i & 1u, bars, p.status)) break;
            if (!wait_bar(&bars->d_empty, ((uint32_t)i & 1u) ^ 1u, bars, p.status)) break;
            if constexpr (GATED) {
                if (!wait_bar(&bars->kscaled, (uint32_t)i & 1u, bars, p.status)) break;
            }
            if (lane == 0) {
                KKT_TRACE_EVENT(EV_M_READY, i);
                bars->einfo[i & 1] = info;
                mbar_arrive(&bars->einfo_full[i & 1]);
                tc_fence_after();
                const uint32_t b0 = smem_u32(stage_kv(s));
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
                mma_commit(&bars->empty[s]);
                KKT_TRACE_EVENT(EV_M_EPI, i);
            }
            __syncwarp();
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
        const int g = 32 * q / C;           // head within the tile (m / C: C is a multiple of 32)
        const int wp = 32 * q % C / 32;     // warp position within the head (0 for C = 32)
        const int r = 32 * wp + lane;       // row within the chunk (m % C)
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        uint8_t *tm = smem + CF::OFF_T;     // the tile's T, [half][128 rows][128 B], 128-byte swizzle
        // level-32 product Y: the upper-right 32 x 32 of this warp's 64-row block (zero in T)
        uint8_t *ybuf32 = tm + (((C == 128 ? 64 * (q >> 1) : 0) + 32) >> 5) * 16384 + 64 * (q >> 1) * 128;
        // zero this lane's T~ columns (other heads' blocks and the upper triangle stay zero)
        // and its row of T (the upper triangle stays zero there too)
        {
            // (at C = 128 every T~ row is written whole, zeros included, and the epilogue warps may
            // already be putting M10 into these columns: no clear there)
            if constexpr (C != 128) {
                uint32_t zz[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) zz[c] = 0u;
#pragma unroll
                for (int c = 0; c < 128; c += 16) tmem_st16(tmem + lane_base + kColTT + c, zz);
                tmem_wait_st();
            }
#pragma unroll
            for (int j = 0; j < C; j += 4) *tm_vec(tm, m, j) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        int i = 0;
        uint32_t pair_uses = 0;
        while (true) {
            const int s = i % kNS;
            if (!wait_bar(&bars->full[s], (uint32_t)(i / kNS) & 1u, bars, p.status)) break;
            const TileInfo info = *stage_info(s);
            if (info.done) break;
            const float *sb = stage_beta(s) + g * C;
            const float beta_r = *smem_chk(sb + r);
            // gated: the decay factors of Gamma (see form_a_row)
            const float *sg = stage_gate(s) + g * C;
            const float *sw = stage_gw(s) + g * C;
            bool fac = true;
            float g_r = 0.f;
            if constexpr (GATED) {
                g_r = *smem_chk(sg + r);
                const int *sf = stage_gflag(s) + g * C / 32;
#pragma unroll
                for (int h = 0; h < CF::T_HALVES; ++h) fac = fac && *smem_chk(sf + h) != 0;
            }

            if (!wait_bar(&bars->gram_full, (uint32_t)i & 1u, bars, p.status)) break;
            tc_fence_after();
            if (q == 0 && lane == 0) KKT_TRACE_EVENT(EV_I_GRAM, i);
            // this warp's previous T store has read its rows of the T buffer
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            if (q == 1 && lane == 0) KKT_TRACE_EVENT(EV_I_BW, i);
            // Gram row -> row of A into the T buffer; columns above 32 (wp + 1) stay zero.  At C = 128
            // columns 0..63 of rows 64..127 (M10 of the level-64 coupling) are not formed here: the
            // epilogue warps of those lanes form them straight into tensor memory for the level-64
            // MMA (see level64_tc), so that these rows cost the inverse warps no more than the others.
            form_a_row<GATED>(tm, tmem + lane_base + kColGram + g * C, m, r, (C == 128 && q >= 2) ? 2 : 0, wp, beta_r,
                              fac, g_r, sg, sw);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->gram_empty);
            if (q == 1 && lane == 0) KKT_TRACE_EVENT(EV_I_LD, i);

            // diagonal 16 x 16 blocks (§2.1), one column per lane: right-looking substitution,
            // s[k] <- s[k] - L[k][m] x_m once x_m = s[m] is final.  L is read four columns at a
            // time (one 16-byte chunk per row) before the four steps that use them.

            {
                const int c = lane & 15;
                const int rb = 32 * wp + 16 * (lane >> 4);
                const int mb = g * C + rb;
                float sc[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) sc[k] = (k == c) ? 1.f : 0.f;
#pragma unroll
                for (int m0s = 0; m0s < 16; m0s += 4) {
                    float4 lk[16];
#pragma unroll
                    for (int k = m0s + 1; k < 16; ++k) lk[k] = *tm_vec(tm, mb + k, rb + m0s);
#pragma unroll
                    for (int d = 0; d < 4; ++d) {
                        const int ms = m0s + d;
                        if (ms < 15) {
                            const float xm = sc[ms];
#pragma unroll
                            for (int k = ms + 1; k < 16; ++k) {
                                const float l = d == 0 ? lk[k].x : d == 1 ? lk[k].y : d == 2 ? lk[k].z : lk[k].w;
                                sc[k] = fmaf(-l, xm, sc[k]);
                            }
                        }
                    }
                }
                __syncwarp();
#pragma unroll
                for (int k = 1; k < 16; ++k) *tm_elem(tm, mb + k, rb + c) = sc[k];
                __syncwarp();
            }
            if (q == 1 && lane == 0) KKT_TRACE_EVENT(EV_I_DIAG, i);

            // level 16 (§2.2): the warp's two diagonal blocks, T10 = -X11 (L10 X00).  Y = L10 X00 is
            // kept in the block's upper-right 16 x 16 (rows m0 .. m0 + 15, columns c0 + 16 .. c0 + 31),
            // zero in T and cleared again once read.
            {
                // lane -> rows ii and ii + 8 of the 16 x 16 result, columns jb .. jb + 3.  The 8 lanes
                // of a quarter-warp take 8 different rows of one column group, so their 16-byte
                // accesses fall in 8 different swizzled chunks (no bank conflict)
                const int ii = lane & 7;
                const int jb = (lane >> 3) * 4;
                const int m0 = g * C + 32 * wp;
                const int c0 = 32 * wp;
                float a[2][16];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 16; k += 4) {
                        const float4 t4 = *tm_vec(tm, m0 + 16 + ii + 8 * h, c0 + k);
                        a[h][k] = t4.x; a[h][k + 1] = t4.y; a[h][k + 2] = t4.z; a[h][k + 3] = t4.w;
                    }
                float2 y[2][2];
#pragma unroll
                for (int h = 0; h < 2; ++h) y[h][0] = y[h][1] = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float4 b = *tm_vec(tm, m0 + k, c0 + jb);
                    const float2 b01 = make_float2(b.x, b.y), b23 = make_float2(b.z, b.w);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 ak = make_float2(a[h][k], a[h][k]);
                        y[h][0] = ffma2(ak, b01, y[h][0]);
                        y[h][1] = ffma2(ak, b23, y[h][1]);
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *tm_vec(tm, m0 + ii + 8 * h, c0 + 16 + jb) = make_float4(y[h][0].x, y[h][0].y, y[h][1].x, y[h][1].y);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 16; k += 4) {
                        const float4 t4 = *tm_vec(tm, m0 + 16 + ii + 8 * h, c0 + 16 + k);
                        a[h][k] = t4.x; a[h][k + 1] = t4.y; a[h][k + 2] = t4.z; a[h][k + 3] = t4.w;
                    }
                __syncwarp();
#pragma unroll
                for (int h = 0; h < 2; ++h) y[h][0] = y[h][1] = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float4 b = *tm_vec(tm, m0 + k, c0 + 16 + jb);
                    const float2 b01 = make_float2(b.x, b.y), b23 = make_float2(b.z, b.w);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 ak = make_float2(a[h][k], a[h][k]);
                        y[h][0] = ffma2(ak, b01, y[h][0]);
                        y[h][1] = ffma2(ak, b23, y[h][1]);
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *tm_vec(tm, m0 + 16 + ii + 8 * h, c0 + jb) = make_float4(-y[h][0].x, -y[h][0].y, -y[h][1].x, -y[h][1].y);
                __syncwarp();
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *tm_vec(tm, m0 + ii + 8 * h, c0 + 16 + jb) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (q == 1 && lane == 0) KKT_TRACE_EVENT(EV_I_C16, i);

            bool ok = true;
            if constexpr (C >= 64) {
                // level 32 in each 64-row block (a head at C = 64, half the chunk at C = 128): its
                // rows 32..63 get -M11^-1 M10 M00^-1 (see level32)
                const int pr = q >> 1;
                ok = group_sync(&bars->pair_sync[pr], pair_uses, bars, p.status);
                if (q == 1 && lane == 0) KKT_TRACE_EVENT(EV_I_PAIR, i);
                if (ok) {
                    ok = level32<C == 128 ? 2 : 1>(wp & 1, tm, ybuf32, 64 * pr, C == 128 ? 64 * pr : 0, lane,
                                                   &bars->pair_sync[pr], pair_uses, bars, p.status);
                }
                if constexpr (C == 128) {
                    // level 64: rows 64..127 of the chunk, on the tensor core (see level64_tc)
                    if (q == 1 && lane == 0) KKT_TRACE_EVENT(EV_I_L32, i);
                    if (q == 3 && lane == 0) KKT_TRACE_EVENT(EV_I_L32B, i);
                    if (ok) ok = level64_tc(q, m, i, tm, tmem, lane_base, lane, bars, p.status, KKT_TRACE_ROW(i));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (q == 3 && lane == 0) KKT_TRACE_EVENT(EV_I_INVB, i);
                }
            } else {
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (!ok) break;
            if (q == 1 && lane == 0) KKT_TRACE_EVENT(EV_I_INV, i);

            // T rows in fp32: TMA store of the warp's 32 rows when all are valid, else plain stores
            // (none without T_out: W and U~ only; fp16 T is written after T~, below)
            if (p.T_out == nullptr || TF16) {
            } else if (32 * wp + 32 <= info.Lc) {
                if (lane == 0) {
                    for (int h = 0; h < CF::T_HALVES; ++h)
                        tma_store_3d(&map_t, tm + h * 16384 + 32 * q * 128, 32 * h, info.h0 + g,
                                     (int)(info.t0 + 32 * wp));
                    bulk_commit();
                }
            } else if (r < info.Lc && info.h0 + g < p.H) {
                float4 *dst = reinterpret_cast<float4 *>(gmem_chk(static_cast<float *>(p.T_out),
                                                                  ((info.t0 + r) * p.H + info.h0 + g) * C,
                                                                  p.ntok * p.H * C, C));
#pragma unroll
                for (int j = 0; j < C; j += 4) dst[j / 4] = *tm_vec(tm, m, j);
            }
            if (q == 1 && lane == 0) KKT_TRACE_EVENT(EV_I_TSTORE, i);

            // T~ = T diag(beta), split into bf16 hi + lo, into tensor memory (A operand)
            if (!wait_bar(&bars->tt_empty, ((uint32_t)i & 1u) ^ 1u, bars, p.status)) break;
            tc_fence_after();
            if (q == 1 && lane == 0) KKT_TRACE_EVENT(EV_I_TTW, i);
            // fp16 T (TF16): each row rounded to fp16 as T~ reads it.  The warp's 32 rows go out by
            // one TMA store per 64 columns when all are valid: columns 64 h .. 64 h + 63 of a row are
            // packed into the first 128 bytes of its block h (the 128-byte-swizzled layout of a TMA box
            // of 64 fp16), which hold fp32 values T~ has already read.  Other rows (and C = 32) are
            // written by plain stores.
            const bool t16_tma = TF16 && C >= 64 && p.T_out != nullptr && 32 * wp + 32 <= info.Lc;
            const bool t16_row = TF16 && !t16_tma && p.T_out != nullptr && r < info.Lc && info.h0 + g < p.H;
            {
                uint32_t hi[16], lo[16];
#pragma unroll(C == 128 ? 1 : CF::T_HALVES)
                for (int blk = 0; blk < CF::T_HALVES; ++blk) {
                    float4 *t16s = tm_vec(tm, m, 0);  // row m of block blk / 2, chunk base below
                    if constexpr (TF16) t16s = reinterpret_cast<float4 *>(tm + (blk >> 1) * 16384 + m * 128);
                    if (blk <= wp) {
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            const float4 ta = *tm_vec(tm, m, 32 * blk + c);
                            const float4 tb = *tm_vec(tm, m, 32 * blk + c + 4);
                            const float4 ba = *smem_chk(reinterpret_cast<const float4 *>(sb + 32 * blk + c));
                            const float4 bb = *smem_chk(reinterpret_cast<const float4 *>(sb + 32 * blk + c + 4));
                            split_bf16(fmul2(make_float2(ta.x, ta.y), make_float2(ba.x, ba.y)), hi[c / 2], lo[c / 2]);
                            split_bf16(fmul2(make_float2(ta.z, ta.w), make_float2(ba.z, ba.w)), hi[c / 2 + 1], lo[c / 2 + 1]);
                            split_bf16(fmul2(make_float2(tb.x, tb.y), make_float2(bb.x, bb.y)), hi[c / 2 + 2], lo[c / 2 + 2]);
                            split_bf16(fmul2(make_float2(tb.z, tb.w), make_float2(bb.z, bb.w)), hi[c / 2 + 3], lo[c / 2 + 3]);
                            if constexpr (TF16) {
                                const float4 h8 = make_float4(pack_f16(ta.x, ta.y), pack_f16(ta.z, ta.w),
                                                              pack_f16(tb.x, tb.y), pack_f16(tb.z, tb.w));
                                if (t16_tma)
                                    *smem_chk(t16s + ((4 * (blk & 1) + c / 8) ^ (m & 7))) = h8;
                                else if (t16_row)
                                    *reinterpret_cast<float4 *>(gmem_chk(static_cast<__half *>(p.T_out),
                                                                         ((info.t0 + r) * p.H + info.h0 + g) * C + 32 * blk + c,
                                                                         p.ntok * p.H * C, 8)) = h8;
                            }
                        }
                        const uint32_t col = (uint32_t)(g * C + 32 * blk) / 2;
                        tmem_st16(tmem + lane_base + kColTT + col, hi);
                        tmem_st16(tmem + lane_base + kColTT + 64 + col, lo);
                    } else {
                        if constexpr (C == 128) {
                            // the level-64 products used these columns (see level64_tc): zeros above
                            // the diagonal block
#pragma unroll
                            for (int e = 0; e < 16; ++e) hi[e] = 0u;
                            const uint32_t col = (uint32_t)(32 * blk) / 2;
                            tmem_st16(tmem + lane_base + kColTT + col, hi);
                            tmem_st16(tmem + lane_base + kColTT + 64 + col, hi);
                        }
                        if constexpr (TF16) {
                            // columns above the diagonal block: zeros
                            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (t16_tma)
                                    *smem_chk(t16s + ((4 * (blk & 1) + e) ^ (m & 7))) = z;
                                else if (t16_row)
                                    *reinterpret_cast<float4 *>(gmem_chk(static_cast<__half *>(p.T_out),
                                                                         ((info.t0 + r) * p.H + info.h0 + g) * C + 32 * blk + 8 * e,
                                                                         p.ntok * p.H * C, 8)) = z;
                            }
                        }
                    }
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars->tt_full);
                if (q == 1) KKT_TRACE_EVENT(EV_I_TT, i);
            }
            if (t16_tma) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    for (int h = 0; h < C / 64; ++h)
                        tma_store_3d(&map_t, tm + h * 16384 + 32 * q * 128, 64 * h, info.h0 + g,
                                     (int)(info.t0 + 32 * wp));
                    bulk_commit();
                }
            }
            ++i;
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
        // ------------------------------------------------------------------ epilogue warps
        const int q = warp & 3;             // rows 32 q .. 32 q + 31 of D
        const int g = 32 * q / C;
        const int wp = 32 * q % C / 32;
        const int r = 32 * wp + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        uint8_t *wstage = smem + CF::OFF_WU + q * CF::WU_BUFS * 4096;  // WU_BUFS x [32 rows][128 B]
        int i = 0;
        uint32_t nstore = 0;  // TMA store groups issued by this warp
        bool keys_done = false;  // gated: the stage that ends the work has been seen
        // C = 128, epilogue warps 2 and 3: M10 of tile t, formed from the tile's Gram rows straight into
        // tensor memory (level 64's first A operand, in T~'s columns).  Runs once the previous tile's
        // W|U MMA has read T~ (its D is full), before that D is drained; the next Gram waits for it.
        bool m10_end = false;  // C = 128: the stage that ends the work has been seen
        auto m10_to_tmem = [&](int t) -> bool {
            const int s = t % kNS;
            if (!wait_bar(&bars->full[s], (uint32_t)(t / kNS) & 1u, bars, p.status)) return false;
            if (stage_info(s)->done) {
                m10_end = true;
                return true;
            }
            if (!wait_bar(&bars->gram_full, (uint32_t)t & 1u, bars, p.status)) return false;
            tc_fence_after();
            const int m = 32 * q + lane;  // the row, and its token in the chunk (one head)
            bool fac = true;
            float g_r = 0.f;
            if constexpr (GATED) {
                g_r = *smem_chk(stage_gate(s) + m);
#pragma unroll
                for (int h = 0; h < CF::T_HALVES; ++h) fac = fac && *smem_chk(stage_gflag(s) + h) != 0;
            }
            m10_from_gram<GATED>(tmem + lane_base + kColGram, tmem + lane_base + kColL64M10, m,
                                 *smem_chk(stage_beta(s) + m), fac, g_r, stage_gate(s), stage_gw(s));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars->gram_empty);
                mbar_arrive(&bars->l64_ops);
                if (q == 3) KKT_TRACE_EVENT(EV_E_M10, t);
            }
            return true;
        };
        if constexpr (C == 128) {
            if (q >= 2 && !m10_to_tmem(0)) i = -1;  // a timeout: skip the loop
        }
        while (i >= 0) {
            if constexpr (GATED) {
                // The keys of W carry the gate's decay from the chunk's start through their own token,
                // W = T diag(beta) diag(gamma) K with gamma_j = exp2(G_j) (G the prefix sums the
                // producer left in the stage, log2 units).  Once the Gram MMA has read the stage's K,
                // each thread scales its row of K in place by gamma rounded to bf16, one packed bf16
                // multiply per pair (the Gram used the unscaled keys), before the W|U MMA of the tile
                // reads it.  Three times fewer instructions than widening to fp32: the inverse warps
                // share the SM's issue slots with this pass.  A row's 16-byte chunks
                // are visited in swizzled order, so the 8 rows of a quarter-warp hit 8 different bank
                // groups.
                if (!keys_done) {
                    const int s = i % kNS;
                    if (!wait_bar(&bars->full[s], (uint32_t)(i / kNS) & 1u, bars, p.status)) break;
                    if (stage_info(s)->done) {
                        keys_done = true;
                    } else {
                        if (!wait_bar(&bars->kread[s], (uint32_t)(i / kNS) & 1u, bars, p.status)) break;
                        const int m = 32 * q + lane;
                        const float gam = exp2f(*smem_chk(stage_gate(s) + m));
                        const uint32_t gg = pack_bf16(gam, gam);  // gamma rounded to bf16, then each product
                        uint8_t *row = stage_kv(s) + m * 128;
                        // a loop, not unrolled: the kernel is sensitive to its code size
#pragma unroll 1
                        for (int ce = 0; ce < 8 * CF::NBK; ++ce) {
                            uint4 *pv = smem_chk(reinterpret_cast<uint4 *>(row + (ce >> 3) * 16384 + (((ce & 7) ^ (m & 7)) << 4)));
                            uint4 x = *pv;
                            x.x = mul_bf16x2(x.x, gg);
                            x.y = mul_bf16x2(x.y, gg);
                            x.z = mul_bf16x2(x.z, gg);
                            x.w = mul_bf16x2(x.w, gg);
                            *pv = x;
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->kscaled);
                    }
                }
            }
            if (!wait_bar(&bars->einfo_full[i & 1], (uint32_t)(i >> 1) & 1u, bars, p.status)) break;
            const TileInfo info = bars->einfo[i & 1];
            if (info.done) break;
            if (!wait_bar(&bars->d_full, (uint32_t)i & 1u, bars, p.status)) break;
            tc_fence_after();
            if (q == 0 && lane == 0) KKT_TRACE_EVENT(EV_E_DFULL, i);
            if constexpr (C == 128) {
                if (q >= 2 && !m10_end && !m10_to_tmem(i + 1)) break;
            }
            const bool warp_full = 32 * wp + 32 <= info.Lc;
            const bool row_ok = r < info.Lc && info.h0 + g < p.H;
            const int64_t grow = (info.t0 + r) * p.H + info.h0 + g;
#pragma unroll 1
            for (int cc = 0; cc < CF::NBKV; ++cc) {  // 64 columns of D at a time: those of W, then of U~
                uint32_t v0[32], v1[32];
                tmem_ld32(tmem + lane_base + kColD + 64 * cc, v0);
                tmem_ld32(tmem + lane_base + kColD + 64 * cc + 32, v1);
                tmem_wait_ld();
                if (cc == CF::NBKV - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bars->d_empty);
                        if (q == 0) KKT_TRACE_EVENT(EV_E_DEMPTY, i);
                    }
                }
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    pk[e] = pack_bf16(__uint_as_float(v0[2 * e]), __uint_as_float(v0[2 * e + 1]));
                    pk[16 + e] = pack_bf16(__uint_as_float(v1[2 * e]), __uint_as_float(v1[2 * e + 1]));
                }
                if (warp_full) {
                    uint8_t *buf = wstage + (nstore % CF::WU_BUFS) * 4096;
                    if (lane == 0) bulk_wait_read<CF::WU_BUFS - 1>();
                    __syncwarp();
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        *smem_chk(reinterpret_cast<uint4 *>(buf + sw128((uint32_t)(lane * 128 + 16 * e)))) =
                            make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(cc < CF::NBK ? &map_w : &map_u, buf, 64 * (cc < CF::NBK ? cc : cc - CF::NBK), info.h0 + g,
                                     (int)(info.t0 + 32 * wp));
                        bulk_commit();
                    }
                    ++nstore;
                } else if (row_ok) {
                    const int dw = cc < CF::NBK ? DK : DV;  // this group's tensor width
                    __nv_bfloat16 *base = gmem_chk(cc < CF::NBK ? p.W_out : p.U_out,
                                                   grow * dw + 64 * (cc < CF::NBK ? cc : cc - CF::NBK),
                                                   p.ntok * p.H * dw, 64);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        reinterpret_cast<uint4 *>(base)[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            if (q == 0 && lane == 0) KKT_TRACE_EVENT(EV_E_DONE, i);
            ++i;
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    KKT_TRACE_CALIB(1);
    if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// host side

template <int C, int DK, int DV>
int launch_tc_t(const Problem &pb) {
    using CF = Cfg<C, DK, DV>;
    CUtensorMap mk, mv, mw, mu, mt;
    if (!make_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pb.k, pb.ntok, pb.H, pb.dk, 64, C) ||
        !make_map(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pb.v, pb.ntok, pb.H, pb.dv, 64, C) ||
        !make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pb.W_out, pb.ntok, pb.H, pb.dk, 64, 32) ||
        !make_map(&mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pb.U_out, pb.ntok, pb.H, pb.dv, 64, 32) ||
        (pb.T_out && !pb.t_f16 && !make_map(&mt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pb.T_out, pb.ntok, pb.H, C, 32, 32)) ||
        (pb.T_out && pb.t_f16 && C >= 64 && !make_map(&mt, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, pb.T_out, pb.ntok, pb.H, C, 64, 32)))
        return KKT_ERR_CUDA;
    if (!pb.T_out || (pb.t_f16 && C < 64)) mt = CUtensorMap{};  // never used: no T, or fp16 T by plain stores
    TcParams p;
    p.beta = pb.beta;
    p.g = pb.g;
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
    p.trace = static_cast<unsigned long long *>(pb.trace);
    p.tile_counter = pb.tile_counter;
    p.stall_first_tile = pb.stall_first_tile;
    auto kern = pb.g ? (pb.t_f16 ? kkt_tc_kernel<C, DK, DV, true, true> : kkt_tc_kernel<C, DK, DV, false, true>)
                     : (pb.t_f16 ? kkt_tc_kernel<C, DK, DV, true, false> : kkt_tc_kernel<C, DK, DV, false, false>);
    const bool attr_ok =
        pb.g ? (pb.t_f16 ? ensure_max_smem<kkt_tc_kernel<C, DK, DV, true, true>>(CF::SMEM_BYTES)
                         : ensure_max_smem<kkt_tc_kernel<C, DK, DV, false, true>>(CF::SMEM_BYTES))
             : (pb.t_f16 ? ensure_max_smem<kkt_tc_kernel<C, DK, DV, true, false>>(CF::SMEM_BYTES)
                         : ensure_max_smem<kkt_tc_kernel<C, DK, DV, false, false>>(CF::SMEM_BYTES));
    if (!attr_ok) return KKT_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return KKT_ERR_CUDA;
    const int64_t grid = p.tiles < sms ? p.tiles : sms;
    // programmatic stream serialisation: this launch may start while the previous kernel on the
    // stream finishes (the kernel waits for it before touching global memory)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = CF::SMEM_BYTES;
    cfg.stream = pb.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mk, mv, mw, mu, mt, p) != cudaSuccess) return KKT_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KKT_OK : KKT_ERR_CUDA;
}

}  // namespace
}  // namespace kkt
