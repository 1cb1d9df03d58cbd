/*
 * kkt.h -- C ABI of the GB300 (sm_103a) kkt_solve library, libkkt.so.
 *
 * kkt_solve is the chunk-local UT transform of Gated DeltaNet chunked
 * prefill, as described on the page "TileLang 实战：单位下三角矩阵求逆"
 * (TileLang in practice: inverting a unit lower-triangular matrix):
 *
 *   For every chunk of C consecutive tokens of one sequence and one head
 *   (section 1, the coefficient matrix; section 3.2, beta scales rows and the
 *   diagonal is one):
 *       A  = I + strictLower(diag(beta) K K^T)          (C x C)
 *       T  = A^-1                                        (section 2.2 blocked recursion)
 *       W  = T diag(beta) K,   U~ = T diag(beta) V       (section 1)
 *   Chunks restart at every sequence start; the last chunk of a sequence may
 *   be shorter than C (Lc rows), and is the leading Lc x Lc block of the
 *   general case (A is lower triangular, so padding never reaches it).
 *
 * Tensor layouts follow the [B, T, H, d] convention of the FlashQLA API
 * (FlashQLA announcement, section "使用方式" / usage): row-major, contiguous,
 * one K per value head (H_k = H_v = H).
 *
 *   k     [B, T, H, dk]   input  (bf16, or fp32 with KKT_IO_F32)
 *   v     [B, T, H, dv]   input  (same dtype as k)
 *   beta  [B, T, H]       input  fp32, expected in (0, 1)
 *   T_out [B, T, H, C]    output fp32 (fp16 with KKT_T_OUT_F16, kkt_solve_fwd_ex
 *                         only); row (b, t, h) holds row (t - chunk start)
 *                         of its chunk's T, zeros in columns >= Lc.  May be NULL:
 *                         T is then computed but not written, and the call
 *                         produces W and U~ only (the page materialises T
 *                         because W and U~ both use it, section 5 item 10; a
 *                         caller that needs only W and U~ saves the 4C bytes
 *                         per token and head of the T write)
 *   W_out [B, T, H, dk]   output (dtype of k)
 *   U_out [B, T, H, dv]   output (dtype of k)
 *
 * Variable-length batches: pass cu_seqlens = int32[B + 1] offsets into a
 * packed token axis (cu_seqlens[0] = 0, nondecreasing, cu_seqlens[B] = T);
 * the tensors are then [1, T, H, .] with T the total token count and B the
 * number of sequences.  With cu_seqlens == NULL the batch is B sequences of
 * T tokens each.
 *
 * Ownership and execution: every pointer is a device pointer owned by the
 * caller (cu_seqlens included).  The library allocates no memory.  Calls are
 * asynchronous on `stream` (NULL = the legacy default stream) and never
 * synchronise the host.  k, v, T_out, W_out and U_out must be 16-byte aligned
 * (they are moved by TMA), beta and cu_seqlens 4-byte aligned.  Outputs must
 * not alias inputs.
 *
 * Errors: invalid arguments return a nonzero kkt_status WITHOUT launching.
 * Problems only the device can see (a malformed cu_seqlens, a bounded wait
 * that expired) are recorded in a per-device status word, read and cleared by
 * kkt_device_status(); the kernels skip the affected chunks and never fault
 * or trap on them.
 */
#ifndef KKT_H_
#define KKT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

typedef enum kkt_status {
    KKT_OK = 0,
    KKT_ERR_ARG = 1,         /* null pointer, nonpositive size, inconsistent shapes */
    KKT_ERR_UNSUPPORTED = 2, /* (C, dk, dv, io dtype, kernel) combination not built */
    KKT_ERR_ALIGN = 3,       /* a pointer is misaligned (16 B for tensors moved by TMA, 4 B for beta) */
    KKT_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed */
    KKT_ERR_SEQLENS = 5,     /* device saw a malformed cu_seqlens (kkt_device_status) */
    KKT_ERR_TIMEOUT = 6,     /* a device-side bounded wait expired (kkt_device_status) */
    KKT_ERR_NO_DEVICE = 7    /* no usable CUDA device / not an sm_103 device */
} kkt_status;

/* I/O dtype of k, v, W_out, U_out (beta is always fp32; T_out is fp32 unless KKT_T_OUT_F16). */
enum { KKT_IO_BF16 = 0, KKT_IO_F32 = 1 };

/* Flag for the io_dtype of kkt_solve_fwd_ex: T_out holds fp16 (2C bytes per row, round to
 * nearest) instead of fp32.  The page's own kernel stores T in the input's half precision
 * ("TileLang 实战：单位下三角矩阵求逆" section 3.1); W and U~ are unchanged (they are formed from
 * T before it is rounded). */
#define KKT_T_OUT_F16 0x100

/* Minimum size of the optional workspace of kkt_solve_fwd_ex, in bytes. */
#define KKT_WORKSPACE_BYTES 256

/* Kernel selection for kkt_solve_fwd_ex. */
enum {
    KKT_KERNEL_AUTO = 0, /* tcgen05/TMA kernel when it supports the shape, else the SIMT kernel */
    KKT_KERNEL_SIMT = 1, /* one CTA per (chunk, head), fp32 CUDA-core arithmetic throughout */
    KKT_KERNEL_TC = 2    /* persistent tcgen05 + TMA kernel (bf16 I/O, dk, dv in {64, 128}) */
};

/*
 * kkt_solve_fwd -- bf16 k, v, W_out, U_out; fp32 beta, T_out.
 *   B, T, H   batch, tokens per sequence (total tokens with cu_seqlens), heads (>= 1; T >= 0)
 *   dk, dv    64 or 128
 *   C         chunk size: 32, 64 or 128 (recursion depth 1, 2, 3 to a 16 x 16 base,
 *             "TileLang 实战：单位下三角矩阵求逆" section 2.3, second table)
 * Returns KKT_OK or a kkt_status.  T == 0 is valid and launches nothing.
 */
int kkt_solve_fwd(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                  int B, int T, int H, int dk, int dv, int C,
                  float *T_out, void *W_out, void *U_out, struct CUstream_st *stream);

/*
 * kkt_solve_fwd_ex -- as kkt_solve_fwd, with the I/O dtype (KKT_IO_BF16 or
 * KKT_IO_F32, optionally ORed with KKT_T_OUT_F16) and the kernel (KKT_KERNEL_*)
 * chosen explicitly.  fp32 I/O runs
 * the SIMT kernel only; asking for KKT_KERNEL_TC with it returns
 * KKT_ERR_UNSUPPORTED (the tcgen05 kernel covers every bf16 shape, d_k and d_v
 * each 64 or 128, d_k = d_v or not).
 * KKT_KERNEL_AUTO takes the tcgen05 kernel whenever it covers the call.
 *
 * workspace: NULL, or caller-owned device memory of at least
 * KKT_WORKSPACE_BYTES (workspace_bytes), 16-byte aligned, zero-filled before its
 * first use.  With it the tensor-core kernel hands out work dynamically (an
 * atomic tile counter) instead of in a fixed round robin, which evens out SMs
 * that run at different speeds.  Every call leaves the workspace zero-filled
 * again when its kernel ends (the kernel's last CTA clears it), so consecutive
 * calls on one stream share it with no clear in between, and back-to-back calls
 * are plain kernel launches; calls that may run at the same time need distinct
 * workspaces.
 *
 * The tensor-core kernel is launched with programmatic stream serialisation: its
 * CTAs may be scheduled while the previous kernel on the stream finishes, and
 * they wait for that kernel to complete before touching global memory.
 */
int kkt_solve_fwd_ex(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                     int B, int T, int H, int dk, int dv, int C,
                     void *T_out, void *W_out, void *U_out,
                     int io_dtype, int kernel, void *workspace, size_t workspace_bytes,
                     struct CUstream_st *stream);

/*
 * kkt_solve_fwd_gated -- the gated variant of kkt_solve_fwd_ex.  With a gate
 * the coefficient becomes diag(beta)(Gamma o K K^T) ("TileLang 实战：单位下三角
 * 矩阵求逆" section 5 item 12):
 *
 *   A = I + strictLower(diag(beta) (Gamma o K K^T)),
 *   Gamma[i][j] = exp(g_{j+1} + ... + g_i)   (i > j, tokens of the same chunk),
 *
 * the product of the per-token decays alpha_t = exp(g_t) between token j and
 * token i.  T = A^-1, W = T diag(beta) K and U~ = T diag(beta) V as in the
 * ungated call (the page states no other change).  The gate restarts at every
 * chunk.
 *
 *   g [B, T, H]   input fp32, the per-token log decay (the `g` argument of the
 *                 FlashQLA API, "FlashQLA" page, usage section); expected <= 0
 *                 (decays in (0, 1]).  Layout as beta; 4-byte aligned.
 *
 * g == NULL is the ungated call.  Every other argument, the layouts,
 * ownership and errors are those of kkt_solve_fwd_ex.
 */
int kkt_solve_fwd_gated(const void *k, const void *v, const float *beta, const float *g,
                        const int32_t *cu_seqlens, int B, int T, int H, int dk, int dv, int C,
                        void *T_out, void *W_out, void *U_out,
                        int io_dtype, int kernel, void *workspace, size_t workspace_bytes,
                        struct CUstream_st *stream);

/* Size of the scratch array compiled into the library for kkt_solve_fwd_noalloc. */
#define KKT_NOALLOC_SCRATCH_BYTES 256

/*
 * kkt_solve_fwd_noalloc -- kkt_solve_fwd for callers that cannot allocate.
 * The pages have no counterpart to this entry point; it is a deployment aid.
 *
 * Some callers may not allocate device memory at all: code that runs under a
 * framework which has already handed every byte of the GPU to its own caching
 * allocator, plug-ins and custom operators that receive only their inputs and
 * outputs, and serving loops where a cudaMalloc would synchronise the device and
 * stall other work.  kkt_solve_fwd_ex needs a caller-provided workspace for the
 * tensor-core kernel's work counter; this entry point uses instead a
 * KKT_NOALLOC_SCRATCH_BYTES array compiled into the library (one per device,
 * kept by every GPU that loads the library until the process exits), so it
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *
 *   Arguments, layouts, ownership and errors: as kkt_solve_fwd (bf16 I/O), run
 *   on the tensor-core kernel only, which covers every shape kkt_solve_fwd
 *   accepts (bf16; other shapes return KKT_ERR_UNSUPPORTED).  The scratch a call
 *   needs does not grow with the problem: 16 bytes (two 64-bit counters) of the
 *   array, for every problem size, so no size is rejected for want of scratch.
 *   The first call on a device looks up the array's device address (with that
 *   device current) and caches it; make that first call before any stream
 *   capture.  cudaDeviceReset invalidates the cached address, so calls after a
 *   reset of the device are not supported.
 *   Every call shares the array.  Each call clears the 16 bytes on `stream`
 *   (cudaMemsetAsync, which allocates nothing) before its launch, and its kernel
 *   leaves them zero when it ends.  Calls whose work overlaps on the GPU (other
 *   streams, other host threads) race on the counters, which can leave tiles of
 *   the overlapping calls uncomputed; the caller must serialise such calls.  The
 *   clear keeps a raced or timed-out call from affecting later calls.
  */
int kkt_solve_fwd_noalloc(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                          int B, int T, int H, int dk, int dv, int C,
                          float *T_out, void *W_out, void *U_out, struct CUstream_st *stream);

/*
 * gdn_chunk_state_fwd -- the chunk state recurrence and output of Gated DeltaNet chunked prefill,
 * the computation that consumes kkt_solve's W and U~ (the FlashQLA page, section "Tilelang
 * Warp-Specialized Kernel", forward: V', S and O per chunk; the API's q, k, g, scale,
 * initial_state and final state, section "使用方式").  The pages' own formula of the recurrence
 * was lost; the one taken is the gated delta rule,
 *
 *   S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,   o_t = scale S_t^T q_t,
 *
 * alpha_t = exp(g_t) (1 without a gate), S_0 the initial state (zero when NULL), which the call
 * computes chunk by chunk from W and U~: for a chunk of Lc tokens entered with state S, with
 * G_i = g_0 + ... + g_i from the chunk's first token and Gamma[i][j] = exp(G_i - G_j),
 *
 *   V' = U~ - W S
 *   O  = scale (diag(e^G) Q S + (Gamma o tril(Q K^T)) V')      (the diagonal included)
 *   S <- e^{G_{Lc-1}} S + (diag(e^{G_{Lc-1} - G}) K)^T V'.
 *
 * The chunks are those of kkt_solve: C tokens, restarting at every sequence start.  W and U~ are
 * the W_out and U_out of kkt_solve_fwd (ungated, g == NULL here) or kkt_solve_fwd_gated (with the
 * same g) on the same k, beta, cu_seqlens and C.
 *
 *   q, k, w   [B, T, H, dk] bf16       u, o  [B, T, H, dv] bf16 (o: output)
 *   g         [B, T, H] fp32 per-token log decays (<= 0), or NULL (no gate)
 *   initial_state, final_state   [nseq, H, dk, dv] fp32 (nseq = B), each may be NULL
 *   cu_seqlens, B, T, H           as in kkt_solve_fwd
 *   dk = dv = 128 and C = 64 (other values return KKT_ERR_UNSUPPORTED)
 *   scale     multiplies o (the FlashQLA API's `scale`; commonly dk^-1/2)
 *
 * Precision: the products run on the tensor cores with bf16 operands (S, V' and the masked
 * Q K^T rounded to bf16) and fp32 accumulation; the state is kept and returned in fp32.
 * Ownership, alignment (16 B for the bf16 tensors and the states, 4 B for g and cu_seqlens),
 * asynchrony and errors: as kkt_solve_fwd.  With no tokens the call copies the initial state (or
 * zero) to final_state.  o rows of padding do not exist: only the tokens' rows are written.
 */
int gdn_chunk_state_fwd(const void *q, const void *k, const void *w, const void *u, const float *g,
                        const float *initial_state, const int32_t *cu_seqlens, int B, int T, int H,
                        int dk, int dv, int C, float scale, void *o, float *final_state,
                        struct CUstream_st *stream);

/*
 * kkt_solve_fwd_host -- kkt_solve on HOST buffers: the call copies the inputs to the device, runs
 * kkt_solve and copies T, W and U~ back, pipelined in consecutive pieces of the token axis so that
 * the two copy directions and the kernels overlap.  The operation, shapes and dtypes are those of
 * kkt_solve_fwd_gated (the page "TileLang 实战：单位下三角矩阵求逆", section 1); the pages have no
 * host-memory entry point: this one serves callers whose tensors live in host memory, and is the
 * call the end-to-end measurement makes.
 *
 *   k, v, beta, g, T_out, W_out, U_out   HOST pointers, the shapes and dtypes of kkt_solve_fwd_ex
 *                   (g may be NULL: ungated; T_out may be NULL: W and U~ only).  Page-locked
 *                   (pinned) memory lets the copies run asynchronously and overlap; with pageable
 *                   memory the results are the same, but the copies serialise.
 *   cu_seqlens      NULL, or a HOST int32 array of B + 1 offsets, as in kkt_solve_fwd (checked on
 *                   the host: nondecreasing, from 0 to T, else KKT_ERR_SEQLENS)
 *   io_dtype, kernel  as in kkt_solve_fwd_ex
 *   pieces          1 .. KKT_HOST_MAX_PIECES consecutive parts of the token axis; a sequence is cut
 *                   only at a multiple of C from its start, so every chunk, and every result, is
 *                   that of one call on the whole batch
 *   workspace       DEVICE memory of at least kkt_host_workspace_bytes(...) bytes, 256-byte
 *                   aligned, owned by the caller: the device copies of every tensor and the
 *                   kernel's work counter.  Calls that may run at the same time need distinct
 *                   workspaces.
 *   stream          the call runs after the work already on `stream`, and the work enqueued on
 *                   `stream` after it runs after it; it returns without waiting (synchronise
 *                   `stream` before reading the outputs or reusing the inputs).  The copies run on
 *                   two streams of the library's own per device, created on the first call and kept
 *                   until the process exits (cudaDeviceReset invalidates them: calls after a reset
 *                   are not supported).  Host threads may call it at the same time: the enqueueing
 *                   is serialised.
 *
 * Returns the statuses of kkt_solve_fwd_gated (argument errors without enqueueing anything);
 * KKT_ERR_ARG also for a workspace that is too small or misaligned.
 */
#define KKT_HOST_MAX_PIECES 64
/* Workspace bytes of kkt_solve_fwd_host for the same B, T, H, dk, dv, C and io_dtype; gated: g != NULL;
 * varlen: cu_seqlens != NULL (the token axis then has T rows, else B * T).  Host-only, no CUDA call. */
size_t kkt_host_workspace_bytes(int B, int T, int H, int dk, int dv, int C, int io_dtype, int gated, int varlen,
                                int pieces);
int kkt_solve_fwd_host(const void *k, const void *v, const float *beta, const float *g,
                       const int32_t *cu_seqlens, int B, int T, int H, int dk, int dv, int C,
                       void *T_out, void *W_out, void *U_out, int io_dtype, int kernel, int pieces,
                       void *workspace, size_t workspace_bytes, struct CUstream_st *stream);

/*
 * kkt_device_status -- synchronises `stream`, then returns and clears the
 * status word of the current device: KKT_OK, or the first device-side error
 * (KKT_ERR_SEQLENS, KKT_ERR_TIMEOUT) recorded since the last call; KKT_ERR_CUDA
 * if the synchronisation itself failed.
 */
int kkt_device_status(struct CUstream_st *stream);

/* Which kernel kkt_solve_fwd_ex would run (KKT_KERNEL_SIMT / _TC), or a
 * negated kkt_status if the arguments are unsupported.  Host-only, no CUDA call. */
int kkt_select_kernel(int dk, int dv, int C, int io_dtype, int kernel);

/* Static string for a kkt_status value. */
const char *kkt_status_string(int status);

/* Library version, (major << 16) | (minor << 8) | patch. */
int kkt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KKT_H_ */
