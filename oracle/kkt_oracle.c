/*
 * kkt_oracle.c -- fp64 CPU oracle for kkt_solve, the chunk-local UT transform
 * of Gated DeltaNet chunked prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link, load or call this file.  Only
 * tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg
 * use it.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes, following "TileLang 实战：单位下三角矩阵求逆" (TileLang in
 * practice: inverting a unit lower-triangular matrix):
 *
 *   For every chunk of C consecutive tokens of one sequence and one head
 *   (the last chunk of a sequence may be shorter: Lc <= C rows):
 *
 *   1. §1 (the coefficient matrix) and §3.2 (beta scales rows, the diagonal
 *      is set to one):
 *          A = I + strictLower(diag(beta) K K^T)
 *      i.e. A[i][i] = 1, A[i][j] = beta_i * <k_i, k_j> for i > j, 0 above.
 *   2. §2.1 (row-wise forward substitution):
 *          X[r,:] = e_r^T - sum_{j<r} A[r][j] X[j,:],   T = X = A^{-1}.
 *      The oracle deliberately does NOT use the blocked recursion of §2.2;
 *      it is the plain definition of the inverse of a unit lower-triangular
 *      matrix, solved one row after another.
 *   3. §1 (the two products the inverse feeds):
 *          W = T diag(beta) K,    U~ = T diag(beta) V.
 *
 *   Gated variant ("TileLang 实战：单位下三角矩阵求逆" §5 item 12: with a gate
 *   the coefficient becomes diag(beta)(Gamma o K K^T)).  The gate input is a
 *   per-token log decay g_t (the FlashQLA page's `g`, "FlashQLA" usage
 *   section; its decay alpha_t = exp(g_t) lies in (0, 1), "Gate 衰减性质"
 *   section).  Gamma[i][j] is the decay from token j to token i of the same
 *   chunk, the product of alpha_t over j < t <= i, computed as
 *   exp(sum_{t=j+1..i} g_t).  Step 1 becomes
 *          A = I + strictLower(diag(beta)(Gamma o K K^T)),
 *   step 2 is as above, and in step 3 the keys carry the decay from the
 *   chunk's start through their own token, gamma_j = exp(g_0 + ... + g_j)
 *   (token 0 being the chunk's first):
 *          W = T diag(beta) diag(gamma) K,    U~ = T diag(beta) V.
 *   The decay in W is what the gated delta rule needs downstream: the state
 *   the chunk starts from reaches token j's update decayed by gamma_j, so the
 *   chunk's correction of that state is W S (see gdn_oracle.c, which pins the
 *   chunkwise form against the token-by-token recurrence).  With g = 0 every
 *   gamma_j is 1 and W is the ungated one.  The gate restarts at every chunk:
 *   Gamma and gamma involve only tokens of the chunk.
 *
 *   Output layout (the CUDA library's layout, fixed by its C header):
 *     T_out[n][h][0..C)  row n holds row (n - chunk start) of its chunk's T,
 *                        with zeros in columns j >= Lc;
 *     W_out[n][h][0..dk), U_out[n][h][0..dv)  one row per token.
 *   n is the flat token index (b*T + t for fixed-length batches, or the
 *   packed index for variable-length batches described by cu_seqlens).
 *
 * All arithmetic is in double precision on the values the caller passes (the
 * tests pass the bf16-rounded inputs widened to double, and beta's fp32
 * value widened to double).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Gamma[i][j] for j < i: the gate's decay from token j to token i of the
 * chunk, exp of the sum of the log decays of tokens j+1 .. i. */
static double gate_decay(const double *gc, int j, int i)
{
    double s = 0.0;
    for (int t = j + 1; t <= i; ++t)
        s += gc[t];
    return exp(s);
}

/* Step 1: A = I + strictLower(diag(beta) K K^T), C x C, row-major, times
 * Gamma elementwise when the chunk has a gate (gc: its log decays, or NULL).
 * Rows and columns >= Lc (padding of a short last chunk) are those of the
 * identity. */
static void build_coefficients(const double *kc, const double *bc, const double *gc,
                               int Lc, int C, int dk, double *A)
{
    for (int i = 0; i < C; ++i) {
        for (int j = 0; j < C; ++j) {
            double a = 0.0;
            if (i == j) {
                a = 1.0;
            } else if (i > j && i < Lc) {
                double dot = 0.0;
                for (int d = 0; d < dk; ++d)
                    dot += kc[(int64_t)i * dk + d] * kc[(int64_t)j * dk + d];
                a = bc[i] * dot;
                if (gc)
                    a *= gate_decay(gc, j, i);
            }
            A[(int64_t)i * C + j] = a;
        }
    }
}

/* Step 2: X = A^{-1} by forward substitution, one row after another. */
static void invert_unit_lower(const double *A, int C, double *X)
{
    for (int r = 0; r < C; ++r) {
        double *xr = X + (int64_t)r * C;
        for (int c = 0; c < C; ++c)
            xr[c] = (c == r) ? 1.0 : 0.0;
        for (int j = 0; j < r; ++j) {
            const double arj = A[(int64_t)r * C + j];
            const double *xj = X + (int64_t)j * C;
            for (int c = 0; c < C; ++c)
                xr[c] -= arj * xj[c];
        }
    }
}

/* gamma_j: the gate's decay from the chunk's start through token j, exp of the
 * sum of the log decays of tokens 0 .. j. */
static double decay_from_start(const double *gc, int j)
{
    double acc = 0.0;
    for (int t = 0; t <= j; ++t)
        acc += gc[t];
    return exp(acc);
}

/* Step 3: rows of Y = T diag(beta) M for M = V (width dv), or for M = K
 * (width dk) Y = T diag(beta) diag(gamma) K when the chunk has a gate (gc:
 * its log decays; NULL for V and for ungated chunks). */
static void apply_scaled(const double *X, const double *bc, const double *gc, const double *mc,
                         int Lc, int C, int width, double *out)
{
    for (int i = 0; i < Lc; ++i) {
        for (int e = 0; e < width; ++e) {
            double s = 0.0;
            for (int j = 0; j < Lc; ++j) {
                double f = bc[j];
                if (gc)
                    f *= decay_from_start(gc, j);
                s += X[(int64_t)i * C + j] * f * mc[(int64_t)j * width + e];
            }
            out[(int64_t)i * width + e] = s;
        }
    }
}

/*
 * One chunk, contiguous inputs.
 *   kc [Lc][dk], vc [Lc][dv], bc [Lc]       (rows of one head)
 *   gc [Lc] log decays of the gated variant, or NULL
 *   T  [Lc][C]  (zeros in columns >= Lc), W [Lc][dk], U [Lc][dv]
 *   A_out, if not NULL, receives the C x C coefficient matrix.
 * Returns 0, or -1 on bad sizes / allocation failure.
 */
int kkt_oracle_chunk(const double *kc, const double *vc, const double *bc,
                     const double *gc, int Lc, int C, int dk, int dv,
                     double *T, double *W, double *U, double *A_out)
{
    if (Lc < 1 || Lc > C || C < 1 || dk < 1 || dv < 1)
        return -1;
    double *A = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *X = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *bz = (double *)calloc((size_t)C, sizeof(double));
    if (!A || !X || !bz) {
        free(A); free(X); free(bz);
        return -1;
    }
    memcpy(bz, bc, sizeof(double) * (size_t)Lc);
    build_coefficients(kc, bz, gc, Lc, C, dk, A);
    invert_unit_lower(A, C, X);
    for (int i = 0; i < Lc; ++i)
        for (int j = 0; j < C; ++j)
            T[(int64_t)i * C + j] = (j < Lc) ? X[(int64_t)i * C + j] : 0.0;
    apply_scaled(X, bz, gc, kc, Lc, C, dk, W);
    apply_scaled(X, bz, NULL, vc, Lc, C, dv, U);
    if (A_out)
        memcpy(A_out, A, sizeof(double) * (size_t)C * C);
    free(A); free(X); free(bz);
    return 0;
}

/*
 * Whole tensors.
 *   k    [N][H][dk], v [N][H][dv], beta [N][H]  (N = B*T fixed-length, or the
 *        packed token count T when cu_seqlens is given)
 *   g    [N][H] log decays of the gated variant, or NULL
 *   cu_seqlens: NULL for B sequences of T tokens each; otherwise B+1
 *        nondecreasing offsets with cu_seqlens[0] = 0, cu_seqlens[B] = T.
 *   T_out [N][H][C], W_out [N][H][dk], U_out [N][H][dv].
 *   nthreads <= 0 uses the OpenMP default.
 * Returns 0, -1 on bad arguments, -2 on a malformed cu_seqlens.
 */
int kkt_oracle_fwd(const double *k, const double *v, const double *beta,
                   const double *g, const int64_t *cu_seqlens, int64_t B, int64_t T, int64_t H,
                   int64_t dk, int64_t dv, int64_t C,
                   double *T_out, double *W_out, double *U_out, int nthreads)
{
    if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1 || C < 1)
        return -1;
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0 || cu_seqlens[B] != T)
            return -2;
        for (int64_t s = 0; s < B; ++s)
            if (cu_seqlens[s + 1] < cu_seqlens[s])
                return -2;
    }
    /* Enumerate chunks: (first token, length). */
    int64_t nchunks = 0;
    for (int64_t s = 0; s < B; ++s) {
        int64_t t0 = cu_seqlens ? cu_seqlens[s] : s * T;
        int64_t t1 = cu_seqlens ? cu_seqlens[s + 1] : (s + 1) * T;
        nchunks += (t1 - t0 + C - 1) / C;
    }
    int64_t *cstart = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nchunks + 1));
    int *clen = (int *)malloc(sizeof(int) * (size_t)(nchunks + 1));
    if (!cstart || !clen) {
        free(cstart); free(clen);
        return -1;
    }
    int64_t q = 0;
    for (int64_t s = 0; s < B; ++s) {
        int64_t t0 = cu_seqlens ? cu_seqlens[s] : s * T;
        int64_t t1 = cu_seqlens ? cu_seqlens[s + 1] : (s + 1) * T;
        for (int64_t a = t0; a < t1; a += C) {
            cstart[q] = a;
            clen[q] = (int)((t1 - a) < C ? (t1 - a) : C);
            ++q;
        }
    }
    int status = 0;
    const int64_t units = nchunks * H;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *kc = (double *)malloc(sizeof(double) * (size_t)(C * dk));
        double *vc = (double *)malloc(sizeof(double) * (size_t)(C * dv));
        double *bc = (double *)malloc(sizeof(double) * (size_t)C);
        double *gc = (double *)malloc(sizeof(double) * (size_t)C);
        double *Tc = (double *)malloc(sizeof(double) * (size_t)(C * C));
        double *Wc = (double *)malloc(sizeof(double) * (size_t)(C * dk));
        double *Uc = (double *)malloc(sizeof(double) * (size_t)(C * dv));
        int ok = kc && vc && bc && gc && Tc && Wc && Uc;
#pragma omp for schedule(dynamic, 4)
        for (int64_t u = 0; u < units; ++u) {
            if (!ok)
                continue;
            const int64_t c = u / H, h = u % H;
            const int64_t n0 = cstart[c];
            const int Lc = clen[c];
            for (int i = 0; i < Lc; ++i) {
                const int64_t n = n0 + i;
                memcpy(kc + (int64_t)i * dk, k + (n * H + h) * dk, sizeof(double) * (size_t)dk);
                memcpy(vc + (int64_t)i * dv, v + (n * H + h) * dv, sizeof(double) * (size_t)dv);
                bc[i] = beta[n * H + h];
                if (g)
                    gc[i] = g[n * H + h];
            }
            if (kkt_oracle_chunk(kc, vc, bc, g ? gc : NULL, Lc, (int)C, (int)dk, (int)dv, Tc, Wc, Uc,
                                 NULL) != 0) {
#pragma omp atomic write
                status = -1;
                continue;
            }
            for (int i = 0; i < Lc; ++i) {
                const int64_t n = n0 + i;
                memcpy(T_out + (n * H + h) * C, Tc + (int64_t)i * C, sizeof(double) * (size_t)C);
                memcpy(W_out + (n * H + h) * dk, Wc + (int64_t)i * dk, sizeof(double) * (size_t)dk);
                memcpy(U_out + (n * H + h) * dv, Uc + (int64_t)i * dv, sizeof(double) * (size_t)dv);
            }
        }
        if (!ok) {
#pragma omp atomic write
            status = -1;
        }
        free(kc); free(vc); free(bc); free(gc); free(Tc); free(Wc); free(Uc);
    }
    free(cstart);
    free(clen);
    return status;
}

/* Number of OpenMP threads a parallel region of kkt_oracle_fwd would use. */
int kkt_oracle_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        return nthreads;
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}
