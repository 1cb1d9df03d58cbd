/*
 * gdn_oracle.c -- fp64 CPU oracle for the chunk state recurrence and output of
 * Gated DeltaNet chunked prefill: the computation that consumes W and U~, the
 * outputs of kkt_solve (kkt_oracle.c).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link, load or call this file.  Only
 * tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg
 * use it.  It shares no code, header, table or helper with the CUDA path, and
 * none with kkt_oracle.c either.
 *
 * The recurrence.  The FlashQLA page ("FLA GDN Chunked Prefill 面临的主要问题"
 * and "利用 Gate 衰减性质") recalls the GDN recurrence, but its formula did not
 * survive the page's text extraction; what the pages do state fixes the
 * reading taken here:
 *   - the state S is updated token by token with a write strength beta_t in
 *     (0, 1) and an L2-normalised key k_t ("TileLang 实战：单位下三角矩阵求逆"
 *     §1, the delta rule of the DeltaNet family, whose chunkwise UT transform
 *     gives T, W and U~);
 *   - a per-token decay alpha_t in (0, 1) makes every earlier state's
 *     influence decay exponentially (FlashQLA page, "利用 Gate 衰减性质"),
 *     alpha_t = exp(g_t) with g the `g` input of its API ("使用方式");
 *   - the API takes q, k, v, g, beta, scale and an optional initial state
 *     [B, H_v, K, V], and returns o and the final state.
 * Per sequence and head, with S_t of size dk x dv and S_0 the initial state
 * (zero when none is given):
 *
 *     S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * i.e. the state decays, then the value stored under k_t is replaced by v_t
 * with strength beta_t: S_t = alpha_t S_{t-1} + beta_t k_t (v_t - alpha_t
 * S_{t-1}^T k_t)^T.  Without a gate alpha_t = 1.
 *
 * gdn_oracle_recurrent computes exactly that, one token after another: the
 * definition.
 *
 * gdn_oracle_chunked computes the same result chunk by chunk from W and U~,
 * which is the form the consumer of kkt_solve takes (FlashQLA page,
 * "Tilelang Warp-Specialized Kernel", forward: V', S and O per chunk).  For a
 * chunk of Lc tokens (the chunks of kkt_solve: C tokens, restarting at every
 * sequence start) entered with state S, and G_i = g_0 + ... + g_i the decay
 * from the chunk's start through token i (G = 0 without a gate):
 *
 *     V' = U~ - W S
 *     O  = scale (diag(e^G) Q S + (Gamma o tril(Q K^T)) V'),
 *          Gamma[i][j] = e^{G_i - G_j}, the diagonal included
 *     S <- e^{G_{Lc-1}} S + (diag(e^{G_{Lc-1} - G}) K)^T V'
 *
 * Row i of V' is beta_i times token i's correction (v_i - alpha_i S_{i-1}^T
 * k_i): W S supplies the decayed starting state's part of it (the keys of W
 * carry the decay e^{G_j}) and U~ the rest.  The test suite checks this form,
 * fed with kkt_oracle's W and U~, against gdn_oracle_recurrent.
 *
 * Layouts (the CUDA library's, row-major):
 *   q, k, w [N][H][dk]; v, u, o [N][H][dv]; beta, g [N][H];
 *   h0, ht [nseq][H][dk][dv] (state of sequence s, head h).
 *   N = nseq * T for fixed-length batches (cu_seqlens NULL), or the packed
 *   token count T with nseq + 1 offsets in cu_seqlens.
 * All arithmetic is in double precision on the values the caller passes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int check_bounds(const int64_t *cu, int64_t nseq, int64_t T)
{
    if (!cu)
        return 0;
    if (cu[0] != 0 || cu[nseq] != T)
        return -2;
    for (int64_t s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s])
            return -2;
    return 0;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* One token of the recurrence on the state S (dk x dv, row-major). */
static void recurrent_token(double *S, const double *qt, const double *kt, const double *vt,
                            double bt, double at, double scale, int dk, int dv, double *ot, double *tmp)
{
    /* tmp = S^T k_t (dv) */
    for (int e = 0; e < dv; ++e) {
        double s = 0.0;
        for (int d = 0; d < dk; ++d)
            s += S[(int64_t)d * dv + e] * kt[d];
        tmp[e] = s;
    }
    /* S <- alpha (S - beta k (S^T k)^T) + beta k v^T */
    for (int d = 0; d < dk; ++d)
        for (int e = 0; e < dv; ++e) {
            const int64_t x = (int64_t)d * dv + e;
            S[x] = at * (S[x] - bt * kt[d] * tmp[e]) + bt * kt[d] * vt[e];
        }
    /* o_t = scale S^T q_t */
    for (int e = 0; e < dv; ++e) {
        double s = 0.0;
        for (int d = 0; d < dk; ++d)
            s += S[(int64_t)d * dv + e] * qt[d];
        ot[e] = scale * s;
    }
}

/*
 * The recurrence, token by token.  g may be NULL (no gate), h0 may be NULL
 * (zero initial state), ht may be NULL (final state not wanted).
 * Returns 0, -1 on bad arguments or allocation failure, -2 on a malformed
 * cu_seqlens.
 */
int gdn_oracle_recurrent(const double *q, const double *k, const double *v, const double *beta,
                         const double *g, const double *h0, const int64_t *cu_seqlens, int64_t nseq,
                         int64_t T, int64_t H, int64_t dk, int64_t dv, double scale,
                         double *o, double *ht, int nthreads)
{
    if (nseq < 1 || T < 0 || H < 1 || dk < 1 || dv < 1)
        return -1;
    if (check_bounds(cu_seqlens, nseq, T))
        return -2;
    int status = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
        double *tmp = (double *)malloc(sizeof(double) * (size_t)dv);
        const int ok = S && tmp;
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < nseq * H; ++u) {
            if (!ok)
                continue;
            const int64_t s = u / H, h = u % H;
            const int64_t t0 = cu_seqlens ? cu_seqlens[s] : s * T;
            const int64_t t1 = cu_seqlens ? cu_seqlens[s + 1] : (s + 1) * T;
            const int64_t st = (s * H + h) * dk * dv;
            if (h0)
                memcpy(S, h0 + st, sizeof(double) * (size_t)(dk * dv));
            else
                memset(S, 0, sizeof(double) * (size_t)(dk * dv));
            for (int64_t n = t0; n < t1; ++n) {
                const double at = g ? exp(g[n * H + h]) : 1.0;
                recurrent_token(S, q + (n * H + h) * dk, k + (n * H + h) * dk, v + (n * H + h) * dv,
                                beta[n * H + h], at, scale, (int)dk, (int)dv, o + (n * H + h) * dv, tmp);
            }
            if (ht)
                memcpy(ht + st, S, sizeof(double) * (size_t)(dk * dv));
        }
        if (!ok) {
#pragma omp atomic write
            status = -1;
        }
        free(S);
        free(tmp);
    }
    return status;
}

/* One chunk of the chunkwise form: rows n0 .. n0+Lc-1 of head h, state S updated in place. */
static void chunk_step(double *S, const double *q, const double *k, const double *w, const double *u,
                       const double *g, int64_t n0, int Lc, int64_t H, int64_t h, int dk, int dv,
                       double scale, double *o, double *G, double *Vp)
{
    /* G_i: the decay from the chunk's start through token i, in log units */
    double acc = 0.0;
    for (int i = 0; i < Lc; ++i) {
        if (g)
            acc += g[(n0 + i) * H + h];
        G[i] = acc;
    }
    /* V' = U~ - W S */
    for (int i = 0; i < Lc; ++i) {
        const double *wi = w + ((n0 + i) * H + h) * dk;
        const double *ui = u + ((n0 + i) * H + h) * dv;
        for (int e = 0; e < dv; ++e) {
            double s = 0.0;
            for (int d = 0; d < dk; ++d)
                s += wi[d] * S[(int64_t)d * dv + e];
            Vp[(int64_t)i * dv + e] = ui[e] - s;
        }
    }
    /* O = scale (diag(e^G) Q S + (Gamma o tril(Q K^T)) V') */
    for (int i = 0; i < Lc; ++i) {
        const double *qi = q + ((n0 + i) * H + h) * dk;
        double *oi = o + ((n0 + i) * H + h) * dv;
        const double gi = exp(G[i]);
        for (int e = 0; e < dv; ++e) {
            double s = 0.0;
            for (int d = 0; d < dk; ++d)
                s += qi[d] * S[(int64_t)d * dv + e];
            oi[e] = gi * s;
        }
        for (int j = 0; j <= i; ++j) {
            const double *kj = k + ((n0 + j) * H + h) * dk;
            double qk = 0.0;
            for (int d = 0; d < dk; ++d)
                qk += qi[d] * kj[d];
            const double c = exp(G[i] - G[j]) * qk;
            for (int e = 0; e < dv; ++e)
                oi[e] += c * Vp[(int64_t)j * dv + e];
        }
        for (int e = 0; e < dv; ++e)
            oi[e] *= scale;
    }
    /* S <- e^{G_last} S + (diag(e^{G_last - G}) K)^T V' */
    const double glast = G[Lc - 1];
    const double decay = exp(glast);
    for (int d = 0; d < dk; ++d)
        for (int e = 0; e < dv; ++e)
            S[(int64_t)d * dv + e] *= decay;
    for (int j = 0; j < Lc; ++j) {
        const double *kj = k + ((n0 + j) * H + h) * dk;
        const double f = exp(glast - G[j]);
        for (int d = 0; d < dk; ++d) {
            const double kd = f * kj[d];
            for (int e = 0; e < dv; ++e)
                S[(int64_t)d * dv + e] += kd * Vp[(int64_t)j * dv + e];
        }
    }
}

/*
 * The chunkwise form from W and U~ (chunks of C tokens restarting at every
 * sequence start).  g, h0 and ht as in gdn_oracle_recurrent.
 * Returns 0, -1 on bad arguments or allocation failure, -2 on a malformed
 * cu_seqlens.
 */
int gdn_oracle_chunked(const double *q, const double *k, const double *w, const double *u,
                       const double *g, const double *h0, const int64_t *cu_seqlens, int64_t nseq,
                       int64_t T, int64_t H, int64_t dk, int64_t dv, int64_t C, double scale,
                       double *o, double *ht, int nthreads)
{
    if (nseq < 1 || T < 0 || H < 1 || dk < 1 || dv < 1 || C < 1)
        return -1;
    if (check_bounds(cu_seqlens, nseq, T))
        return -2;
    int status = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
        double *G = (double *)malloc(sizeof(double) * (size_t)C);
        double *Vp = (double *)malloc(sizeof(double) * (size_t)(C * dv));
        const int ok = S && G && Vp;
#pragma omp for schedule(dynamic, 1)
        for (int64_t x = 0; x < nseq * H; ++x) {
            if (!ok)
                continue;
            const int64_t s = x / H, h = x % H;
            const int64_t t0 = cu_seqlens ? cu_seqlens[s] : s * T;
            const int64_t t1 = cu_seqlens ? cu_seqlens[s + 1] : (s + 1) * T;
            const int64_t st = (s * H + h) * dk * dv;
            if (h0)
                memcpy(S, h0 + st, sizeof(double) * (size_t)(dk * dv));
            else
                memset(S, 0, sizeof(double) * (size_t)(dk * dv));
            for (int64_t n0 = t0; n0 < t1; n0 += C) {
                const int Lc = (int)((t1 - n0) < C ? (t1 - n0) : C);
                chunk_step(S, q, k, w, u, g, n0, Lc, H, h, (int)dk, (int)dv, scale, o, G, Vp);
            }
            if (ht)
                memcpy(ht + st, S, sizeof(double) * (size_t)(dk * dv));
        }
        if (!ok) {
#pragma omp atomic write
            status = -1;
        }
        free(S);
        free(G);
        free(Vp);
    }
    return status;
}
