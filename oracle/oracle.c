/*
 * oracle.c -- plain, slow, fp64 CPU definition of masked multi-head attention
 * and of the Pre-LayerNorm cross-attention variant.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity oracle for the CUDA
 * kernels in masked_head_attention_gb300/csrc.  It shares no code, header,
 * table or constant with them and neither side includes the other.  Only the
 * tests, the smoke check in __graft_entry__ and the cpu_baseline leg of
 * bench.py may load it.  The product path never calls it.
 *
 * Sources (pages cited by title and section):
 *  - "How to fuse cross-attention and layer-norm into a single CUDA kernel?"
 *    (cms365.cn interview answer), section "Knowledge points": the chain
 *    S = Q K^T -> P = softmax(S) -> O = P V, softmax per row with max and sum.
 *  - Same page, "Answer", step two: Pre-LayerNorm of the query rows with
 *    per-row mean and variance, then gamma/beta applied to Q.
 *  - "masked multi head attention" CUDA article (2kiu.com/news/6063113),
 *    section 3.1: causal rule, position (row, col) is kept when row >= col and
 *    otherwise its logit becomes -infinity before the softmax; section 3.2:
 *    subtract the row maximum before exponentiating.
 *  - "Why attention must compute the max first" essay (gsyq.cn/news/340375),
 *    section 2.1: three-pass softmax (max, exp-sum, divide); section 3.1:
 *    every shifted logit is <= 0, so every exponential is in [0, 1];
 *    section 5.2: logits are divided by sqrt(d_k); section 3.3: the softmax
 *    Jacobian d p_j / d s_k = p_j (delta_jk - p_k), used by the backward
 *    pass (oracle_mha_bwd) together with the row log-sum-exp (oracle_mha_lse).
 *
 * Readings taken where the pages are silent:
 *  - scale is passed explicitly (the kernels' default is 1/sqrt(D));
 *  - causal alignment is top-left: key j is visible to query i iff j <= i;
 *  - the padding mask hides keys j >= len_b; query rows are all computed;
 *  - len_b is clamped to [0, Lk];
 *  - a row with no visible key returns a row of zeros (and so passes no
 *    gradient back: its output is a constant);
 *  - the backward pass is the gradient of L = sum(dout * O) with respect to
 *    q, k and v, in the same fp64 arithmetic;
 *  - LayerNorm uses the biased variance (divide by N) and eps inside the
 *    square root; Q is the head slice of LN(x), with no projection after it.
 *
 * Every function here is the definition written out, in fp64, with no
 * blocking, fusion or reordering beyond it.  The only parallelism is OpenMP
 * over independent (b, h) problems, which does not change any result.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_MASK_CAUSAL 1
#define ORC_MASK_KV_LEN 2

/* Number of host threads OpenMP will use (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Effective key length of batch b: Lk, or len_b clamped to [0, Lk]. */
static int visible_len(int mask_kind, const int32_t *kv_lengths, int b, int Lk) {
    if (!(mask_kind & ORC_MASK_KV_LEN) || kv_lengths == NULL) return Lk;
    int len = kv_lengths[b];
    if (len < 0) len = 0;
    if (len > Lk) len = Lk;
    return len;
}

/* Mask rule: 2kiu.com article section 3.1 (causal, row >= col) and the
 * per-sequence padding rule (keys at or beyond the valid length are hidden). */
static int key_visible(int i, int j, int mask_kind, int len) {
    if (j >= len) return 0;
    if ((mask_kind & ORC_MASK_CAUSAL) && j > i) return 0;
    return 1;
}

/*
 * One query row of one (b, h) problem.
 *   qi  : D values of query row i
 *   K,V : Lk x D, row-major
 *   s   : Lk scratch values (logits, then unnormalised weights)
 *   o   : D outputs
 *   p   : optional Lk outputs, the softmax row (0 at hidden keys)
 * Pass 1 forms the scaled logits and their maximum over visible keys, pass 2
 * the shifted exponentials and their sum, pass 3 divides and contracts with V.
 */
static void attend_row(const double *qi, const double *K, const double *V,
                       int Lk, int D, double scale, int mask_kind, int len,
                       int i, double *s, double *o, double *p) {
    double M = -INFINITY;
    int any = 0;
    for (int j = 0; j < Lk; ++j) {
        if (!key_visible(i, j, mask_kind, len)) continue;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qi[d] * K[(size_t)j * D + d];
        s[j] = scale * dot;
        if (!any || s[j] > M) M = s[j];
        any = 1;
    }
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (!any) {
        if (p) for (int j = 0; j < Lk; ++j) p[j] = 0.0;
        return;
    }
    double Z = 0.0;
    for (int j = 0; j < Lk; ++j) {
        if (!key_visible(i, j, mask_kind, len)) { s[j] = 0.0; continue; }
        s[j] = exp(s[j] - M);
        Z += s[j];
    }
    for (int j = 0; j < Lk; ++j) {
        double w = s[j] / Z;          /* exactly 0 at hidden keys */
        if (p) p[j] = w;
        if (w == 0.0) continue;
        for (int d = 0; d < D; ++d) o[d] += w * V[(size_t)j * D + d];
    }
}

static int bad_shape(int B, int H, int Lq, int Lk, int D) {
    return B < 0 || H < 0 || Lq < 0 || Lk < 0 || D <= 0;
}

/*
 * Full forward: q [B,H,Lq,D], k and v [B,H,Lk,D], out [B,H,Lq,D], all fp64
 * row-major.  kv_lengths [B] is read only when mask_kind has the KV_LEN bit.
 * Returns 0, or -1 for a bad shape, -2 when the scratch allocation fails.
 */
int oracle_mha_fwd(const double *q, const double *k, const double *v,
                   int mask_kind, const int32_t *kv_lengths, double *out,
                   int B, int H, int Lq, int Lk, int D, double scale) {
    if (bad_shape(B, H, Lq, Lk, D)) return -1;
    int fail = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : fail)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
            if (!s) { fail = 1; continue; }
            size_t bh = (size_t)b * H + h;
            const double *Q = q + bh * (size_t)Lq * D;
            const double *K = k + bh * (size_t)Lk * D;
            const double *V = v + bh * (size_t)Lk * D;
            double *O = out + bh * (size_t)Lq * D;
            int len = visible_len(mask_kind, kv_lengths, b, Lk);
            for (int i = 0; i < Lq; ++i)
                attend_row(Q + (size_t)i * D, K, V, Lk, D, scale, mask_kind, len,
                           i, s, O + (size_t)i * D, NULL);
            free(s);
        }
    }
    return fail ? -2 : 0;
}

/*
 * Selected rows only, for checks at sizes where the full oracle is too slow.
 * rows holds n triples (b, h, i); out_rows receives n x D values.
 */
int oracle_mha_rows(const double *q, const double *k, const double *v,
                    int mask_kind, const int32_t *kv_lengths,
                    const int64_t *rows, int64_t n, double *out_rows,
                    int B, int H, int Lq, int Lk, int D, double scale) {
    if (bad_shape(B, H, Lq, Lk, D)) return -1;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : fail)
    for (int64_t r = 0; r < n; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= Lq) { fail = 1; continue; }
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        if (!s) { fail = 1; continue; }
        size_t bh = (size_t)b * H + (size_t)h;
        attend_row(q + (bh * Lq + (size_t)i) * D, k + bh * (size_t)Lk * D,
                   v + bh * (size_t)Lk * D, Lk, D, scale, mask_kind,
                   visible_len(mask_kind, kv_lengths, (int)b, Lk), (int)i, s,
                   out_rows + (size_t)r * D, NULL);
        free(s);
    }
    return fail ? -1 : 0;
}

/*
 * The softmax matrix itself, p [B,H,Lq,Lk], for small cases: lets the tests
 * check that each row sums to one and is exactly zero at hidden keys.
 */
int oracle_softmax_probs(const double *q, const double *k, int mask_kind,
                         const int32_t *kv_lengths, double *p,
                         int B, int H, int Lq, int Lk, int D, double scale) {
    if (bad_shape(B, H, Lq, Lk, D)) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
    double *o = (double *)malloc(sizeof(double) * (size_t)D);
    double *zeros = (double *)calloc((size_t)(Lk > 0 ? Lk : 1) * (size_t)D, sizeof(double));
    if (!s || !o || !zeros) { free(s); free(o); free(zeros); return -2; }
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            size_t bh = (size_t)b * H + h;
            int len = visible_len(mask_kind, kv_lengths, b, Lk);
            for (int i = 0; i < Lq; ++i)
                attend_row(q + (bh * Lq + (size_t)i) * D, k + bh * (size_t)Lk * D,
                           zeros, Lk, D, scale, mask_kind, len, i, s, o,
                           p + (bh * Lq + (size_t)i) * Lk);
        }
    free(s); free(o); free(zeros);
    return 0;
}

/*
 * LayerNorm over the last dimension (cms365.cn answer, step two):
 * y = (x - mean) / sqrt(var + eps) * gamma + beta, with mean and the biased
 * variance taken over the N features of each row, in two plain passes.
 */
int oracle_layer_norm(const double *x, const double *gamma, const double *beta,
                      double eps, double *y, int64_t rows, int N) {
    if (rows < 0 || N <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + (size_t)r * N;
        double mean = 0.0;
        for (int c = 0; c < N; ++c) mean += xr[c];
        mean /= N;
        double var = 0.0;
        for (int c = 0; c < N; ++c) var += (xr[c] - mean) * (xr[c] - mean);
        var /= N;
        double rstd = 1.0 / sqrt(var + eps);
        for (int c = 0; c < N; ++c)
            y[(size_t)r * N + c] = (xr[c] - mean) * rstd * gamma[c] + beta[c];
    }
    return 0;
}

/* Head split of a [B, Lq, H*D] activation into [B, H, Lq, D]. */
static void split_heads(const double *x, double *q, int B, int H, int Lq, int D) {
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < Lq; ++i)
            for (int h = 0; h < H; ++h)
                for (int d = 0; d < D; ++d)
                    q[(((size_t)b * H + h) * Lq + i) * D + d] =
                        x[((size_t)b * Lq + i) * (size_t)H * D + (size_t)h * D + d];
}

/* Inverse of split_heads: [B, H, Lq, D] back to [B, Lq, H*D]. */
static void merge_heads(const double *o, double *y, int B, int H, int Lq, int D) {
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < Lq; ++i)
            for (int h = 0; h < H; ++h)
                for (int d = 0; d < D; ++d)
                    y[((size_t)b * Lq + i) * (size_t)H * D + (size_t)h * D + d] =
                        o[(((size_t)b * H + h) * Lq + i) * D + d];
}

/*
 * Pre-LayerNorm cross-attention (cms365.cn answer, steps two and three):
 * Q = heads(LN(x)), O = attention(Q, K, V) with the padding mask only, and
 * out = [B, Lq, H*D].  x is [B, Lq, H*D]; k, v are [B, H, Lk, D].
 */
int oracle_prenorm_cross_attn(const double *x, const double *gamma,
                              const double *beta, double eps,
                              const double *k, const double *v,
                              const int32_t *kv_lengths, double *out,
                              int B, int H, int Lq, int Lk, int D, double scale) {
    if (bad_shape(B, H, Lq, Lk, D)) return -1;
    size_t n = (size_t)B * Lq * (size_t)H * D;
    double *xn = (double *)malloc(sizeof(double) * (n ? n : 1));
    double *q = (double *)malloc(sizeof(double) * (n ? n : 1));
    double *o = (double *)malloc(sizeof(double) * (n ? n : 1));
    int rc = -2;
    if (xn && q && o) {
        rc = oracle_layer_norm(x, gamma, beta, eps, xn, (int64_t)B * Lq, H * D);
        if (rc == 0) {
            split_heads(xn, q, B, H, Lq, D);
            rc = oracle_mha_fwd(q, k, v, kv_lengths ? ORC_MASK_KV_LEN : 0,
                                kv_lengths, o, B, H, Lq, Lk, D, scale);
        }
        if (rc == 0) merge_heads(o, out, B, H, Lq, D);
    }
    free(xn); free(q); free(o);
    return rc;
}

/*
 * Selected output rows of the Pre-LN variant.  rows holds n triples
 * (b, h, i); out_rows receives n x D values, the slice of out[b, i, :] that
 * belongs to head h.
 */
int oracle_prenorm_rows(const double *x, const double *gamma, const double *beta,
                        double eps, const double *k, const double *v,
                        const int32_t *kv_lengths, const int64_t *rows, int64_t n,
                        double *out_rows, int B, int H, int Lq, int Lk, int D,
                        double scale) {
    if (bad_shape(B, H, Lq, Lk, D)) return -1;
    int N = H * D;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : fail)
    for (int64_t r = 0; r < n; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= Lq) { fail = 1; continue; }
        double *xn = (double *)malloc(sizeof(double) * (size_t)N);
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        if (!xn || !s) { free(xn); free(s); fail = 1; continue; }
        oracle_layer_norm(x + ((size_t)b * Lq + (size_t)i) * N, gamma, beta, eps, xn, 1, N);
        size_t bh = (size_t)b * H + (size_t)h;
        int mk = kv_lengths ? ORC_MASK_KV_LEN : 0;
        attend_row(xn + (size_t)h * D, k + bh * (size_t)Lk * D, v + bh * (size_t)Lk * D,
                   Lk, D, scale, mk, visible_len(mk, kv_lengths, (int)b, Lk), (int)i, s,
                   out_rows + (size_t)r * D, NULL);
        free(xn); free(s);
    }
    return fail ? -1 : 0;
}

/*
 * Pre-LN cross-attention with the residual add of the same page ("How to
 * fuse cross-attention and layer-norm into a single CUDA kernel?", answer
 * step four: the attention output is added to the query-side input src):
 * out = x + prenorm_cross_attn(x).  Same shapes as oracle_prenorm_cross_attn.
 */
int oracle_prenorm_cross_attn_residual(const double *x, const double *gamma,
                                       const double *beta, double eps,
                                       const double *k, const double *v,
                                       const int32_t *kv_lengths, double *out,
                                       int B, int H, int Lq, int Lk, int D,
                                       double scale) {
    int rc = oracle_prenorm_cross_attn(x, gamma, beta, eps, k, v, kv_lengths, out,
                                       B, H, Lq, Lk, D, scale);
    if (rc != 0) return rc;
    size_t n = (size_t)B * Lq * (size_t)H * D;
    for (size_t e = 0; e < n; ++e) out[e] = x[e] + out[e];
    return 0;
}

/*
 * Selected rows of the residual variant: rows holds n triples (b, h, i);
 * out_rows receives n x D values, x[b, i, h*D .. h*D + D) plus the head-h
 * slice of the attention output of row (b, i).
 */
int oracle_prenorm_residual_rows(const double *x, const double *gamma,
                                 const double *beta, double eps, const double *k,
                                 const double *v, const int32_t *kv_lengths,
                                 const int64_t *rows, int64_t n, double *out_rows,
                                 int B, int H, int Lq, int Lk, int D, double scale) {
    int rc = oracle_prenorm_rows(x, gamma, beta, eps, k, v, kv_lengths, rows, n, out_rows,
                                 B, H, Lq, Lk, D, scale);
    if (rc != 0) return rc;
    for (int64_t r = 0; r < n; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        const double *src = x + ((size_t)b * Lq + (size_t)i) * (size_t)H * D + (size_t)h * D;
        for (int d = 0; d < D; ++d) out_rows[(size_t)r * D + d] = src[d] + out_rows[(size_t)r * D + d];
    }
    return 0;
}


/*
 * Log-sum-exp of each row's scaled logits over its visible keys, the softmax
 * statistic a backward pass recomputes the weights from:
 *     lse[b,h,i] = log sum_{visible j} exp(s_ij),   s_ij = scale * q_i . k_j,
 * taken as M + log(sum exp(s_ij - M)) with M the row maximum (the max-first
 * order of the gsyq.cn essay "Why attention must compute the max first",
 * sections 2.1 and 3.1).  A row with no visible key gets -INFINITY.
 * q [B,H,Lq,D], k [B,H,Lk,D], lse [B,H,Lq].
 */
int oracle_mha_lse(const double *q, const double *k, int mask_kind,
                   const int32_t *kv_lengths, double *lse,
                   int B, int H, int Lq, int Lk, int D, double scale) {
    if (bad_shape(B, H, Lq, Lk, D)) return -1;
    int fail = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : fail)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
            if (!s) { fail = 1; continue; }
            size_t bh = (size_t)b * H + h;
            const double *Q = q + bh * (size_t)Lq * D;
            const double *K = k + bh * (size_t)Lk * D;
            int len = visible_len(mask_kind, kv_lengths, b, Lk);
            for (int i = 0; i < Lq; ++i) {
                double M = -INFINITY;
                int any = 0;
                for (int j = 0; j < Lk; ++j) {
                    if (!key_visible(i, j, mask_kind, len)) continue;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += Q[(size_t)i * D + d] * K[(size_t)j * D + d];
                    s[j] = dot * scale;
                    if (!any || M < s[j]) M = s[j];
                    any = 1;
                }
                if (!any) { lse[bh * Lq + (size_t)i] = -INFINITY; continue; }
                double Z = 0.0;
                for (int j = 0; j < Lk; ++j)
                    if (key_visible(i, j, mask_kind, len)) Z += exp(s[j] - M);
                lse[bh * Lq + (size_t)i] = M + log(Z);
            }
            free(s);
        }
    }
    return fail ? -2 : 0;
}

/*
 * Gradients of the forward above for the loss L = sum(dout * O), i.e. the
 * backward pass: dq [B,H,Lq,D], dk and dv [B,H,Lk,D] from dout [B,H,Lq,D].
 * Per query row i the softmax row p_i is formed again (attend_row), then the
 * softmax Jacobian of the gsyq.cn essay, section 3.3,
 *     d p_ij / d s_ik = p_ij (delta_jk - p_ik),
 * is applied to dP_ij = dL/dp_ij = dout_i . v_j:
 *     c_i   = sum_j p_ij dP_ij
 *     dS_ij = p_ij (dP_ij - c_i)
 * and the three products are accumulated over the visible keys j:
 *     dv_j += p_ij dout_i
 *     dq_i += scale * dS_ij k_j
 *     dk_j += scale * dS_ij q_i
 * Hidden keys have p_ij = 0 and receive nothing; a row with no visible key
 * has a constant (zero) output and contributes nothing.
 */
int oracle_mha_bwd(const double *q, const double *k, const double *v,
                   const double *dout, int mask_kind, const int32_t *kv_lengths,
                   double *dq, double *dk, double *dv,
                   int B, int H, int Lq, int Lk, int D, double scale) {
    if (bad_shape(B, H, Lq, Lk, D)) return -1;
    int fail = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(| : fail)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            size_t nk = (size_t)(Lk > 0 ? Lk : 1);
            double *s = (double *)malloc(sizeof(double) * nk);
            double *p = (double *)malloc(sizeof(double) * nk);
            double *dP = (double *)malloc(sizeof(double) * nk);
            double *o = (double *)malloc(sizeof(double) * (size_t)D);
            if (!s || !p || !dP || !o) {
                free(s); free(p); free(dP); free(o);
                fail = 1;
                continue;
            }
            size_t bh = (size_t)b * H + h;
            const double *Q = q + bh * (size_t)Lq * D;
            const double *K = k + bh * (size_t)Lk * D;
            const double *V = v + bh * (size_t)Lk * D;
            const double *dO = dout + bh * (size_t)Lq * D;
            double *dQ = dq + bh * (size_t)Lq * D;
            double *dK = dk + bh * (size_t)Lk * D;
            double *dV = dv + bh * (size_t)Lk * D;
            for (size_t e = 0; e < (size_t)Lq * D; ++e) dQ[e] = 0.0;
            for (size_t e = 0; e < (size_t)Lk * D; ++e) { dK[e] = 0.0; dV[e] = 0.0; }
            int len = visible_len(mask_kind, kv_lengths, b, Lk);
            for (int i = 0; i < Lq; ++i) {
                const double *qi = Q + (size_t)i * D;
                const double *gi = dO + (size_t)i * D;
                attend_row(qi, K, V, Lk, D, scale, mask_kind, len, i, s, o, p);
                double c = 0.0;
                for (int j = 0; j < Lk; ++j) {
                    dP[j] = 0.0;
                    if (!key_visible(i, j, mask_kind, len)) continue;
                    for (int d = 0; d < D; ++d) dP[j] += gi[d] * V[(size_t)j * D + d];
                    c += p[j] * dP[j];
                }
                for (int j = 0; j < Lk; ++j) {
                    if (!key_visible(i, j, mask_kind, len)) continue;
                    double dS = p[j] * (dP[j] - c);
                    for (int d = 0; d < D; ++d) {
                        dV[(size_t)j * D + d] += p[j] * gi[d];
                        dQ[(size_t)i * D + d] += scale * dS * K[(size_t)j * D + d];
                        dK[(size_t)j * D + d] += scale * dS * qi[d];
                    }
                }
            }
            free(s); free(p); free(dP); free(o);
        }
    }
    return fail ? -2 : 0;
}
