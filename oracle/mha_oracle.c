/*
 * Float64 CPU oracle for multi-head scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the tests, the package's smoke entry and the benchmark's CPU-baseline leg
 * may build, load or call it.  It shares no code, header, table or helper with
 * the CUDA library, and it includes nothing from it.
 *
 * What it computes, for every sequence b, head h and query row i
 * ("Attention Is All You Need", Section 3.2.1, Equation (1):
 *  Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V, applied to every head in
 *  parallel as in Section 3.2.2 and the cookipedia article, section
 *  "Transformer の構造"), written out one row at a time as the formula page
 *  (transformer-attention, section 証明) states it:
 *
 *   1. score      s_j = scale * (q . k_j)                (証明, first step)
 *   2. weights    a_j = e^{s_j} / sum_i e^{s_i}          (証明, second step)
 *   3. output     o   = sum_j a_j v_j                    (証明, third step)
 *
 * Readings taken where the pages leave a step open:
 *   - scale defaults to 1/sqrt(d_k) (Equation (1) and the cookipedia article;
 *     the formula page's rendering drops the square root, but its own worked
 *     example divides by 2 for d_k = 4).  The caller passes it explicitly.
 *   - the causal mask (cookipedia, decoder section; formula page, 応用,
 *     "先を読まない仕掛け") removes key j > i, keeping the diagonal; a removed
 *     key has weight exactly 0 and is left out of the sum.
 *   - key padding (not on the pages): keys j >= key_lens[b] are removed for
 *     every head and query of sequence b; key_lens[b] is clamped to [0, Lk].
 *   - both masks together (mask kind 3, a decoder over padded sequences):
 *     key j is visible to row i when it passes both, j <= i and
 *     j < key_lens[b].
 *   - d_v may differ from d_k (Equation (1) takes values of dimension d_v):
 *     scores use the d_k columns of q and k, the output has the d_v columns
 *     of v.
 *   - a row with no visible key has output 0 and log-sum-exp -inf.
 *   - before the exponentials the row maximum m is subtracted from every
 *     score.  The formula page (証明, weight-ratio step) shows that adding one
 *     constant to all scores leaves the weights unchanged, so this changes
 *     nothing but the rounding and keeps e^{s} from overflowing.
 *
 * Layout: q is [B, Lq, H, d_k], k is [B, Lk, H, d_k], v is [B, Lk, H, d_v],
 * out is [B, Lq, H, d_v], all row-major float64 (the head split of a
 * d_model = H*d vector per step is the innermost H*d block).  lse (optional, may be NULL) is [B, H, Lq] and
 * receives m + log(sum_j e^{s_j - m}) of each row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    ORACLE_MASK_NONE = 0,
    ORACLE_MASK_CAUSAL = 1,
    ORACLE_MASK_KEY_PADDING = 2,
    ORACLE_MASK_CAUSAL_KEY_PADDING = 3  /* both */
};

/* Number of keys row i of sequence b may attend to: keys 0 .. n-1. */
static int64_t visible_keys(int64_t i, int64_t b, int64_t Lk, int mask_kind,
                            const int32_t* key_lens)
{
    int64_t n = Lk;
    if (mask_kind & ORACLE_MASK_CAUSAL) {
        n = i + 1 < Lk ? i + 1 : Lk;
    }
    if (mask_kind & ORACLE_MASK_KEY_PADDING) {
        int64_t len = key_lens[b];
        if (len < 0) len = 0;
        if (len > Lk) len = Lk;
        if (len < n) n = len;
    }
    return n;
}

/* The argument rules both entry points share: 0 when the mask is usable. */
static int check_mask(int mask_kind, int64_t B, int64_t Lq, int64_t Lk,
                      const int32_t* key_lens)
{
    if (mask_kind < ORACLE_MASK_NONE || mask_kind > ORACLE_MASK_CAUSAL_KEY_PADDING) return 1;
    if ((mask_kind & ORACLE_MASK_CAUSAL) && Lq != Lk) return 1;
    if ((mask_kind & ORACLE_MASK_KEY_PADDING) && key_lens == NULL && B > 0) return 1;
    return 0;
}

/* One query row.  s is caller-provided scratch of at least Lk doubles. */
static void attend_row(const double* q_row, const double* k, const double* v,
                       double* o_row, double* lse_out, int64_t n, int64_t d_k,
                       int64_t d_v, int64_t k_row_stride, int64_t v_row_stride,
                       double scale, double* s)
{
    if (n == 0) {
        for (int64_t c = 0; c < d_v; ++c) o_row[c] = 0.0;
        if (lse_out) *lse_out = -INFINITY;
        return;
    }
    /* 1. scores */
    for (int64_t j = 0; j < n; ++j) {
        const double* k_row = k + j * k_row_stride;
        double dot = 0.0;
        for (int64_t c = 0; c < d_k; ++c) dot += q_row[c] * k_row[c];
        s[j] = scale * dot;
    }
    /* 2. weights, with the row maximum taken out of every exponent */
    double m = s[0];
    for (int64_t j = 1; j < n; ++j)
        if (s[j] > m) m = s[j];
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        sum += s[j];
    }
    for (int64_t j = 0; j < n; ++j) s[j] /= sum;
    /* 3. weighted mean of the value rows */
    for (int64_t c = 0; c < d_v; ++c) o_row[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double* v_row = v + j * v_row_stride;
        for (int64_t c = 0; c < d_v; ++c) o_row[c] += s[j] * v_row[c];
    }
    if (lse_out) *lse_out = m + log(sum);
}

/*
 * Returns 0 on success, 1 on a bad argument (negative size, NULL pointer
 * where data is needed, unknown mask kind, causal with Lq != Lk), 2 when the
 * score scratch cannot be allocated.
 * n_threads <= 0 uses the OpenMP default.  Rows are independent, so the
 * thread count changes no result bit.
 */
int oracle_mha_dv_f64(const double* q, const double* k, const double* v,
                      double* out, double* lse,
                      int64_t B, int64_t H, int64_t Lq, int64_t Lk, int64_t d_k,
                      int64_t d_v, int mask_kind, const int32_t* key_lens, double scale,
                      int n_threads)
{
    if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || d_k < 1 || d_v < 1) return 1;
    if (check_mask(mask_kind, B, Lq, Lk, key_lens) != 0) return 1;
    const int64_t rows = B * H * Lq;
    if (rows == 0) return 0;
    if (q == NULL || out == NULL) return 1;
    if (Lk > 0 && (k == NULL || v == NULL)) return 1;

#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#else
    n_threads = 1;
#endif
    /* one score buffer of Lk doubles per thread */
    const int64_t per_thread = Lk > 0 ? Lk : 1;
    double* scratch = (double*)malloc((size_t)n_threads * (size_t)per_thread * sizeof(double));
    if (scratch == NULL) return 2;
#ifdef _OPENMP
#pragma omp parallel for num_threads(n_threads) schedule(dynamic, 8)
#endif
    for (int64_t r = 0; r < rows; ++r) {
#ifdef _OPENMP
        double* s = scratch + (int64_t)omp_get_thread_num() * per_thread;
#else
        double* s = scratch;
#endif
        /* row r enumerates (b, h, i) with i fastest */
        const int64_t i = r % Lq;
        const int64_t h = (r / Lq) % H;
        const int64_t b = r / (Lq * H);
        const int64_t n = visible_keys(i, b, Lk, mask_kind, key_lens);
        const double* q_row = q + ((b * Lq + i) * H + h) * d_k;
        const double* k_bh = k ? k + (b * Lk * H + h) * d_k : NULL;
        const double* v_bh = v ? v + (b * Lk * H + h) * d_v : NULL;
        double* o_row = out + ((b * Lq + i) * H + h) * d_v;
        double* lse_row = lse ? lse + (b * H + h) * Lq + i : NULL;
        attend_row(q_row, k_bh, v_bh, o_row, lse_row, n, d_k, d_v, H * d_k, H * d_v, scale, s);
    }
    free(scratch);
    return 0;
}

/* The same with d_v = d_k = d. */
int oracle_mha_f64(const double* q, const double* k, const double* v,
                   double* out, double* lse,
                   int64_t B, int64_t H, int64_t Lq, int64_t Lk, int64_t d,
                   int mask_kind, const int32_t* key_lens, double scale,
                   int n_threads)
{
    return oracle_mha_dv_f64(q, k, v, out, lse, B, H, Lq, Lk, d, d, mask_kind, key_lens,
                             scale, n_threads);
}

/*
 * Gradient ("backward") of the same operation for a loss L whose gradient
 * with respect to the output is dout (layout of out): dq, dk, dv receive
 * dL/dq, dL/dk, dL/dv (layouts of q, k, v).  For every row, with the scores
 * s_j and weights a_j of steps 1 and 2:
 *
 *   4. g_j      = dL/da_j = dout . v_j           (step 3: o = sum_j a_j v_j)
 *   5. dL/ds_i  = sum_j g_j da_j/ds_i with the formula page's derivative of the
 *                 weights by the scores, da_j/ds_i = a_j (delta_ij - a_i)
 *                 (証明, the step after the temperature form), which sums to
 *                 dL/ds_i = a_i (g_i - sum_j a_j g_j)
 *   6. dq      += scale * sum_j dL/ds_j k_j        (step 1: s_j = scale q . k_j)
 *      dk_j    += scale * dL/ds_j q
 *      dv_j    += a_j dout                        (step 3)
 *
 * Removed keys (mask, padding, rows past Lk) get no gradient; a row with no
 * visible key contributes nothing.  (b, h) pairs are independent and the rows
 * of one pair are visited in order, so no result depends on the thread count.
 * Returns as oracle_mha_f64.
 */
int oracle_mha_bwd_f64(const double* q, const double* k, const double* v,
                       const double* dout, double* dq, double* dk, double* dv,
                       int64_t B, int64_t H, int64_t Lq, int64_t Lk, int64_t d,
                       int mask_kind, const int32_t* key_lens, double scale,
                       int n_threads)
{
    if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || d < 1) return 1;
    if (check_mask(mask_kind, B, Lq, Lk, key_lens) != 0) return 1;
    if (B * H == 0) return 0;
    if (Lq > 0 && (q == NULL || dout == NULL || dq == NULL)) return 1;
    if (Lk > 0 && (k == NULL || v == NULL || dk == NULL || dv == NULL)) return 1;
    for (int64_t x = 0; x < B * Lk * H * d; ++x) {
        dk[x] = 0.0;
        dv[x] = 0.0;
    }

#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#else
    n_threads = 1;
#endif
    /* weights a and upstream gradients g: 2 Lk doubles per thread */
    const int64_t per_thread = 2 * (Lk > 0 ? Lk : 1);
    double* scratch = (double*)malloc((size_t)n_threads * (size_t)per_thread * sizeof(double));
    if (scratch == NULL) return 2;
    const int64_t pairs = B * H;
#ifdef _OPENMP
#pragma omp parallel for num_threads(n_threads) schedule(dynamic, 1)
#endif
    for (int64_t bh = 0; bh < pairs; ++bh) {
#ifdef _OPENMP
        double* a = scratch + (int64_t)omp_get_thread_num() * per_thread;
#else
        double* a = scratch;
#endif
        double* g = a + per_thread / 2;
        const int64_t b = bh / H, h = bh % H;
        const int64_t rs = H * d;  /* stride between consecutive rows of one head */
        const int64_t kv_off = (b * Lk * H + h) * d;  /* key 0 of head h */
        const double* k_bh = k ? k + kv_off : NULL;
        const double* v_bh = v ? v + kv_off : NULL;
        double* dk_bh = dk ? dk + kv_off : NULL;
        double* dv_bh = dv ? dv + kv_off : NULL;
        for (int64_t i = 0; i < Lq; ++i) {
            const int64_t row_off = ((b * Lq + i) * H + h) * d;  /* row i of head h */
            const double* q_row = q + row_off;
            const double* do_row = dout + row_off;
            double* dq_row = dq + row_off;
            for (int64_t c = 0; c < d; ++c) dq_row[c] = 0.0;
            const int64_t n = visible_keys(i, b, Lk, mask_kind, key_lens);
            if (n == 0) continue;
            /* steps 1-2: scores and weights (row maximum taken out) */
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += q_row[c] * k_bh[j * rs + c];
                a[j] = scale * dot;
                if (a[j] > m) m = a[j];
            }
            double sum = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                a[j] = exp(a[j] - m);
                sum += a[j];
            }
            for (int64_t j = 0; j < n; ++j) a[j] /= sum;
            /* step 4: g_j = dout . v_j, and sum_j a_j g_j */
            double ag = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += do_row[c] * v_bh[j * rs + c];
                g[j] = dot;
                ag += a[j] * dot;
            }
            /* steps 5-6 */
            for (int64_t j = 0; j < n; ++j) {
                const double ds = a[j] * (g[j] - ag);
                for (int64_t c = 0; c < d; ++c) {
                    dq_row[c] += scale * ds * k_bh[j * rs + c];
                    dk_bh[j * rs + c] += scale * ds * q_row[c];
                    dv_bh[j * rs + c] += a[j] * do_row[c];
                }
            }
        }
    }
    free(scratch);
    return 0;
}

/* Threads the OpenMP runtime would use by default (1 without OpenMP). */
int oracle_default_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
