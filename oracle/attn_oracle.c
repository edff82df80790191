/*
 * attn_oracle.c -- float64 CPU oracle for scaled dot-product causal
 * multi-head self-attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg load this library.  The CUDA product path
 * never calls it, links it or shares a line of code with it.
 *
 * What it computes is the plain definition, written out with no blocking,
 * fusion or reordering:
 *
 *   "Механизм внимания" (llm-arch-research.openidealab.com/textbook/attention),
 *   section "Scaled dot-product attention":
 *       Attention(Q, K, V) = softmax(Q K^T / sqrt(d_h) + M) V
 *   taken in the four steps that section lists for every query position:
 *     1. dot the query with every key,                     s_j = q . k_j
 *     2. scale,                                            s_j *= scale
 *     3. softmax over the keys, M in {0, -inf} added first
 *        (masked keys get exactly zero weight, section "Маскирование";
 *        the max-subtracted form is the numerically stable softmax of
 *        "多头注意力机制" (blog.euler0525.cn), section "Flash Attention"),
 *     4. o = sum_j p_j v_j.
 *
 * Head grouping follows section "Виды по числу голов K/V: MHA, GQA, MQA" of
 * the same textbook page: query head h reads K/V head g(h) = floor(h / (H/G)).
 *
 * The mask M:
 *   - causal (section "Маскирование"): key j is visible to the query at
 *     absolute position i iff j <= i;
 *   - sliding window (section "Скользящее окно"): that page's own rule is
 *     0 <= i - j <= W (W + 1 keys); the page also gives the narrower
 *     HuggingFace form i - j < W (W keys including the query's own).  The
 *     window_p4 flag selects the page's rule; the default is the i - j < W form.
 *   - keys past key_len[b] do not exist (a KV cache holds key_len[b] rows).
 *
 * Every score row is materialised in full (all Skv keys, masked ones
 * included) before the softmax, as the definition has it.
 *
 * The backward pass (oracle_attention_bwd) is the chain rule through those
 * same four steps, with the softmax derivative the textbook page derives in
 * section "Почему делить на корень из d_h":
 *     dp_i / dz_j = p_i (delta_ij - p_j)
 * (oracle_softmax_jacobian writes that matrix out).  The page's
 * "Эффективные реализации" section notes that FlashAttention recomputes the
 * weights block by block in the backward pass instead of storing them; this
 * oracle simply recomputes each full row.
 *
 * All arithmetic is IEEE double; exp() and log() are the C library's.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Query rows evaluated together per (b, h) work item. */
#define ORACLE_ROW_BLOCK 64

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* The mask M of the definition: 1 where the key is visible, 0 where M = -inf. */
static int key_visible(int64_t i, int64_t j, int64_t key_len, int causal,
                       int window, int window_p4)
{
    if (j < 0 || j >= key_len) return 0;
    if (causal && j > i) return 0;
    if (window > 0) {
        int64_t back = i - j;
        if (window_p4) {
            if (back > window) return 0;   /* 0 <= i - j <= W  */
        } else {
            if (back >= window) return 0;  /* i - j < W        */
        }
    }
    return 1;
}

/*
 * Numerically stable softmax of one row: p_j = exp(x_j - m) / sum_k exp(x_k - m),
 * m = max_j x_j.  Entries equal to -inf get exactly 0 (exp(-inf) = 0).
 * A row with no finite entry has no distribution; it is returned as all zeros
 * and the function returns 0 (1 otherwise).
 */
int oracle_softmax(const double* x, int64_t n, double* p)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (x[j] > m) m = x[j];
    if (m == -INFINITY) {
        for (int64_t j = 0; j < n; ++j) p[j] = 0.0;
        return 0;
    }
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        p[j] = exp(x[j] - m);
        sum += p[j];
    }
    for (int64_t j = 0; j < n; ++j) p[j] /= sum;
    return 1;
}

/*
 * The softmax derivative of section "Почему делить на корень из d_h":
 * J[i][j] = dp_i / dz_j = p_i (delta_ij - p_j), p = softmax(x), written to
 * J [n * n] row-major.  Returns what oracle_softmax returns.
 */
int oracle_softmax_jacobian(const double* x, int64_t n, double* J)
{
    double* p = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    const int ok = oracle_softmax(x, n, p);
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j)
            J[i * n + j] = p[i] * ((i == j ? 1.0 : 0.0) - p[j]);
    free(p);
    return ok;
}

/* log sum_j exp(x_j), taken as m + log sum_j exp(x_j - m) with m = max_j x_j;
 * -inf when every entry is -inf. */
double oracle_logsumexp(const double* x, int64_t n)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (x[j] > m) m = x[j];
    if (m == -INFINITY) return -INFINITY;
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) sum += exp(x[j] - m);
    return m + log(sum);
}

/*
 * q      [B, Hq,  Sq,  Dh]   queries
 * k, v   [B, Hkv, Skv, Dh]   keys / values (a KV cache when Skv > Sq)
 * key_len[b]  number of keys that exist for sequence b (<= Skv)
 * q_pos0[b]   absolute position of query row 0 of sequence b; row r sits at
 *             q_pos0[b] + r (0 for a prefill, seqlen - 1 for a decode step)
 * rows[nrows] the query rows to evaluate (the same for every (b, h));
 *             NULL with nrows == Sq means every row
 * out    [B, Hq, nrows, Dh]
 * probs  optional [B, Hq, nrows, Skv]: the softmax rows P
 * lse    optional [B, Hq, nrows]: log sum_j exp(s_j) of each evaluated row
 *        (the masked scores included as -inf)
 * Returns 0 on success, -1 on a bad argument, -2 when some evaluated row has
 * no visible key (its output is left at zero).
 */
int oracle_attention(const double* q, const double* k, const double* v,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Skv,
                     int64_t Dh, const int64_t* key_len, const int64_t* q_pos0,
                     const int64_t* rows, int64_t nrows, int causal, int window,
                     int window_p4, double scale, double* out, double* probs, double* lse)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv < 0 || Dh <= 0 || nrows < 0)
        return -1;
    if (Hq % Hkv != 0) return -1;  /* the group size H/G must be whole */
    if (!rows && nrows != Sq) return -1;
    const int64_t group = Hq / Hkv;
    const int64_t nblk = (nrows + ORACLE_ROW_BLOCK - 1) / ORACLE_ROW_BLOCK;
    const int64_t items = B * Hq * nblk;
    int status = 0;

#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1) * ORACLE_ROW_BLOCK);
        double* prow = (double*)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t it = 0; it < items; ++it) {
            const int64_t blk = it % nblk;
            const int64_t h = (it / nblk) % Hq;
            const int64_t b = it / (nblk * Hq);
            const int64_t g = h / group;                 /* g(h) = floor(h / (H/G)) */
            const double* kb = k + (b * Hkv + g) * Skv * Dh;
            const double* vb = v + (b * Hkv + g) * Skv * Dh;
            const int64_t r0 = blk * ORACLE_ROW_BLOCK;
            const int64_t r1 = r0 + ORACLE_ROW_BLOCK < nrows ? r0 + ORACLE_ROW_BLOCK : nrows;

            /* steps 1-2 and the mask: the full score rows of this block */
            for (int64_t r = r0; r < r1; ++r) {
                const int64_t row = rows ? rows[r] : r;
                const double* qi = q + ((b * Hq + h) * Sq + row) * Dh;
                const int64_t i = q_pos0[b] + row;
                double* s = srow + (r - r0) * Skv;
                for (int64_t j = 0; j < Skv; ++j) {
                    double dot = 0.0;
                    const double* kj = kb + j * Dh;
                    for (int64_t d = 0; d < Dh; ++d) dot += qi[d] * kj[d];
                    s[j] = dot * scale;
                    if (!key_visible(i, j, key_len[b], causal, window, window_p4))
                        s[j] = -INFINITY;
                }
            }
            /* steps 3-4 */
            for (int64_t r = r0; r < r1; ++r) {
                double* o = out + ((b * Hq + h) * nrows + r) * Dh;
                for (int64_t d = 0; d < Dh; ++d) o[d] = 0.0;
                if (!oracle_softmax(srow + (r - r0) * Skv, Skv, prow)) {
#pragma omp atomic write
                    status = -2;
                }
                if (probs) memcpy(probs + ((b * Hq + h) * nrows + r) * Skv, prow, sizeof(double) * (size_t)Skv);
                if (lse) lse[(b * Hq + h) * nrows + r] = oracle_logsumexp(srow + (r - r0) * Skv, Skv);
                for (int64_t j = 0; j < Skv; ++j) {
                    const double pj = prow[j];
                    const double* vj = vb + j * Dh;
                    for (int64_t d = 0; d < Dh; ++d) o[d] += pj * vj[d];
                }
            }
        }
        free(srow);
        free(prow);
    }
    return status;
}

/*
 * Backward pass of o = softmax(scale * q K^T + M) V for a full sequence
 * (Sq = Skv = S, query row i at position i), given the upstream gradient
 * dout = dL/do.  For every (b, h) and query row i, with g = g(h):
 *
 *   s_j   = scale * q_i . k_j, or -inf where masked     (forward step 1-3)
 *   p     = softmax(s)
 *   dv_j += p_j * dout_i                                 (o_i = sum_j p_j v_j)
 *   dp_j  = dout_i . v_j                                 (dL/dp_j)
 *   ds_j  = sum_k dp_k * (dp_k/ds_j) = sum_k dp_k p_k (delta_kj - p_j)
 *         = p_j * (dp_j - sum_k p_k dp_k)                (the page's Jacobian, contracted)
 *   dq_i  = scale * sum_j ds_j k_j
 *   dk_j += scale * ds_j * q_i
 *
 * dk and dv of K/V head g sum over every query head of its group and every
 * query row.  rows[nrows] selects the dq rows to return (NULL with
 * nrows == S: all; nrows == 0: none); keys[nkeys] the dk/dv rows (NULL with
 * nkeys == S: all; nkeys == 0: none, and then only the selected query rows
 * are evaluated).
 *
 * dq [B, Hq, nrows, Dh]; dk, dv [B, Hkv, nkeys, Dh].  Returns 0, -1 on a bad
 * argument, -2 when an evaluated row has no visible key.
 */
int oracle_attention_bwd(const double* q, const double* k, const double* v, const double* dout,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t S, int64_t Dh,
                         int causal, int window, int window_p4, double scale,
                         const int64_t* rows, int64_t nrows, const int64_t* keys, int64_t nkeys,
                         double* dq, double* dk, double* dv)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || S < 0 || Dh <= 0 || nrows < 0 || nkeys < 0) return -1;
    if (Hq % Hkv != 0) return -1;
    if ((!rows && nrows != S && nrows != 0) || (!keys && nkeys != S && nkeys != 0)) return -1;
    const int64_t group = Hq / Hkv;
    int status = 0;
    /* where each query row / key lands in dq / dk, dv (-1: not asked for) */
    int64_t* row_at = (int64_t*)malloc(sizeof(int64_t) * (size_t)(S > 0 ? S : 1));
    int64_t* key_at = (int64_t*)malloc(sizeof(int64_t) * (size_t)(S > 0 ? S : 1));
    for (int64_t i = 0; i < S; ++i) row_at[i] = key_at[i] = -1;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= S) { free(row_at); free(key_at); return -1; }
        row_at[i] = r;
    }
    for (int64_t m = 0; m < nkeys; ++m) {
        const int64_t j = keys ? keys[m] : m;
        if (j < 0 || j >= S) { free(row_at); free(key_at); return -1; }
        key_at[j] = m;
    }
    memset(dq, 0, sizeof(double) * (size_t)(B * Hq * nrows * Dh));
    memset(dk, 0, sizeof(double) * (size_t)(B * Hkv * nkeys * Dh));
    memset(dv, 0, sizeof(double) * (size_t)(B * Hkv * nkeys * Dh));

    /* one work item per (b, g): it owns dk, dv of that K/V head and dq of
       the query heads of its group, so no two threads write one value */
#pragma omp parallel
    {
        const size_t n = (size_t)(S > 0 ? S : 1);
        double* s = (double*)malloc(sizeof(double) * n);
        double* p = (double*)malloc(sizeof(double) * n);
        double* dp = (double*)malloc(sizeof(double) * n);
#pragma omp for schedule(dynamic, 1)
        for (int64_t it = 0; it < B * Hkv; ++it) {
            const int64_t b = it / Hkv, g = it % Hkv;
            const double* kb = k + (b * Hkv + g) * S * Dh;
            const double* vb = v + (b * Hkv + g) * S * Dh;
            double* dkb = dk + (b * Hkv + g) * nkeys * Dh;
            double* dvb = dv + (b * Hkv + g) * nkeys * Dh;
            for (int64_t h = g * group; h < (g + 1) * group; ++h) {
                for (int64_t i = 0; i < S; ++i) {
                    if (nkeys == 0 && row_at[i] < 0) continue;
                    const double* qi = q + ((b * Hq + h) * S + i) * Dh;
                    const double* doi = dout + ((b * Hq + h) * S + i) * Dh;
                    for (int64_t j = 0; j < S; ++j) {
                        double dot = 0.0;
                        for (int64_t d = 0; d < Dh; ++d) dot += qi[d] * kb[j * Dh + d];
                        s[j] = key_visible(i, j, S, causal, window, window_p4) ? dot * scale
                                                                                : -INFINITY;
                    }
                    if (!oracle_softmax(s, S, p)) {
#pragma omp atomic write
                        status = -2;
                    }
                    double pdp = 0.0;   /* sum_k p_k dp_k */
                    for (int64_t j = 0; j < S; ++j) {
                        double dot = 0.0;
                        for (int64_t d = 0; d < Dh; ++d) dot += doi[d] * vb[j * Dh + d];
                        dp[j] = dot;
                        pdp += p[j] * dot;
                    }
                    double* dqi = row_at[i] >= 0 ? dq + ((b * Hq + h) * nrows + row_at[i]) * Dh : NULL;
                    for (int64_t j = 0; j < S; ++j) {
                        const double ds = p[j] * (dp[j] - pdp);
                        if (dqi)
                            for (int64_t d = 0; d < Dh; ++d) dqi[d] += scale * ds * kb[j * Dh + d];
                        const int64_t m = key_at[j];
                        if (m >= 0) {
                            for (int64_t d = 0; d < Dh; ++d) {
                                dvb[m * Dh + d] += p[j] * doi[d];
                                dkb[m * Dh + d] += scale * ds * qi[d];
                            }
                        }
                    }
                }
            }
        }
        free(s);
        free(p);
        free(dp);
    }
    free(row_at);
    free(key_at);
    return status;
}
