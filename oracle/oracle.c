/*
 * Oracle for the fused attention forward -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load or call this file.  The product path (the CUDA library and its
 * Python binding) never links, imports or executes it.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition of masked softmax attention with a
 * per-row log-sum-exp, as fixed by
 *   - "b200-flash-attention4-planner", section E step 1 (the math semantics:
 *     Q/K/V shapes and layout, head_dim, causal flag, GQA ratio, scale, the
 *     output and the LSE), and
 *   - the same page, section A1 "Streaming online softmax": the streaming
 *     method only reorganises the computation; after the last key block the
 *     result is O / row_sum, i.e. exactly softmax(scale * Q K^T + mask) V.
 * The oracle therefore does NOT stream or tile: for each query row it makes
 * one pass over all valid keys to collect the scaled scores and their
 * maximum, and a second pass to form the exponentials, their sum and the
 * weighted sum of value rows (a two-pass softmax).  Everything is fp64 with
 * libm exp/log, single-threaded, compiled without fast-math.
 *
 * Readings of points the pages leave open (each is also listed in the design
 * notes of the repository):
 *   - Layout: Q, O are [B, Hq, Sq, d]; K, V are [B, Hkv, Sk, d]; LSE is
 *     [B, Hq, Sq]; all contiguous, row-major.
 *   - GQA ("b200-flash-attention4-planner" E.7 asks for an explicit mapping):
 *     query head h reads key/value head h / (Hq / Hkv), i.e. consecutive
 *     query heads share one key/value head.
 *   - Causal alignment: bottom-right.  With L = valid key count of the batch
 *     entry, key j is visible to query row i iff j <= i + (L - Sq).  For
 *     Sq == Sk == L this is the ordinary lower-triangular mask.
 *   - Per-sequence key lengths: keys j >= L are excluded (never read).
 *     L = seqlens_k[b] clamped to [0, Sk]; a NULL seqlens_k means L = Sk.
 *   - Masked keys are excluded from the softmax, not given a large negative
 *     score.  A row with no visible key has O = 0 and LSE = -infinity.
 *   - LSE is in natural-log units of the scaled score:
 *     LSE_i = ln sum_j exp(scale * q_i . k_j)   ("b200-flash-attention4-planner"
 *     E.2 asks that the exp basis be stated; the GPU may use exp2 internally
 *     but reports this quantity).
 *   - Inputs are bf16 bit patterns (decoded exactly to double) or doubles.
 *   - Sliding window ("2026-05-28_STATUS.md", items D3 "SWA length mask" and
 *     D4 "causal mask on SWA"): with window W > 0, key j is visible to row i
 *     only if j > p_i - W, where p_i = i + (L - Sq) is the row's aligned key
 *     position; with causal this keeps the row's own key and the W - 1 keys
 *     before it.  W <= 0 means no window.
 *   - Attention sink (same page, item D5c "sink merge": one softmax over the
 *     scores and the sink): an optional per-query-head logit sigma_h in the
 *     units of the scaled score joins the softmax's normaliser but carries no
 *     value, so O_i = sum_j e^{s_j} v_j / (e^{sigma_h} + sum_j e^{s_j}) and
 *     LSE_i = ln(e^{sigma_h} + sum_j e^{s_j}); a row with no visible key then
 *     has O = 0 and LSE = sigma_h.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double oracle_bf16_bits_to_double(uint16_t bits)
{
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* Element reader: kind 0 = bf16 bit patterns, kind 1 = double. */
static double oracle_load(const void *base, int kind, int64_t index)
{
    if (kind == 0)
        return oracle_bf16_bits_to_double(((const uint16_t *)base)[index]);
    return ((const double *)base)[index];
}

/* One query row, flattened index r = (b * Hq + h) * Sq + i. */
static void oracle_one_row(const void *q, const void *k, const void *v, int kind,
                           int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq,
                           int64_t Sk, int64_t d, const int32_t *seqlens_k,
                           double scale, int causal, int64_t window,
                           const double *sinks, int64_t r,
                           double *scores, double *o_row, double *lse_out)
{
    int64_t i = r % Sq;
    int64_t h = (r / Sq) % Hq;
    int64_t b = r / (Sq * Hq);
    int64_t group = Hq / Hkv;          /* query heads per key/value head */
    int64_t hk = h / group;            /* key/value head read by query head h */
    int64_t L = Sk;                    /* valid keys of batch entry b */
    int64_t first, last, n, j, c;
    double sink = -INFINITY;           /* sink logit of head h (none: -inf) */
    const int64_t q_off = ((b * Hq + h) * Sq + i) * d;
    const int64_t kv_head_off = (b * Hkv + hk) * Sk * d;
    double m, l;

    (void)B;
    if (seqlens_k != NULL) {
        L = seqlens_k[b];
        if (L < 0) L = 0;
        if (L > Sk) L = Sk;
    }
    if (sinks != NULL)
        sink = sinks[h];
    last = L - 1;                      /* last visible key */
    if (causal && i + (L - Sq) < last)
        last = i + (L - Sq);
    first = 0;                         /* first visible key */
    if (window > 0 && i + (L - Sq) - window + 1 > first)
        first = i + (L - Sq) - window + 1;
    n = last + 1;                      /* visible keys are j = first .. n-1 */

    for (c = 0; c < d; ++c)
        o_row[c] = 0.0;
    if (n <= first) {                  /* no visible key */
        *lse_out = sink;               /* -inf without a sink */
        return;
    }

    /* pass 1: scaled scores s_j = scale * sum_c q[c] k_j[c], and their max
       (the sink logit counts as one more score) */
    m = sink;
    for (j = first; j < n; ++j) {
        double dot = 0.0;
        for (c = 0; c < d; ++c)
            dot += oracle_load(q, kind, q_off + c) *
                   oracle_load(k, kind, kv_head_off + j * d + c);
        scores[j] = scale * dot;
        if (scores[j] > m)
            m = scores[j];
    }

    /* pass 2: weights exp(s_j - m), their sum l (with the sink's weight, which
       multiplies no value row), and sum_j weight_j * v_j */
    l = (sinks != NULL) ? exp(sink - m) : 0.0;
    for (j = first; j < n; ++j) {
        double w = exp(scores[j] - m);
        l += w;
        for (c = 0; c < d; ++c)
            o_row[c] += w * oracle_load(v, kind, kv_head_off + j * d + c);
    }
    for (c = 0; c < d; ++c)
        o_row[c] /= l;
    *lse_out = m + log(l);
}

/*
 * Computes the selected query rows.  rows[t] is a flattened row index
 * (b * Hq + h) * Sq + i; if rows is NULL, all B*Hq*Sq rows are computed in
 * order.  o_out receives n_rows * d doubles, lse_out n_rows doubles.
 * Returns 0 on success, -1 on invalid arguments, -2 if scratch memory could
 * not be obtained.
 */
static int oracle_rows(const void *q, const void *k, const void *v, int kind,
                       int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq,
                       int64_t Sk, int64_t d, const int32_t *seqlens_k,
                       double scale, int causal, int64_t window,
                       const double *sinks, const int64_t *rows,
                       int64_t n_rows, double *o_out, double *lse_out)
{
    int64_t t, total;
    double *scores;

    if (!q || !k || !v || !o_out || !lse_out) return -1;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    total = B * Hq * Sq;
    if (rows == NULL) n_rows = total;
    scores = (double *)malloc((size_t)Sk * sizeof(double));
    if (!scores) return -2;
    for (t = 0; t < n_rows; ++t) {
        int64_t r = rows ? rows[t] : t;
        if (r < 0 || r >= total) { free(scores); return -1; }
        oracle_one_row(q, k, v, kind, B, Hq, Hkv, Sq, Sk, d, seqlens_k, scale,
                       causal, window, sinks, r, scores, o_out + t * d, lse_out + t);
    }
    free(scores);
    return 0;
}

/* Inputs as bf16 bit patterns (uint16). */
int oracle_attention_fwd_bf16(const uint16_t *q, const uint16_t *k,
                              const uint16_t *v, int64_t B, int64_t Hq,
                              int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d,
                              const int32_t *seqlens_k, double scale,
                              int causal, const int64_t *rows, int64_t n_rows,
                              double *o_out, double *lse_out)
{
    return oracle_rows(q, k, v, 0, B, Hq, Hkv, Sq, Sk, d, seqlens_k, scale,
                       causal, 0, NULL, rows, n_rows, o_out, lse_out);
}

/* Inputs as doubles (used by the closed-form checks of the oracle itself). */
int oracle_attention_fwd_f64(const double *q, const double *k, const double *v,
                             int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq,
                             int64_t Sk, int64_t d, const int32_t *seqlens_k,
                             double scale, int causal, const int64_t *rows,
                             int64_t n_rows, double *o_out, double *lse_out)
{
    return oracle_rows(q, k, v, 1, B, Hq, Hkv, Sq, Sk, d, seqlens_k, scale,
                       causal, 0, NULL, rows, n_rows, o_out, lse_out);
}

/* Same, with a sliding window (window <= 0: none) and per-query-head sink
   logits (sinks: Hq doubles, or NULL for none); kind 0 = bf16 bits,
   1 = doubles. */
int oracle_attention_fwd_ex(const void *q, const void *k, const void *v, int kind,
                            int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq,
                            int64_t Sk, int64_t d, const int32_t *seqlens_k,
                            double scale, int causal, int64_t window,
                            const double *sinks, const int64_t *rows,
                            int64_t n_rows, double *o_out, double *lse_out)
{
    if (kind != 0 && kind != 1) return -1;
    return oracle_rows(q, k, v, kind, B, Hq, Hkv, Sq, Sk, d, seqlens_k, scale,
                       causal, window, sinks, rows, n_rows, o_out, lse_out);
}
