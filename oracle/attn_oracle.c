/*
 * attn_oracle.c -- plain fp64 CPU oracle for the attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library; the attention library never does,
 * and nothing here is shared with it.
 *
 * What it computes is the plain definition of the operation the pages describe
 * (Flash-Attention: Context (CTE), "Abstract": O = softmax(scale * Q K^T) V for one
 * (batch*head) problem), with the masks of the same pages.  For each query row it
 * materialises the whole score row, takes the softmax over the allowed keys, and
 * multiplies by V.  The online-softmax recurrence of the pages is an identity
 * transformation of this result (minfer "03 - 8n FA-style tiled prefill attention",
 * section 2.1 "Online softmax"), so the oracle is the definition, not the recurrence.
 * Inputs are bf16 bit patterns widened exactly to double; all arithmetic is double.
 *
 * Parity status: every function here is pinned by tests/test_oracle_pins.py
 * (closed forms, invariants, hand-worked golden cases, an independent library
 * routine and brute force on tiny inputs).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_PAGE 2
#define ORACLE_ERR_NOMEM 3

/* bf16 -> double: a bf16 value is the top half of an IEEE float32. */
double oracle_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static void widen(const uint16_t *src, long n, double *dst)
{
    for (long i = 0; i < n; ++i) dst[i] = oracle_bf16_to_f64(src[i]);
}

/* GQA head map.  Heads are grouped: query head h reads kv head h / (hq / hkv)
 * (Flash-Attention: Context (CTE), "GQA and multi-head"; minfer 8n, section 3.1,
 * "GQA slicing").  Requires hq % hkv == 0. */
int oracle_kv_head(int h, int hq, int hkv)
{
    return h / (hq / hkv);
}

/* Position of query row i when sq queries sit at the tail of skv keys.  The pages
 * place new queries after the cached keys (Flash-Attention: Decode (TKG), "New-token
 * K/V append"; minfer 8n, "kv_end = positions[last_t] + 1"); with sq == skv this is
 * the CTE kernel's q_pos = grp*128 + p. */
long oracle_q_pos(long i, long sq, long skv)
{
    return i + (skv - sq);
}

/* The mask predicate for key j of a query at q_pos.
 *   validity: j < skv (padding / cache-length cut, TKG "gen_mask_tkg" type A)
 *   causal:   q_pos >= k_pos                    (CTE "The diagonal affine_select mask")
 *   window:   k_pos >= q_pos - window + 1       (optimum-neuron "Sliding window",
 *             chained after the causal predicate); window == 0 means no window. */
int oracle_allowed(long j, long skv, long q_pos, int causal, long window)
{
    if (j < 0 || j >= skv) return 0;
    if (causal && j > q_pos) return 0;
    if (window > 0 && j < q_pos - window + 1) return 0;
    return 1;
}

/* Scores of one query row: s_j = scale * sum_x q[x] * k[j][x]  (CTE "Scale": the scale
 * multiplies Q K^T). q: [d] double, k: [skv][d] double. */
void oracle_scores(const double *q, const double *k, long skv, int d, double scale, double *s)
{
    for (long j = 0; j < skv; ++j) {
        double acc = 0.0;
        for (int x = 0; x < d; ++x) acc += q[x] * k[j * (long)d + x];
        s[j] = scale * acc;
    }
}

/* Softmax over the allowed entries of one score row, with an optional attention sink.
 * The sink is one extra logit of the row that joins the maximum and the sum but has no
 * value row (Flash-Attention: Context (CTE), "Algorithm - the per-section max update":
 * the sink logit is appended as one more column of the max; "Algorithm - fused exp and
 * the running sum": exp(sink - max) is appended to the row sum).  sink = -inf means no
 * sink.
 *   M = max(max over allowed s_j, sink);  l = sum_allowed exp(s_j - M) + exp(sink - M);
 *   P_j = exp(s_j - M) / l, P_j = 0 where not allowed;  LSE = M + ln l.
 * A row with nothing allowed and no sink has P = 0 and LSE = -inf (minfer 8n, "rows
 * with l == 0 stay 0"); with a sink it has P = 0 and LSE = sink.  Returns LSE. */
double oracle_softmax_sink(const double *s, const unsigned char *allowed, long n, double sink,
                           double *p)
{
    double m = sink;
    for (long j = 0; j < n; ++j)
        if (allowed[j] && s[j] > m) m = s[j];
    if (m == -INFINITY) {
        for (long j = 0; j < n; ++j) p[j] = 0.0;
        return -INFINITY;
    }
    double l = exp(sink - m); /* exactly 0 without a sink */
    for (long j = 0; j < n; ++j) {
        p[j] = allowed[j] ? exp(s[j] - m) : 0.0;
        l += p[j];
    }
    for (long j = 0; j < n; ++j) p[j] = p[j] / l;
    return m + log(l);
}

/* The softmax without a sink (see oracle_softmax_sink). */
double oracle_softmax(const double *s, const unsigned char *allowed, long n, double *p)
{
    return oracle_softmax_sink(s, allowed, n, -INFINITY, p);
}

/* O = sum_j P_j * V_j.  v: [n][d] double. */
void oracle_pv(const double *p, const double *v, long n, int d, double *o)
{
    for (int x = 0; x < d; ++x) o[x] = 0.0;
    for (long j = 0; j < n; ++j) {
        if (p[j] == 0.0) continue; /* a zero weight adds nothing (and skips NaN padding) */
        for (int x = 0; x < d; ++x) o[x] += p[j] * v[j * (long)d + x];
    }
}

/* One query row end to end, on already widened K and V of its kv head. */
static int row_f64(const double *q, const double *k, const double *v, long skv, int d,
                   double scale, long q_pos, int causal, long window, double sink, double *o,
                   double *lse, double *p_out)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(skv > 0 ? skv : 1));
    double *p = p_out ? p_out : (double *)malloc(sizeof(double) * (size_t)(skv > 0 ? skv : 1));
    unsigned char *al = (unsigned char *)malloc((size_t)(skv > 0 ? skv : 1));
    if (!s || !p || !al) {
        free(s); free(al); if (!p_out) free(p);
        return ORACLE_ERR_NOMEM;
    }
    oracle_scores(q, k, skv, d, scale, s);
    for (long j = 0; j < skv; ++j) al[j] = (unsigned char)oracle_allowed(j, skv, q_pos, causal, window);
    *lse = oracle_softmax_sink(s, al, skv, sink, p);
    oracle_pv(p, v, skv, d, o);
    free(s); free(al);
    if (!p_out) free(p);
    return ORACLE_OK;
}

/* Rows of one head, given as bf16 bits: q_rows [n][d], k and v [skv][d], q_pos [n],
 * with the head's sink logit (-inf for none).  Writes o [n][d] and lse [n]; p_out
 * (nullable) receives [n][skv] probabilities. */
int oracle_attention_rows_sink(const uint16_t *q_rows, long n, const uint16_t *k,
                               const uint16_t *v, long skv, int d, double scale,
                               const long *q_pos, int causal, long window, double sink,
                               double *o, double *lse, double *p_out)
{
    if (n < 0 || skv < 0 || d <= 0) return ORACLE_ERR_ARG;
    double *kd = (double *)malloc(sizeof(double) * (size_t)(skv * d + 1));
    double *vd = (double *)malloc(sizeof(double) * (size_t)(skv * d + 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);
    if (!kd || !vd || !qd) { free(kd); free(vd); free(qd); return ORACLE_ERR_NOMEM; }
    widen(k, skv * d, kd);
    widen(v, skv * d, vd);
    int rc = ORACLE_OK;
    for (long r = 0; r < n && rc == ORACLE_OK; ++r) {
        widen(q_rows + r * d, d, qd);
        rc = row_f64(qd, kd, vd, skv, d, scale, q_pos[r], causal, window, sink, o + r * d,
                     lse + r, p_out ? p_out + r * skv : NULL);
    }
    free(kd); free(vd); free(qd);
    return rc;
}

/* oracle_attention_rows_sink without a sink. */
int oracle_attention_rows(const uint16_t *q_rows, long n, const uint16_t *k, const uint16_t *v,
                          long skv, int d, double scale, const long *q_pos, int causal,
                          long window, double *o, double *lse, double *p_out)
{
    return oracle_attention_rows_sink(q_rows, n, k, v, skv, d, scale, q_pos, causal, window,
                                      -INFINITY, o, lse, p_out);
}

/* Prefill over flattened heads [bh_begin, bh_end) of q [B][HQ][SQ][D] against
 * k, v [B][HKV][SKV][D]; o [B][HQ][SQ][D], lse [B][HQ][SQ].  sink: [HQ] logits, one per
 * query head (shared by every batch; CTE and TKG keep the sink per query head), or NULL
 * for none. */
int oracle_prefill_sink(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int HQ,
                        int HKV, long SQ, long SKV, int D, double scale, int causal, long window,
                        const double *sink, long bh_begin, long bh_end, double *o, double *lse)
{
    if (HKV <= 0 || HQ % HKV != 0) return ORACLE_ERR_ARG;
    long *qp = (long *)malloc(sizeof(long) * (size_t)(SQ > 0 ? SQ : 1));
    if (!qp) return ORACLE_ERR_NOMEM;
    for (long i = 0; i < SQ; ++i) qp[i] = oracle_q_pos(i, SQ, SKV);
    int rc = ORACLE_OK;
    for (long bh = bh_begin; bh < bh_end && rc == ORACLE_OK; ++bh) {
        long b = bh / HQ;
        int h = (int)(bh % HQ);
        int g = oracle_kv_head(h, HQ, HKV);
        const uint16_t *qh = q + (size_t)bh * SQ * D;
        const uint16_t *kh = k + ((size_t)b * HKV + g) * SKV * D;
        const uint16_t *vh = v + ((size_t)b * HKV + g) * SKV * D;
        rc = oracle_attention_rows_sink(qh, SQ, kh, vh, SKV, D, scale, qp, causal, window,
                                        sink ? sink[h] : -INFINITY, o + (size_t)bh * SQ * D,
                                        lse + (size_t)bh * SQ, NULL);
    }
    free(qp);
    return rc;
}

/* oracle_prefill_sink without a sink. */
int oracle_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int HQ, int HKV,
                   long SQ, long SKV, int D, double scale, int causal, long window,
                   long bh_begin, long bh_end, double *o, double *lse)
{
    return oracle_prefill_sink(q, k, v, B, HQ, HKV, SQ, SKV, D, scale, causal, window, NULL,
                               bh_begin, bh_end, o, lse);
}

/* Packed (variable-length) prefill: nseq sequences packed along the sequence axis of one
 * batch, sequence s holding query rows [cu_q[s], cu_q[s+1]) and key rows [cu_k[s],
 * cu_k[s+1]).  Each sequence is its own attention problem: its queries sit at the tail of
 * its keys (a key count above the query count is a cached prefix), with the causal and
 * window masks taken inside the sequence and no key of another sequence allowed
 * (Flash-Attention: Context (CTE), "Algorithm - the dynamic range_select family": per-row
 * key bounds for sequence packing and dynamic prefix length).  q [HQ][SQ][D] and k, v
 * [HKV][SKV][D] with SQ = cu_q[nseq], SKV = cu_k[nseq]; o [HQ][SQ][D], lse [HQ][SQ]; heads
 * [h_begin, h_end); sink as oracle_prefill_sink. */
int oracle_prefill_varlen(const uint16_t *q, const uint16_t *k, const uint16_t *v, int HQ, int HKV,
                          int D, const int32_t *cu_q, const int32_t *cu_k, int nseq, double scale,
                          int causal, long window, const double *sink, long h_begin, long h_end,
                          double *o, double *lse)
{
    if (HKV <= 0 || HQ % HKV != 0 || nseq < 0) return ORACLE_ERR_ARG;
    for (int s = 0; s < nseq; ++s)
        if (cu_q[s + 1] < cu_q[s] || cu_k[s + 1] < cu_k[s]) return ORACLE_ERR_ARG;
    const long SQ = cu_q[nseq], SKV = cu_k[nseq];
    int rc = ORACLE_OK;
    for (long h = h_begin; h < h_end && rc == ORACLE_OK; ++h) {
        int g = oracle_kv_head((int)h, HQ, HKV);
        for (int s = 0; s < nseq && rc == ORACLE_OK; ++s) {
            const long q0 = cu_q[s], nq = cu_q[s + 1] - q0, k0 = cu_k[s], nk = cu_k[s + 1] - k0;
            if (nq == 0) continue;
            long *qp = (long *)malloc(sizeof(long) * (size_t)nq);
            if (!qp) return ORACLE_ERR_NOMEM;
            for (long i = 0; i < nq; ++i) qp[i] = oracle_q_pos(i, nq, nk);
            rc = oracle_attention_rows_sink(q + ((size_t)h * SQ + q0) * D, nq,
                                            k + ((size_t)g * SKV + k0) * D,
                                            v + ((size_t)g * SKV + k0) * D, nk, D, scale, qp,
                                            causal, window, sink ? sink[h] : -INFINITY,
                                            o + ((size_t)h * SQ + q0) * D, lse + (size_t)h * SQ + q0,
                                            NULL);
            free(qp);
        }
    }
    return rc;
}

/* Paged gather: logical token j of a sequence lives in physical page table_row[j / page],
 * slot j % page; the cache is [num_pages][hkv][page][d] (Flash-Attention: Decode (TKG),
 * "Paged / block cache": the reference gather is block_cache[active_blocks_table[b]]).
 * An entry >= num_pages is an error, never dereferenced. */
int oracle_gather_paged(const uint16_t *cache, const uint32_t *table_row, long num_pages, int hkv,
                        int g, int page, int d, long len, uint16_t *out)
{
    for (long j = 0; j < len; ++j) {
        uint32_t pg = table_row[j / page];
        if ((long)pg >= num_pages) return ORACLE_ERR_PAGE;
        const uint16_t *src = cache + (((size_t)pg * hkv + g) * page + (size_t)(j % page)) * d;
        memcpy(out + (size_t)j * d, src, sizeof(uint16_t) * (size_t)d);
    }
    return ORACLE_OK;
}

/* Decode over flattened (b, h) in [bh_begin, bh_end).  Query t of the s_active new tokens
 * sits at q_pos = cache_len - s_active + t and attends keys j <= q_pos of the cache (whose
 * last s_active slots hold the new tokens' K/V); the softmax runs over the cache axis
 * (TKG "The single-query decode attention").
 * q [B][HQ][s_active][D]; paged cache [num_pages][HKV][page][D] when table != NULL
 * (table [B][max_pages]), else flat cache [B][HKV][max_cache_len][D];
 * o [B][HQ][s_active][D], lse [B][HQ][s_active].  sink: [HQ] logits or NULL, as for
 * oracle_prefill_sink (TKG "GQA / MQA grouped-query broadcast": the sink is per query
 * head, broadcast over the batch). */
int oracle_decode_sink(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                       const uint32_t *table, const int32_t *cache_len, int B, int HQ, int HKV,
                       int D, int s_active, int page, long max_pages, long num_pages,
                       long max_cache_len, double scale, const double *sink, long bh_begin,
                       long bh_end, double *o, double *lse)
{
    if (HKV <= 0 || HQ % HKV != 0 || s_active <= 0) return ORACLE_ERR_ARG;
    int rc = ORACLE_OK;
    for (long bh = bh_begin; bh < bh_end && rc == ORACLE_OK; ++bh) {
        long b = bh / HQ;
        int h = (int)(bh % HQ);
        int g = oracle_kv_head(h, HQ, HKV);
        long len = cache_len[b];
        if (len < s_active || (!table && len > max_cache_len) ||
            (table && (len + page - 1) / page > max_pages))
            return ORACLE_ERR_ARG;
        uint16_t *kf = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(len * D + 1));
        uint16_t *vf = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(len * D + 1));
        long *qp = (long *)malloc(sizeof(long) * (size_t)s_active);
        if (!kf || !vf || !qp) { free(kf); free(vf); free(qp); return ORACLE_ERR_NOMEM; }
        if (table) {
            rc = oracle_gather_paged(k_cache, table + (size_t)b * max_pages, num_pages, HKV, g,
                                     page, D, len, kf);
            if (rc == ORACLE_OK)
                rc = oracle_gather_paged(v_cache, table + (size_t)b * max_pages, num_pages, HKV,
                                         g, page, D, len, vf);
        } else {
            const size_t base = ((size_t)b * HKV + g) * (size_t)max_cache_len * D;
            memcpy(kf, k_cache + base, sizeof(uint16_t) * (size_t)(len * D));
            memcpy(vf, v_cache + base, sizeof(uint16_t) * (size_t)(len * D));
        }
        for (int t = 0; t < s_active; ++t) qp[t] = len - s_active + t;
        if (rc == ORACLE_OK)
            rc = oracle_attention_rows_sink(q + (size_t)bh * s_active * D, s_active, kf, vf, len,
                                            D, scale, qp, 1, 0, sink ? sink[h] : -INFINITY,
                                            o + (size_t)bh * s_active * D,
                                            lse + (size_t)bh * s_active, NULL);
        free(kf); free(vf); free(qp);
    }
    return rc;
}

/* oracle_decode_sink without a sink. */
int oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  const uint32_t *table, const int32_t *cache_len, int B, int HQ, int HKV, int D,
                  int s_active, int page, long max_pages, long num_pages, long max_cache_len,
                  double scale, long bh_begin, long bh_end, double *o, double *lse)
{
    return oracle_decode_sink(q, k_cache, v_cache, table, cache_len, B, HQ, HKV, D, s_active,
                              page, max_pages, num_pages, max_cache_len, scale, NULL, bh_begin,
                              bh_end, o, lse);
}

/* e4m3 -> double, from the format's definition (the 8-bit float with 1 sign, 4 exponent
 * and 3 mantissa bits, exponent bias 7, no infinities, and NaN only at S.1111.111; the
 * FP8-e4m3 KV cache of Flash-Attention: Decode (TKG), "Decode (TKG) vs context (CTE) -
 * the diff").  Exponent field 0 holds the subnormals m/8 * 2^-6. */
double oracle_e4m3_to_f64(uint8_t b)
{
    const int sgn = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* Decode over an e4m3 KV cache: each cache byte stands for e4m3(byte) * k_scale (K) or
 * e4m3(byte) * v_scale (V); otherwise exactly oracle_decode_sink, whose layouts it shares
 * with one byte per cache element.  The dequantised K and V of a sequence are built in
 * double and run through the same row computation. */
int oracle_decode_e4m3(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                       const uint32_t *table, const int32_t *cache_len, int B, int HQ, int HKV,
                       int D, int s_active, int page, long max_pages, long num_pages,
                       long max_cache_len, double scale, double k_scale, double v_scale,
                       const double *sink, long bh_begin, long bh_end, double *o, double *lse)
{
    if (HKV <= 0 || HQ % HKV != 0 || s_active <= 0) return ORACLE_ERR_ARG;
    int rc = ORACLE_OK;
    for (long bh = bh_begin; bh < bh_end && rc == ORACLE_OK; ++bh) {
        long b = bh / HQ;
        int h = (int)(bh % HQ);
        int g = oracle_kv_head(h, HQ, HKV);
        long len = cache_len[b];
        if (len < s_active || (!table && len > max_cache_len) ||
            (table && (len + page - 1) / page > max_pages))
            return ORACLE_ERR_ARG;
        double *kd = (double *)malloc(sizeof(double) * (size_t)(len * D + 1));
        double *vd = (double *)malloc(sizeof(double) * (size_t)(len * D + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        if (!kd || !vd || !qd) { free(kd); free(vd); free(qd); return ORACLE_ERR_NOMEM; }
        for (long j = 0; j < len && rc == ORACLE_OK; ++j) {
            size_t row;
            if (table) {
                uint32_t pg = table[(size_t)b * max_pages + j / page];
                if ((long)pg >= num_pages) { rc = ORACLE_ERR_PAGE; break; }
                row = ((size_t)pg * HKV + g) * page + (size_t)(j % page);
            } else {
                row = ((size_t)b * HKV + g) * (size_t)max_cache_len + (size_t)j;
            }
            for (int x = 0; x < D; ++x) {
                kd[j * D + x] = oracle_e4m3_to_f64(k_cache[row * D + x]) * k_scale;
                vd[j * D + x] = oracle_e4m3_to_f64(v_cache[row * D + x]) * v_scale;
            }
        }
        for (int t = 0; t < s_active && rc == ORACLE_OK; ++t) {
            const size_t r = (size_t)bh * s_active + t;
            widen(q + r * D, D, qd);
            rc = row_f64(qd, kd, vd, len, D, scale, len - s_active + t, 1, 0,
                         sink ? sink[h] : -INFINITY, o + r * D, lse + r, NULL);
        }
        free(kd); free(vd); free(qd);
    }
    return rc;
}

/* Rotary position embedding of one row x [d] at position pos, half-split form: for
 * i < d/2, with theta = pos * inv_freq[i],
 *   x'[i]       = x[i] cos theta - x[i + d/2] sin theta
 *   x'[i + d/2] = x[i + d/2] cos theta + x[i] sin theta
 * (Flash-Attention: Decode (TKG), "Algorithm", step 0: RoPE of Q from inverse
 * frequencies and position ids, fused ahead of the Q.K^T product). */
void oracle_rope_row(double *x, int d, double pos, const double *inv_freq)
{
    const int h = d / 2;
    for (int i = 0; i < h; ++i) {
        const double th = pos * inv_freq[i];
        const double c = cos(th), sn = sin(th);
        const double a = x[i], b = x[i + h];
        x[i] = a * c - b * sn;
        x[i + h] = b * c + a * sn;
    }
}

/* Round to the nearest bf16, ties to even (by way of binary32, whose rounding is the
 * C conversion's round-to-nearest).  The rotated rows are bf16 operands of the product. */
static double round_bf16(double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) return (double)f; /* inf or NaN */
    u += 0x7fffu + ((u >> 16) & 1u);
    u &= 0xffff0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Decode with the options of the pages' decode kernel, on a bf16 cache:
 *   window > 0: new token t (q_pos = len - s_active + t) attends j iff
 *     q_pos - window + 1 <= j <= q_pos (the prefill window band, AGENTS "Sliding
 *     window"; TKG "gen_mask_tkg" type B is this band at the end of the cache);
 *   circular (flat cache only, window > 0): logical position j lives at row
 *     j mod max_cache_len, so cache_len may exceed max_cache_len (type B's wrapped
 *     case); positions before the window are never read;
 *   k_new, v_new ([B][HKV][s_active][D] bf16, or NULL): the new tokens' K and V,
 *     which stand at positions len - s_active .. len - 1 instead of the cache's rows
 *     (TKG "New-token K/V append": the product sees [cached prior | active]);
 *   inv_freq ([D/2], or NULL): RoPE of each query row at its q_pos and of each k_new
 *     row at its position (TKG "Algorithm", step 0; "GQA / MQA grouped-query broadcast":
 *     one rotation for the shared K head), each rotated row rounded to bf16: the rows
 *     are the bf16 operands of the product, and the rotated K is what the cache stores
 *     ("New-token K/V append": the persistent store of the RoPE'd K);
 *   sink ([HQ] or NULL): as oracle_decode_sink.
 * Other arguments and layouts as oracle_decode_sink. */
int oracle_decode_ext(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                      const uint16_t *k_new, const uint16_t *v_new, const uint32_t *table,
                      const int32_t *cache_len, int B, int HQ, int HKV, int D, int s_active,
                      int page, long max_pages, long num_pages, long max_cache_len, double scale,
                      long window, int circular, const double *inv_freq, const double *sink,
                      long bh_begin, long bh_end, double *o, double *lse)
{
    if (HKV <= 0 || HQ % HKV != 0 || s_active <= 0 || window < 0) return ORACLE_ERR_ARG;
    if (circular && (table || window == 0 || window + s_active - 1 > max_cache_len))
        return ORACLE_ERR_ARG;
    int rc = ORACLE_OK;
    for (long bh = bh_begin; bh < bh_end && rc == ORACLE_OK; ++bh) {
        long b = bh / HQ;
        int h = (int)(bh % HQ);
        int g = oracle_kv_head(h, HQ, HKV);
        long len = cache_len[b];
        if (len < s_active || (!table && !circular && len > max_cache_len) ||
            (table && (len + page - 1) / page > max_pages))
            return ORACLE_ERR_ARG;
        /* the oldest position any new token may attend */
        const long lo = window > 0 ? (len - s_active) - window + 1 : 0;
        double *kd = (double *)malloc(sizeof(double) * (size_t)(len * D + 1));
        double *vd = (double *)malloc(sizeof(double) * (size_t)(len * D + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        if (!kd || !vd || !qd) { free(kd); free(vd); free(qd); return ORACLE_ERR_NOMEM; }
        for (long j = 0; j < len && rc == ORACLE_OK; ++j) {
            const long t = j - (len - s_active); /* >= 0: a new token */
            if (k_new && t >= 0) {
                const size_t r = (((size_t)b * HKV + g) * s_active + (size_t)t) * D;
                widen(k_new + r, D, kd + j * D);
                widen(v_new + r, D, vd + j * D);
                if (inv_freq) {
                    oracle_rope_row(kd + j * D, D, (double)j, inv_freq);
                    for (int x = 0; x < D; ++x) kd[j * D + x] = round_bf16(kd[j * D + x]);
                }
                continue;
            }
            if (j < lo) { /* outside every window: never attended, never read */
                for (int x = 0; x < D; ++x) kd[j * D + x] = vd[j * D + x] = NAN;
                continue;
            }
            size_t row;
            if (table) {
                uint32_t pg = table[(size_t)b * max_pages + j / page];
                if ((long)pg >= num_pages) { rc = ORACLE_ERR_PAGE; break; }
                row = ((size_t)pg * HKV + g) * page + (size_t)(j % page);
            } else {
                row = ((size_t)b * HKV + g) * (size_t)max_cache_len +
                      (size_t)(circular ? j % max_cache_len : j);
            }
            widen(k_cache + row * D, D, kd + j * D);
            widen(v_cache + row * D, D, vd + j * D);
        }
        for (int t = 0; t < s_active && rc == ORACLE_OK; ++t) {
            const size_t r = (size_t)bh * s_active + t;
            const long qp = len - s_active + t;
            widen(q + r * D, D, qd);
            if (inv_freq) {
                oracle_rope_row(qd, D, (double)qp, inv_freq);
                for (int x = 0; x < D; ++x) qd[x] = round_bf16(qd[x]);
            }
            rc = row_f64(qd, kd, vd, len, D, scale, qp, 1, window, sink ? sink[h] : -INFINITY,
                         o + r * D, lse + r, NULL);
        }
        free(kd); free(vd); free(qd);
    }
    return rc;
}

/* The decode 0/1 mask, [B][HQ][s_active][max_len] bytes (TKG "gen_mask_tkg"):
 *   type A: position j is attendable iff j < cache_len[b] (cache_len = next write position);
 *   type C: the last s_active slots are the new tokens, and among them query t sees
 *           slot u iff u <= t (the lower-triangular tril(ones(s_active)) block).
 * Returns an error if some cache_len < s_active or > max_len. */
int oracle_decode_mask(const int32_t *cache_len, int B, int HQ, int s_active, long max_len,
                       uint8_t *mask)
{
    for (int b = 0; b < B; ++b) {
        long len = cache_len[b];
        if (len < s_active || len > max_len) return ORACLE_ERR_ARG;
        for (int h = 0; h < HQ; ++h)
            for (int t = 0; t < s_active; ++t) {
                uint8_t *row = mask + (((size_t)b * HQ + h) * s_active + t) * (size_t)max_len;
                for (long j = 0; j < max_len; ++j) row[j] = (uint8_t)(j < len); /* type A */
                long first_new = len - s_active;
                for (int u = 0; u < s_active; ++u)                              /* type C */
                    row[first_new + u] = (uint8_t)(u <= t);
            }
    }
    return ORACLE_OK;
}
