/*
 * attn_oracle.c -- double-precision CPU oracle for single-query grouped-query
 * decode attention over an f16 KV cache.
 *
 * TEST INFRASTRUCTURE. This file is the correctness reference the CUDA path is
 * checked against. Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it; the product path never calls it. It shares no code,
 * header, constant or helper with the CUDA library, and it includes nothing
 * but the C standard library (plus OpenMP for the optional outer loop).
 *
 * What it computes is the plain definition of the operation. The minfer page
 * "10 · R4 -- decode split-attention dim-parallel rewrite" (§2.1) states it as
 * o = softmax(q·Kᵀ·scale)·V and says the split-KV two-stage scheme is
 * mathematically the same as one softmax over the whole context, so the
 * single-pass definition is the oracle:
 *
 *   for every sequence s and query head h:
 *     G    = n_head / n_kv_head,  hk = h / G       (contiguous query-head groups)
 *     n    = clamp(positions[s] + 1, 0, cap)        (§2.2: nkv = positions + 1)
 *     x_j  = scale * sum_d q[s][h][d] * K[s][j][hk][d]           for j < n
 *     w_j  = exp(x_j - max_i x_i)
 *     o[d] = (sum_j w_j * V[s][j][hk][d]) / (sum_j w_j)
 *     o    = 0 when n == 0  (the combine's "S > 0 ? acc/S : 0" rule, §3.2)
 *
 * Everything is evaluated in double: q (f32) and the cache entries (binary16,
 * or bfloat16 through the _kv entry points) convert exactly, each product q*k
 * is exact, exp is libm's double exp.
 *
 * A second entry point restates the two-stage method of §2.1/§2.2 literally
 * (per-split online softmax, then the max-reweighted combine) so that tests
 * can pin the mathematical equivalence of the split form to the single pass.
 *
 * Layouts (row-major, no padding):
 *   q, out      [n_seq][n_head][head_dim]              (f32 in, f64 out)
 *   k, v        [n_seq][cap][n_kv_head][head_dim]      (binary16 or bfloat16 bits)
 *   positions   [n_seq]                                (int32)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16 -> double, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. Exponent 0 holds
 * zero and the subnormals (fraction * 2^-24); exponent 31 holds inf / NaN.
 * ------------------------------------------------------------------------- */
double oracle_f16_to_double(uint16_t bits)
{
    const int sign = (bits >> 15) & 1;
    const int expo = (bits >> 10) & 0x1f;
    const int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -mag : mag;
}

/* ---------------------------------------------------------------------------
 * bfloat16 -> double, from the format's definition: 1 sign bit, 8 exponent
 * bits (bias 127), 7 fraction bits. Exponent 0 holds zero and the subnormals
 * (fraction * 2^-133); exponent 255 holds inf / NaN.
 * ------------------------------------------------------------------------- */
double oracle_bf16_to_double(uint16_t bits)
{
    const int sign = (bits >> 15) & 1;
    const int expo = (bits >> 7) & 0xff;
    const int frac = bits & 0x7f;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -133);
    else if (expo == 255)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + frac), expo - 134);
    return sign ? -mag : mag;
}

typedef double (*decode_fn)(uint16_t);

/* kv_dtype: 0 = binary16, 1 = bfloat16. */
static decode_fn decoder_for(int kv_dtype)
{
    return kv_dtype == 1 ? oracle_bf16_to_double : oracle_f16_to_double;
}

void oracle_f16_to_double_array(const uint16_t *bits, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f16_to_double(bits[i]);
}

void oracle_bf16_to_double_array(const uint16_t *bits, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_to_double(bits[i]);
}

/* Rows attended by sequence s: positions[s] + 1, clamped to [0, cap]. */
static int64_t rows_for(const int32_t *positions, int s, int64_t cap)
{
    int64_t n = (int64_t)positions[s] + 1;
    if (n < 0) n = 0;
    if (n > cap) n = cap;
    return n;
}

static int check_args(const float *q, const uint16_t *k, const uint16_t *v,
                      const int32_t *positions, const double *out, int n_seq,
                      int n_head, int n_kv_head, int head_dim, int64_t cap)
{
    if (!q || !k || !v || !positions || !out) return -1;
    if (n_seq < 0 || n_head <= 0 || n_kv_head <= 0 || head_dim <= 0 || cap < 0) return -1;
    if (n_head % n_kv_head != 0) return -1;
    return 0;
}

/* One query vector against the first n rows of one KV head's cache: a single
 * softmax over all n rows (o = 0 when n <= 0). */
static int one_query(const float *qh, const uint16_t *ks, const uint16_t *vs, int64_t row,
                     int head_dim, int64_t n, double scale, decode_fn dec, double *o)
{
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (n <= 0) return 0;

    double *x = (double *)malloc((size_t)n * sizeof(double));
    if (!x) return -2;

    /* scores x_j = scale * q . k_j */
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += (double)qh[d] * dec(ks[j * row + d]);
        x[j] = scale * dot;
        if (x[j] > m) m = x[j];
    }
    /* softmax weights and the weighted sum of V rows */
    double Z = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double w = exp(x[j] - m);
        Z += w;
        for (int d = 0; d < head_dim; ++d)
            o[d] += w * dec(vs[j * row + d]);
    }
    for (int d = 0; d < head_dim; ++d) o[d] /= Z;
    free(x);
    return 0;
}

/* One (sequence, query head) of a single-query decode. */
static int one_head(const float *q, const uint16_t *k, const uint16_t *v,
                    const int32_t *positions, double *o, int n_head,
                    int n_kv_head, int head_dim, int64_t cap, double scale,
                    int s, int h, decode_fn dec)
{
    const int G = n_head / n_kv_head;
    const int hk = h / G;
    const int64_t n = rows_for(positions, s, cap);
    const int64_t row = (int64_t)n_kv_head * head_dim;          /* elements per cache row */
    const uint16_t *ks = k + (int64_t)s * cap * row + (int64_t)hk * head_dim;
    const uint16_t *vs = v + (int64_t)s * cap * row + (int64_t)hk * head_dim;
    const float *qh = q + ((int64_t)s * n_head + h) * head_dim;
    return one_query(qh, ks, vs, row, head_dim, n, scale, dec, o);
}

/*
 * Full single-pass oracle. n_threads > 1 spreads the independent
 * (sequence, head) pairs over OpenMP threads; the arithmetic per pair is
 * unchanged. Returns 0, -1 (bad arguments) or -2 (out of host memory).
 */
int oracle_attn_decode_kv(const float *q, const uint16_t *k, const uint16_t *v,
                          const int32_t *positions, double *out, int n_seq,
                          int n_head, int n_kv_head, int head_dim, int64_t cap,
                          double scale, int n_threads, int kv_dtype)
{
    const decode_fn dec = decoder_for(kv_dtype);
    if (check_args(q, k, v, positions, out, n_seq, n_head, n_kv_head, head_dim, cap))
        return -1;
    const int64_t pairs = (int64_t)n_seq * n_head;
    int status = 0;
    if (n_threads < 1) n_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads) reduction(min : status)
    for (int64_t p = 0; p < pairs; ++p) {
        const int s = (int)(p / n_head), h = (int)(p % n_head);
        const int rc = one_head(q, k, v, positions, out + p * head_dim, n_head,
                                n_kv_head, head_dim, cap, scale, s, h, dec);
        if (rc < status) status = rc;
    }
    return status;
}

int oracle_attn_decode(const float *q, const uint16_t *k, const uint16_t *v,
                       const int32_t *positions, double *out, int n_seq,
                       int n_head, int n_kv_head, int head_dim, int64_t cap,
                       double scale, int n_threads)
{
    return oracle_attn_decode_kv(q, k, v, positions, out, n_seq, n_head, n_kv_head, head_dim,
                                 cap, scale, n_threads, 0);
}

/* One output row o[s][h][:], for sampled checks on large workloads. */
int oracle_attn_decode_one_kv(const float *q, const uint16_t *k, const uint16_t *v,
                              const int32_t *positions, double *out_row, int n_seq,
                              int n_head, int n_kv_head, int head_dim, int64_t cap,
                              double scale, int s, int h, int kv_dtype)
{
    if (check_args(q, k, v, positions, out_row, n_seq, n_head, n_kv_head, head_dim, cap))
        return -1;
    if (s < 0 || s >= n_seq || h < 0 || h >= n_head) return -1;
    return one_head(q, k, v, positions, out_row, n_head, n_kv_head, head_dim, cap,
                    scale, s, h, decoder_for(kv_dtype));
}

int oracle_attn_decode_one(const float *q, const uint16_t *k, const uint16_t *v,
                           const int32_t *positions, double *out_row, int n_seq,
                           int n_head, int n_kv_head, int head_dim, int64_t cap,
                           double scale, int s, int h)
{
    return oracle_attn_decode_one_kv(q, k, v, positions, out_row, n_seq, n_head, n_kv_head,
                                     head_dim, cap, scale, s, h, 0);
}

/*
 * Several causal query rows per sequence (the variant dotLLM #199 §2 gates
 * out: a query at position p attends cache rows [0, p]). With
 * nkv = clamp(positions[s] + 1, 0, cap), query row t of sequence s sits at
 * position nkv - n_q + t and attends its first nkv - n_q + t + 1 rows
 * (o = 0 when that count is not positive).
 * q, out: [n_seq][n_q][n_head][head_dim].
 */
int oracle_attn_decode_multi(const float *q, const uint16_t *k, const uint16_t *v,
                             const int32_t *positions, double *out, int n_seq, int n_q,
                             int n_head, int n_kv_head, int head_dim, int64_t cap,
                             double scale, int n_threads, int kv_dtype)
{
    if (check_args(q, k, v, positions, out, n_seq, n_head, n_kv_head, head_dim, cap) || n_q < 1)
        return -1;
    const decode_fn dec = decoder_for(kv_dtype);
    const int G = n_head / n_kv_head;
    const int64_t row = (int64_t)n_kv_head * head_dim;
    const int64_t items = (int64_t)n_seq * n_q * n_head;
    int status = 0;
    if (n_threads < 1) n_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads) reduction(min : status)
    for (int64_t it = 0; it < items; ++it) {
        const int h = (int)(it % n_head);
        const int t = (int)((it / n_head) % n_q);
        const int s = (int)(it / ((int64_t)n_head * n_q));
        const int hk = h / G;
        const int64_t n = rows_for(positions, s, cap) - n_q + t + 1;
        const uint16_t *ks = k + (int64_t)s * cap * row + (int64_t)hk * head_dim;
        const uint16_t *vs = v + (int64_t)s * cap * row + (int64_t)hk * head_dim;
        const int rc = one_query(q + it * head_dim, ks, vs, row, head_dim, n, scale, dec,
                                 out + it * head_dim);
        if (rc < status) status = rc;
    }
    return status;
}

/*
 * Two-stage restatement, in the order and notation of "10 · R4" §2.1-§2.2.
 * Split sp covers rows [lo, hi):
 *   split_len == 0 (by count, §2.2): chunk = ceil(nkv / P), lo = sp*chunk
 *   split_len  > 0 (fixed block, Red Lite dev35 "Change"): lo = sp*split_len
 *   hi = min(nkv, lo + chunk); the split is empty when lo >= nkv.
 * Partial, per row s_j (§2.1):
 *   nmx = max(mx, s_j); corr = exp(mx - nmx); e = exp(s_j - nmx);
 *   S = S*corr + e; oc = oc*corr + e*v_j; mx = nmx      (from mx=-inf, S=0, oc=0)
 * Combine (§2.1):
 *   gmx = max_sp mx_sp; w_sp = exp(mx_sp - gmx), taken as 0 for an empty split;
 *   o = (sum_sp w_sp*oc_sp) / (sum_sp w_sp*S_sp), and o = 0 when that sum is 0.
 * Rows past the last split (P*split_len < nkv) are not covered: the caller
 * must pass P >= ceil(nkv / split_len) in block mode.
 */
int oracle_attn_decode_split(const float *q, const uint16_t *k, const uint16_t *v,
                             const int32_t *positions, double *out, int n_seq,
                             int n_head, int n_kv_head, int head_dim, int64_t cap,
                             double scale, int n_splits, int64_t split_len)
{
    if (check_args(q, k, v, positions, out, n_seq, n_head, n_kv_head, head_dim, cap))
        return -1;
    if (n_splits <= 0 || split_len < 0) return -1;
    const int G = n_head / n_kv_head;
    const int64_t row = (int64_t)n_kv_head * head_dim;
    double *mx = (double *)malloc(sizeof(double) * (size_t)n_splits);
    double *S = (double *)malloc(sizeof(double) * (size_t)n_splits);
    double *oc = (double *)malloc(sizeof(double) * (size_t)n_splits * (size_t)head_dim);
    if (!mx || !S || !oc) { free(mx); free(S); free(oc); return -2; }

    for (int s = 0; s < n_seq; ++s) {
        const int64_t nkv = rows_for(positions, s, cap);
        const int64_t chunk = split_len > 0 ? split_len : (nkv + n_splits - 1) / n_splits;
        for (int h = 0; h < n_head; ++h) {
            const int hk = h / G;
            const float *qh = q + ((int64_t)s * n_head + h) * head_dim;
            const uint16_t *ks = k + (int64_t)s * cap * row + (int64_t)hk * head_dim;
            const uint16_t *vs = v + (int64_t)s * cap * row + (int64_t)hk * head_dim;
            /* partial stage */
            for (int sp = 0; sp < n_splits; ++sp) {
                double m_ = -INFINITY, S_ = 0.0;
                double *oc_ = oc + (int64_t)sp * head_dim;
                for (int d = 0; d < head_dim; ++d) oc_[d] = 0.0;
                const int64_t lo = (int64_t)sp * chunk;
                const int64_t hi = lo + chunk < nkv ? lo + chunk : nkv;
                for (int64_t j = lo; j < hi; ++j) {
                    double dot = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        dot += (double)qh[d] * oracle_f16_to_double(ks[j * row + d]);
                    const double sj = dot * scale;
                    const double nmx = sj > m_ ? sj : m_;
                    const double corr = exp(m_ - nmx);
                    const double e = exp(sj - nmx);
                    S_ = S_ * corr + e;
                    for (int d = 0; d < head_dim; ++d)
                        oc_[d] = oc_[d] * corr + e * oracle_f16_to_double(vs[j * row + d]);
                    m_ = nmx;
                }
                mx[sp] = m_;
                S[sp] = S_;
            }
            /* combine stage */
            double gmx = -INFINITY;
            for (int sp = 0; sp < n_splits; ++sp)
                if (mx[sp] > gmx) gmx = mx[sp];
            double Ssum = 0.0;
            double *o = out + ((int64_t)s * n_head + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            for (int sp = 0; sp < n_splits; ++sp) {
                const double w = (mx[sp] == -INFINITY) ? 0.0 : exp(mx[sp] - gmx);
                Ssum += w * S[sp];
                for (int d = 0; d < head_dim; ++d) o[d] += w * oc[(int64_t)sp * head_dim + d];
            }
            for (int d = 0; d < head_dim; ++d) o[d] = Ssum > 0.0 ? o[d] / Ssum : 0.0;
        }
    }
    free(mx); free(S); free(oc);
    return 0;
}
