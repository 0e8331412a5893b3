/*
 * sdpa_oracle.c -- plain, slow, fp64 CPU reference for scaled-dot-product
 * attention: the forward (O, LSE) and the backward (dQ, dK, dV).
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. The GPU library shares no
 * code, header, table or helper with it, and neither side includes the other.
 *
 * Source of the arithmetic ("SDPA Backward (SM120)" page of the cuDNN
 * frontend docs):
 *   - API Usage: tensors are logical (B, H, S, D); `stats` is the natural-log
 *     forward LSE; scale defaults to 1/sqrt(D); K/V carry H_kv heads and
 *     H_kv divides H_q (GQA/MQA).
 *   - Main-kernel pipeline: P replayed from LSE, dP = dO V^T,
 *     delta = rowsum(O * dO), dS = P * (dP - delta), dV = P^T dO,
 *     dQ = scale * dS K, dK = scale * dS^T Q.
 *   - GQA/MQA group reduction: the KV head of query head h is h / group and
 *     dK/dV of a KV head sum over the query heads of its group.
 *   - Causal, sliding-window, and padding masks: diag = 0 (top-left) or
 *     L_kv - L_q (bottom-right, anchored at the actual lengths); causal keeps
 *     k <= q + diag + R; a left window masks k < q + diag - W; keys at or past
 *     seq_kv_lens[b] and queries at or past seq_q_lens[b] are masked; a row
 *     with no visible key has LSE = -inf and gets P = 0 (not NaN).
 *   - Sink tokens (Capabilities list and the `dsink` step of the kernel
 *     chain): a per-query-head sink logit joins every row's softmax
 *     denominator without a value row, so the forward LSE includes it and
 *     dQ/dK/dV keep their formulas; the extra output is
 *     dsink[h] = -sum_{b,q} exp(sink[h] - LSE[b,h,q]) * delta[b,h,q].
 *   - NVFP4 QAT backward (page "NVFP4 Attention QAT Backward", Overview): see
 *     the section of that name at the end of this file.
 *   - Additive bias (Capabilities list): a (1|B, H_q, S_q, S_kv) tensor added
 *     to the scaled scores before the softmax, s_qk = scale * Q_q.K_k +
 *     bias[b,h,q,k]; the forward LSE includes it, so the backward replays P
 *     with it and keeps its formulas. The extra output is the gradient of the
 *     bias, dBias = dS (the softmax VJP without the scale factor), summed over
 *     the batch when one bias batch serves every batch row.
 *
 * Every quantity is computed straight from its definition, one output row at
 * a time, in double precision. There is no tiling, fusion or reordering.
 * Rows are independent, so OpenMP splits the row loops across threads; each
 * output element is written by exactly one thread.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int B, Hq, Hkv, Sq, Skv, Dqk, Dv;
    double scale;         /* applied to Q.K; the caller resolves the default */
    int causal;           /* 1: keep k <= q + diag + max(R, 0)               */
    int bottom_right;     /* 1: diag = L_kv - L_q, else diag = 0             */
    int window_left;      /* W >= 0: mask k < q + diag - W; < 0: no window   */
    int window_right;     /* R: widens the causal diagonal; < 0 means 0      */
    const int32_t *seq_q_lens;   /* (B,) or NULL: every row is S_q long     */
    const int32_t *seq_kv_lens;  /* (B,) or NULL: every row is S_kv long    */
    const double *bias;   /* (bias_batch, Hq, Sq, Skv) additive bias, or NULL */
    int bias_batch;       /* 1 (shared by every batch row) or B              */
} oracle_cfg;

/* ---- the mask predicate ("Causal, sliding-window, and padding masks") ---- */

static void lengths(const oracle_cfg *c, int b, int *Lq, int *Lk) {
    *Lq = c->seq_q_lens ? c->seq_q_lens[b] : c->Sq;
    *Lk = c->seq_kv_lens ? c->seq_kv_lens[b] : c->Skv;
    if (*Lq > c->Sq) *Lq = c->Sq;
    if (*Lk > c->Skv) *Lk = c->Skv;
    if (*Lq < 0) *Lq = 0;
    if (*Lk < 0) *Lk = 0;
}

static int visible(const oracle_cfg *c, int Lq, int Lk, long q, long k) {
    long diag = c->bottom_right ? (long)Lk - (long)Lq : 0;
    if (q >= Lq || k >= Lk) return 0;
    if (c->causal) {
        long R = c->window_right > 0 ? c->window_right : 0;
        if (k > q + diag + R) return 0;
    }
    if (c->window_left >= 0 && k < q + diag - c->window_left) return 0;
    return 1;
}

/* ---- index helpers: contiguous (B, H, S, D) ---- */

static inline const double *row_of(const double *t, long bh, long s, long S, long D) {
    return t + (bh * S + s) * D;
}

static double dot(const double *a, const double *b, int n) {
    double acc = 0.0;
    for (int i = 0; i < n; ++i) acc += a[i] * b[i];
    return acc;
}

/* Bias of query head bh (= b * Hq + h) at (q, k); 0 without a bias. */
static double bias_at(const oracle_cfg *c, long bh, long q, long k) {
    if (!c->bias) return 0.0;
    long b = bh / c->Hq, h = bh % c->Hq;
    long bb = c->bias_batch == 1 ? 0 : b;
    return c->bias[((bb * c->Hq + h) * c->Sq + q) * c->Skv + k];
}

/* The score that enters the softmax: scale * Q_q . K_k + bias. */
static double score(const oracle_cfg *c, const double *qr, const double *kr, long bh, long q,
                    long k) {
    return c->scale * dot(qr, kr, c->Dqk) + bias_at(c, bh, q, k);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Number of visible (q, k) pairs summed over batches and query heads. */
long long oracle_count_visible(const oracle_cfg *c) {
    long long total = 0;
    for (int b = 0; b < c->B; ++b) {
        int Lq, Lk;
        lengths(c, b, &Lq, &Lk);
        long long per_head = 0;
        for (long q = 0; q < c->Sq; ++q)
            for (long k = 0; k < c->Skv; ++k) per_head += visible(c, Lq, Lk, q, k);
        total += per_head * c->Hq;
    }
    return total;
}

/* Forward: LSE_q = log( sum_{visible k} exp(s_qk) [+ exp(sink_h)] ),
 * s_qk = scale * Q_q . K_k [+ bias]; O_q = sum_k exp(s_qk - LSE_q) V_k (the sink has no
 * value row). Without a sink an empty row gives LSE = -inf, O = 0; with one it
 * gives LSE = sink_h, O = 0. Rows at or past seq_q_lens[b] are empty rows.
 * `sink` is (H_q,) or NULL. */
void oracle_forward_sink(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                         const double *sink, double *O, double *LSE) {
    const int G = c->Hq / c->Hkv;
    const long rows = (long)c->B * c->Hq * c->Sq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(c->Skv > 0 ? c->Skv : 1));
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            long q = r % c->Sq, bh = r / c->Sq;
            int b = (int)(bh / c->Hq), h = (int)(bh % c->Hq);
            long bhk = (long)b * c->Hkv + h / G;
            int Lq, Lk;
            lengths(c, b, &Lq, &Lk);
            const double *qr = row_of(Q, bh, q, c->Sq, c->Dqk);
            double *orow = O + r * c->Dv;
            const double sk = sink ? sink[h] : -INFINITY;
            double m = sk;
            for (long k = 0; k < c->Skv; ++k) {
                if (!visible(c, Lq, Lk, q, k)) continue;
                s[k] = score(c, qr, row_of(K, bhk, k, c->Skv, c->Dqk), bh, q, k);
                if (s[k] > m) m = s[k];
            }
            for (int d = 0; d < c->Dv; ++d) orow[d] = 0.0;
            if (m == -INFINITY) { LSE[r] = -INFINITY; continue; }
            double l = sink ? exp(sk - m) : 0.0;
            for (long k = 0; k < c->Skv; ++k)
                if (visible(c, Lq, Lk, q, k)) l += exp(s[k] - m);
            double lse = m + log(l);
            LSE[r] = lse;
            for (long k = 0; k < c->Skv; ++k) {
                if (!visible(c, Lq, Lk, q, k)) continue;
                double p = exp(s[k] - lse);
                const double *vr = row_of(V, bhk, k, c->Skv, c->Dv);
                for (int d = 0; d < c->Dv; ++d) orow[d] += p * vr[d];
            }
        }
        free(s);
    }
}

void oracle_forward(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                    double *O, double *LSE) {
    oracle_forward_sink(c, Q, K, V, NULL, O, LSE);
}

/* dsink[h] = -sum over b and query rows q < L_q of P_sink * delta, with
 * P_sink = exp(sink[h] - LSE[b,h,q]) (0 when LSE = -inf, as for P). Summed in
 * ascending (b, q) order in double precision. */
void oracle_dsink(const oracle_cfg *c, const double *sink, const double *LSE, const double *delta,
                  double *dsink) {
    for (int h = 0; h < c->Hq; ++h) {
        double acc = 0.0;
        for (int b = 0; b < c->B; ++b) {
            int Lq, Lk;
            lengths(c, b, &Lq, &Lk);
            const long bh = (long)b * c->Hq + h;
            for (long q = 0; q < Lq; ++q) {
                const double lse = LSE[bh * c->Sq + q];
                if (lse == -INFINITY) continue;
                acc += exp(sink[h] - lse) * delta[bh * c->Sq + q];
            }
        }
        dsink[h] = -acc;
    }
}

/* delta_q = sum_d dO[q, d] * O[q, d] ("dot" step of the kernel chain). */
void oracle_delta(const oracle_cfg *c, const double *O, const double *dO, double *delta) {
    const long rows = (long)c->B * c->Hq * c->Sq;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) delta[r] = dot(O + r * c->Dv, dO + r * c->Dv, c->Dv);
}

/* P_qk replayed from the given LSE; zero when masked or when LSE = -inf. */
static double prob(const oracle_cfg *c, double s, double lse) {
    (void)c;
    if (lse == -INFINITY) return 0.0;
    return exp(s - lse);
}

/* dQ row (b, h, q): scale * sum_k dS_qk K_k with dS_qk = P_qk (dP_qk - delta_q). */
static void dq_row(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                   const double *dO, const double *LSE, const double *delta, long bh, long q,
                   double *out) {
    const int G = c->Hq / c->Hkv;
    int b = (int)(bh / c->Hq), h = (int)(bh % c->Hq);
    long bhk = (long)b * c->Hkv + h / G;
    int Lq, Lk;
    lengths(c, b, &Lq, &Lk);
    const double *qr = row_of(Q, bh, q, c->Sq, c->Dqk);
    const double *dor = row_of(dO, bh, q, c->Sq, c->Dv);
    double lse = LSE[bh * c->Sq + q], D = delta[bh * c->Sq + q];
    for (int d = 0; d < c->Dqk; ++d) out[d] = 0.0;
    for (long k = 0; k < c->Skv; ++k) {
        if (!visible(c, Lq, Lk, q, k)) continue;
        const double *kr = row_of(K, bhk, k, c->Skv, c->Dqk);
        double p = prob(c, score(c, qr, kr, bh, q, k), lse);
        double dp = dot(dor, row_of(V, bhk, k, c->Skv, c->Dv), c->Dv);
        double ds = p * (dp - D);
        for (int d = 0; d < c->Dqk; ++d) out[d] += ds * kr[d];
    }
    for (int d = 0; d < c->Dqk; ++d) out[d] *= c->scale;
}

/* dK, dV row (b, hk, k): sums over every query head of the KV head's group and
 * every visible query: dK_k = scale * sum dS_qk Q_q, dV_k = sum P_qk dO_q. */
static void dkv_row(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                    const double *dO, const double *LSE, const double *delta, long bhk, long k,
                    double *dk_out, double *dv_out) {
    const int G = c->Hq / c->Hkv;
    int b = (int)(bhk / c->Hkv), hk = (int)(bhk % c->Hkv);
    int Lq, Lk;
    lengths(c, b, &Lq, &Lk);
    const double *kr = row_of(K, bhk, k, c->Skv, c->Dqk);
    const double *vr = row_of(V, bhk, k, c->Skv, c->Dv);
    for (int d = 0; d < c->Dqk; ++d) dk_out[d] = 0.0;
    for (int d = 0; d < c->Dv; ++d) dv_out[d] = 0.0;
    for (int j = 0; j < G; ++j) {
        long bh = (long)b * c->Hq + (long)hk * G + j;
        for (long q = 0; q < c->Sq; ++q) {
            if (!visible(c, Lq, Lk, q, k)) continue;
            const double *qr = row_of(Q, bh, q, c->Sq, c->Dqk);
            const double *dor = row_of(dO, bh, q, c->Sq, c->Dv);
            double p = prob(c, score(c, qr, kr, bh, q, k), LSE[bh * c->Sq + q]);
            double dp = dot(dor, vr, c->Dv);
            double ds = p * (dp - delta[bh * c->Sq + q]);
            for (int d = 0; d < c->Dqk; ++d) dk_out[d] += ds * qr[d];
            for (int d = 0; d < c->Dv; ++d) dv_out[d] += p * dor[d];
        }
    }
    for (int d = 0; d < c->Dqk; ++d) dk_out[d] *= c->scale;
}

/* Full backward: every dQ row and every dK/dV row. */
void oracle_backward(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                     const double *O, const double *dO, const double *LSE, double *dQ,
                     double *dK, double *dV) {
    const long qrows = (long)c->B * c->Hq * c->Sq;
    const long krows = (long)c->B * c->Hkv * c->Skv;
    double *delta = (double *)malloc(sizeof(double) * (size_t)(qrows > 0 ? qrows : 1));
    oracle_delta(c, O, dO, delta);
#pragma omp parallel for schedule(dynamic, 8)
    for (long r = 0; r < qrows; ++r)
        dq_row(c, Q, K, V, dO, LSE, delta, r / c->Sq, r % c->Sq, dQ + r * c->Dqk);
#pragma omp parallel for schedule(dynamic, 8)
    for (long r = 0; r < krows; ++r)
        dkv_row(c, Q, K, V, dO, LSE, delta, r / c->Skv, r % c->Skv, dK + r * c->Dqk,
                dV + r * c->Dv);
    free(delta);
}

/* Sampled backward: dQ at the flat query-row indices q_idx ((b*Hq + h)*Sq + q)
 * and dK/dV at the flat key-row indices k_idx ((b*Hkv + hk)*Skv + k). */
void oracle_backward_sampled(const oracle_cfg *c, const double *Q, const double *K,
                             const double *V, const double *O, const double *dO,
                             const double *LSE, long n_q, const int64_t *q_idx, double *dQ_rows,
                             long n_k, const int64_t *k_idx, double *dK_rows, double *dV_rows) {
    const long qrows = (long)c->B * c->Hq * c->Sq;
    double *delta = (double *)malloc(sizeof(double) * (size_t)(qrows > 0 ? qrows : 1));
    oracle_delta(c, O, dO, delta);
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < n_q; ++i)
        dq_row(c, Q, K, V, dO, LSE, delta, q_idx[i] / c->Sq, q_idx[i] % c->Sq,
               dQ_rows + i * c->Dqk);
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < n_k; ++i)
        dkv_row(c, Q, K, V, dO, LSE, delta, k_idx[i] / c->Skv, k_idx[i] % c->Skv,
                dK_rows + i * c->Dqk, dV_rows + i * c->Dv);
    free(delta);
}

/* dBias (bias_batch, Hq, Sq, Skv): dS_qk = P_qk (dP_qk - delta_q) at every
 * visible pair, 0 elsewhere; with bias_batch = 1 (and B > 1) the batch rows'
 * dS are summed, in ascending b order. Requires c->bias (P replays the biased
 * scores). */
/* One dBias row: flat bias row r = (bb * Hq + h) * Sq + q, all S_kv keys. */
static void dbias_row(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                      const double *dO, const double *LSE, const double *delta, long r,
                      double *out) {
    const int G = c->Hq / c->Hkv;
    const long q = r % c->Sq, bbh = r / c->Sq;
    const int bb = (int)(bbh / c->Hq), h = (int)(bbh % c->Hq);
    for (long k = 0; k < c->Skv; ++k) out[k] = 0.0;
    const int b_lo = c->bias_batch == 1 ? 0 : bb;
    const int b_hi = c->bias_batch == 1 ? c->B : bb + 1;
    for (int b = b_lo; b < b_hi; ++b) {
        int Lq, Lk;
        lengths(c, b, &Lq, &Lk);
        const long bh = (long)b * c->Hq + h, bhk = (long)b * c->Hkv + h / G;
        const double *qr = row_of(Q, bh, q, c->Sq, c->Dqk);
        const double *dor = row_of(dO, bh, q, c->Sq, c->Dv);
        const double lse = LSE[bh * c->Sq + q], D = delta[bh * c->Sq + q];
        for (long k = 0; k < c->Skv; ++k) {
            if (!visible(c, Lq, Lk, q, k)) continue;
            const double *kr = row_of(K, bhk, k, c->Skv, c->Dqk);
            double p = prob(c, score(c, qr, kr, bh, q, k), lse);
            double dp = dot(dor, row_of(V, bhk, k, c->Skv, c->Dv), c->Dv);
            out[k] += p * (dp - D);
        }
    }
}

void oracle_dbias(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                  const double *O, const double *dO, const double *LSE, double *dBias) {
    const long qrows = (long)c->B * c->Hq * c->Sq;
    double *delta = (double *)malloc(sizeof(double) * (size_t)(qrows > 0 ? qrows : 1));
    oracle_delta(c, O, dO, delta);
    const long out_rows = (long)c->bias_batch * c->Hq * c->Sq;
#pragma omp parallel for schedule(dynamic, 8)
    for (long r = 0; r < out_rows; ++r) dbias_row(c, Q, K, V, dO, LSE, delta, r, dBias + r * c->Skv);
    free(delta);
}

/* dBias at the flat bias rows rows[i] = (bb * Hq + h) * Sq + q: out is (n, S_kv). */
void oracle_dbias_rows(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                       const double *O, const double *dO, const double *LSE, long n,
                       const int64_t *rows, double *out) {
    const long qrows = (long)c->B * c->Hq * c->Sq;
    double *delta = (double *)malloc(sizeof(double) * (size_t)(qrows > 0 ? qrows : 1));
    oracle_delta(c, O, dO, delta);
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < n; ++i) dbias_row(c, Q, K, V, dO, LSE, delta, rows[i], out + i * c->Skv);
    free(delta);
}

/* ---- NVFP4 fake quantization and the QAT backward ("NVFP4 Attention QAT
 * Backward" page, Overview). Q, K and V are fake-quantized in blocks of 16
 * consecutive values along the head dimension: each block gets a local scale
 * in E4M3 and its values are rounded to E2M1 multiples of that scale. P = the
 * softmax of the quantized scores; dQ and dK use P itself (straight-through
 * estimator) and dV uses P fake-quantized in blocks of 16 consecutive keys of
 * a query row. The local scale is amax / 6 and each value is divided by the
 * scale, both as correctly rounded fp32 divisions (the page's "precise
 * division"), so that the E2M1 rounding sees exact midpoints as midpoints. ---- */

/* |a| rounded to a multiple of `quantum` (a power of two), ties to even. */
static double round_to_quantum(double a, double quantum) {
    return nearbyint(a / quantum) * quantum;
}

/* Nearest E4M3 value: sign, 4 exponent bits (bias 7), 3 mantissa bits; normal
 * magnitudes 2^-6 .. 448, subnormal steps of 2^-9, no infinities. Ties go to the
 * even mantissa; magnitudes beyond 448 saturate to 448. */
double oracle_round_e4m3(double x) {
    double a = fabs(x), q;
    if (a >= 448.0) {
        q = 448.0;
    } else if (a < 0.015625) {          /* below 2^-6: subnormal grid */
        q = round_to_quantum(a, 0.001953125);
    } else {
        int e;
        frexp(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
        q = round_to_quantum(a, ldexp(1.0, e - 1 - 3));
        if (q > 448.0) q = 448.0;
    }
    return x < 0 ? -q : q;
}

/* Nearest E2M1 value: sign, 2 exponent bits (bias 1), 1 mantissa bit; the
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. Ties go to the even mantissa;
 * magnitudes beyond 6 saturate to 6. */
double oracle_round_e2m1(double x) {
    double a = fabs(x), q;
    if (a < 2.0) q = round_to_quantum(a, 0.5);        /* 0, 0.5 | 1, 1.5 */
    else if (a < 4.0) q = round_to_quantum(a, 1.0);   /* 2, 3 */
    else q = round_to_quantum(a, 2.0);                /* 4, 6 */
    if (q > 6.0) q = 6.0;
    return x < 0 ? -q : q;
}

/* One block of n <= 16 values (a short block at the end of a row counts only
 * its own values). */
static void fake_nvfp4_block(const double *x, double *y, int n) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf((float)x[i]);
        if (a > amax) amax = a;
    }
    const float s = (float)oracle_round_e4m3((double)(amax / 6.0f));
    for (int i = 0; i < n; ++i)
        y[i] = s == 0.0f ? 0.0 : oracle_round_e2m1((double)((float)x[i] / s)) * (double)s;
}

/* Fake-quantizes `rows` rows of `cols` values (blocks of 16 along each row). */
void oracle_fake_nvfp4(const double *x, double *y, long rows, int cols) {
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r)
        for (int c0 = 0; c0 < cols; c0 += 16)
            fake_nvfp4_block(x + r * cols + c0, y + r * cols + c0, cols - c0 < 16 ? cols - c0 : 16);
}

static double *fake_copy(const double *x, long rows, int cols) {
    double *y = (double *)malloc(sizeof(double) * (size_t)(rows * cols > 0 ? rows * cols : 1));
    oracle_fake_nvfp4(x, y, rows, cols);
    return y;
}

/* The fake-quantized probability matrix of query head bh: Ph[q * Skv + k] =
 * fake_nvfp4 of P's row q (blocks of 16 keys), P = exp(score - LSE) at visible
 * pairs and 0 elsewhere, scores from the given (already quantized) Q and K. */
static void qat_probabilities(const oracle_cfg *c, const double *Qh, const double *Kh,
                              const double *LSE, long bh, double *Ph) {
    const int G = c->Hq / c->Hkv;
    const int b = (int)(bh / c->Hq), h = (int)(bh % c->Hq);
    const long bhk = (long)b * c->Hkv + h / G;
    int Lq, Lk;
    lengths(c, b, &Lq, &Lk);
#pragma omp parallel
    {
        double *prow = (double *)malloc(sizeof(double) * (size_t)(c->Skv > 0 ? c->Skv : 1));
#pragma omp for schedule(dynamic, 8)
        for (long q = 0; q < c->Sq; ++q) {
            const double *qr = row_of(Qh, bh, q, c->Sq, c->Dqk);
            const double lse = LSE[bh * c->Sq + q];
            for (long k = 0; k < c->Skv; ++k)
                prow[k] = visible(c, Lq, Lk, q, k)
                              ? prob(c, score(c, qr, row_of(Kh, bhk, k, c->Skv, c->Dqk), bh, q, k), lse)
                              : 0.0;
            oracle_fake_nvfp4(prow, Ph + q * c->Skv, 1, c->Skv);
        }
        free(prow);
    }
}

/* QAT forward: O_hp and LSE are the plain forward of the fake-quantized Q, K,
 * V (O_hp = P V_hat with P unquantized, "high precision"); O_user = fq(P) V_hat
 * is the user-visible output. Any of the outputs may be NULL. */
void oracle_qat_forward(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                        double *O_hp, double *LSE, double *O_user) {
    const long qrows = (long)c->B * c->Hq * c->Sq, krows = (long)c->B * c->Hkv * c->Skv;
    double *Qh = fake_copy(Q, qrows, c->Dqk), *Kh = fake_copy(K, krows, c->Dqk);
    double *Vh = fake_copy(V, krows, c->Dv);
    double *o = O_hp ? O_hp : (double *)malloc(sizeof(double) * (size_t)(qrows * c->Dv > 0 ? qrows * c->Dv : 1));
    double *l = LSE ? LSE : (double *)malloc(sizeof(double) * (size_t)(qrows > 0 ? qrows : 1));
    oracle_forward_sink(c, Qh, Kh, Vh, NULL, o, l);
    if (O_user) {
        const int G = c->Hq / c->Hkv;
        double *Ph = (double *)malloc(sizeof(double) * (size_t)((long)c->Sq * c->Skv > 0 ? (long)c->Sq * c->Skv : 1));
        for (long bh = 0; bh < (long)c->B * c->Hq; ++bh) {
            qat_probabilities(c, Qh, Kh, l, bh, Ph);
            const long bhk = (bh / c->Hq) * c->Hkv + (bh % c->Hq) / G;
#pragma omp parallel for schedule(static)
            for (long q = 0; q < c->Sq; ++q) {
                double *out = O_user + (bh * c->Sq + q) * c->Dv;
                for (int d = 0; d < c->Dv; ++d) out[d] = 0.0;
                for (long k = 0; k < c->Skv; ++k) {
                    const double p = Ph[q * c->Skv + k];
                    if (p == 0.0) continue;
                    const double *vr = row_of(Vh, bhk, k, c->Skv, c->Dv);
                    for (int d = 0; d < c->Dv; ++d) out[d] += p * vr[d];
                }
            }
        }
        free(Ph);
    }
    if (!O_hp) free(o);
    if (!LSE) free(l);
    free(Qh); free(Kh); free(Vh);
}

/* QAT backward: dQ = scale dS K_hat, dK = scale dS^T Q_hat with dS = P (dP -
 * delta), dP = dO V_hat^T, delta = rowsum(O_hp * dO) (P unquantized), and
 * dV = fq(P)^T dO. O is the high-precision forward output, LSE its statistic. */
void oracle_qat_backward(const oracle_cfg *c, const double *Q, const double *K, const double *V,
                         const double *O, const double *dO, const double *LSE, double *dQ,
                         double *dK, double *dV) {
    const int G = c->Hq / c->Hkv;
    const long qrows = (long)c->B * c->Hq * c->Sq, krows = (long)c->B * c->Hkv * c->Skv;
    double *Qh = fake_copy(Q, qrows, c->Dqk), *Kh = fake_copy(K, krows, c->Dqk);
    double *Vh = fake_copy(V, krows, c->Dv);
    double *delta = (double *)malloc(sizeof(double) * (size_t)(qrows > 0 ? qrows : 1));
    double *dv_plain = (double *)malloc(sizeof(double) * (size_t)(krows * c->Dv > 0 ? krows * c->Dv : 1));
    oracle_delta(c, O, dO, delta);
#pragma omp parallel for schedule(dynamic, 8)
    for (long r = 0; r < qrows; ++r)
        dq_row(c, Qh, Kh, Vh, dO, LSE, delta, r / c->Sq, r % c->Sq, dQ + r * c->Dqk);
#pragma omp parallel for schedule(dynamic, 8)
    for (long r = 0; r < krows; ++r)
        dkv_row(c, Qh, Kh, Vh, dO, LSE, delta, r / c->Skv, r % c->Skv, dK + r * c->Dqk,
                dv_plain + r * c->Dv);
    /* dV with the fake-quantized probabilities, head by head of each group */
    for (long r = 0; r < krows * c->Dv; ++r) dV[r] = 0.0;
    double *Ph = (double *)malloc(sizeof(double) * (size_t)((long)c->Sq * c->Skv > 0 ? (long)c->Sq * c->Skv : 1));
    for (long bh = 0; bh < qrows / (c->Sq > 0 ? c->Sq : 1); ++bh) {
        qat_probabilities(c, Qh, Kh, LSE, bh, Ph);
        const long bhk = (bh / c->Hq) * c->Hkv + (bh % c->Hq) / G;
#pragma omp parallel for schedule(static)
        for (long k = 0; k < c->Skv; ++k) {
            double *out = dV + (bhk * c->Skv + k) * c->Dv;
            for (long q = 0; q < c->Sq; ++q) {
                const double p = Ph[q * c->Skv + k];
                if (p == 0.0) continue;
                const double *dor = row_of(dO, bh, q, c->Sq, c->Dv);
                for (int d = 0; d < c->Dv; ++d) out[d] += p * dor[d];
            }
        }
    }
    free(Ph); free(dv_plain); free(delta);
    free(Qh); free(Kh); free(Vh);
}
