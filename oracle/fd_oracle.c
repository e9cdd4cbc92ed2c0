/*
 * fd_oracle.c -- plain fp64 CPU oracle for length-aware GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header or constant with the CUDA
 * library: it reads the same raw input bits (bf16 / int8 / fp32 scales) and
 * computes the definition directly, with no blocking, splitting or online
 * rescaling.
 *
 * What it computes (the plain reading of the pages):
 *   "Qwen3.5 text generation attends over the full KV capacity" issue
 *   (ComfyUI #16509), problem statement: decode computes q @ key and masks
 *   the unused tail of the preallocated cache; the length-aware kernel reads
 *   only the filled part given by a device-side length per sequence.
 *   Same issue, "Existing Solutions": the case is several queries with a
 *   bottom-right-aligned causal mask, GQA, head dims up to 256.
 *   "attend the selected cells instead of masking the window" (llama.cpp
 *   #28244), Conversation: the gather attends only the selected cells, one
 *   list per query, and must give what the mask path gives.
 *   comfy-kitchen #239, commit list ("Add bounded paged INT8 decode cache"):
 *   an int8 KV cache; here with one fp32 scale per (token, kv head).
 *
 * For sequence b, query row i (0 <= i < n_q), query head h, kv head
 * hk = h / (Hq / Hkv):
 *   visible set V:
 *     dense, non-causal : { j : 0 <= j < L }
 *     dense, causal     : { j : 0 <= j <= L - n_q + i }   (bottom-right)
 *     gather            : { idx[b,i,t] : 0 <= t < K, 0 <= idx[b,i,t] < cap }
 *                         (with a per-cell bias: minus the cells whose bias
 *                         bias[b,i,t] is -inf)
 *   with L = kv_lengths[b] clamped to [0, cap].
 *   s_j   = scale * sum_d q[b,i,h,d] * k[b,hk,j,d]   (+ bias[b,i,t] for the
 *           list entry t that names j: "qwen4exp : gather-based sparse
 *           attention for QSA decode", llama.cpp #28213, Overview -- the
 *           per-cell mask entries are gathered with the cells and added)
 *   out   = sum_{j in V} exp(s_j - max s) v[b,hk,j,:] / sum_{j in V} exp(s_j - max s)
 *   out   = 0 when V is empty.
 * k, v are the stored bf16 values, or int8 * fp32 scale for int8 caches
 * (the product taken in fp64).  All arithmetic is fp64.
 *
 * Layouts: every tensor is addressed through element strides, so canonical
 * [B, Hkv, cap, d] and token-major [B, cap, Hkv, d] caches both work.
 *   q   : [B, n_q, Hq, d]  bf16 bits
 *   k,v : [B, Hkv, cap, d] bf16 bits or int8
 *   ks,vs (int8 only): [B, Hkv, cap] fp32
 *   idx : [B, n_q, K]      int32, contiguous
 *   out : [B, n_q, Hq, d]  fp64, contiguous
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: the bf16 value is the fp32 value
 * whose upper 16 bits are the pattern. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const void *k, *v;
    int kv_int8;                  /* 0: bf16 bits, 1: int8 */
    const int64_t *ks, *vs;       /* element strides of k, v (4 each) */
    const float *k_scale, *v_scale;
    const int64_t *ss;            /* element strides of the scales (3) */
} kv_src;

/* Value of k or v at (b, hk, j, dd) as a double. */
static double kv_at(const kv_src *src, int which, int64_t b, int64_t hk,
                    int64_t j, int64_t dd)
{
    const int64_t *st = which ? src->vs : src->ks;
    int64_t off = b * st[0] + hk * st[1] + j * st[2] + dd * st[3];
    if (!src->kv_int8) {
        const uint16_t *p = (const uint16_t *)(which ? src->v : src->k);
        return bf16_bits_to_double(p[off]);
    }
    const int8_t *p = (const int8_t *)(which ? src->v : src->k);
    const float *sc = which ? src->v_scale : src->k_scale;
    double s = (double)sc[b * src->ss[0] + hk * src->ss[1] + j * src->ss[2]];
    return (double)p[off] * s;
}

/* One output row: softmax over the visible keys `vis[0..n)` (a multiset of
 * cache positions), weighted sum of the matching value rows. */
static void attend_row(const kv_src *src, int64_t b, int64_t hk,
                       const double *qrow, int d, double scale,
                       const int64_t *vis, const double *add, int64_t n,
                       double *score, double *orow)
{
    for (int dd = 0; dd < d; ++dd)
        orow[dd] = 0.0;
    if (n == 0)
        return;
    double mx = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int dd = 0; dd < d; ++dd)
            dot += qrow[dd] * kv_at(src, 0, b, hk, vis[t], dd);
        score[t] = scale * dot + (add ? add[t] : 0.0);
        if (score[t] > mx)
            mx = score[t];
    }
    double den = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        score[t] = exp(score[t] - mx);
        den += score[t];
    }
    for (int64_t t = 0; t < n; ++t)
        for (int dd = 0; dd < d; ++dd)
            orow[dd] += score[t] * kv_at(src, 1, b, hk, vis[t], dd);
    for (int dd = 0; dd < d; ++dd)
        orow[dd] /= den;
}

/* mode 0: dense prefix (causal or not); mode 1: index gather (bias: NULL,
 * or one fp32 value per list entry added to its score, -inf dropping it). */
static int run(int mode, const uint16_t *q, const int64_t *qs,
               const kv_src *src, const int32_t *kv_lengths,
               const int32_t *idx, const float *bias, int64_t K, int B, int n_q, int Hq,
               int Hkv, int d, int64_t cap, int causal, double scale,
               double *out)
{
    if (B < 0 || n_q < 1 || Hq < 1 || Hkv < 1 || d < 1 || cap < 0 ||
        Hq % Hkv != 0)
        return -1;
    const int g = Hq / Hkv;
    const int64_t rows = (int64_t)B * n_q * Hq;
    int err = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t b = r / ((int64_t)n_q * Hq);
        const int64_t i = (r / Hq) % n_q;
        const int64_t h = r % Hq;
        const int64_t hk = h / g;
        double *orow = out + r * d;

        int64_t cnt = mode == 0 ? cap : K;
        int64_t *vis = (int64_t *)malloc((size_t)(cnt > 0 ? cnt : 1) * sizeof *vis);
        double *score = (double *)malloc((size_t)(cnt > 0 ? cnt : 1) * sizeof *score);
        double *qrow = (double *)malloc((size_t)d * sizeof *qrow);
        double *add = bias ? (double *)malloc((size_t)(cnt > 0 ? cnt : 1) * sizeof *add) : NULL;
        if (!vis || !score || !qrow || (bias && !add)) {
#pragma omp atomic write
            err = -2;
            free(vis); free(score); free(qrow); free(add);
            continue;
        }
        for (int dd = 0; dd < d; ++dd)
            qrow[dd] = bf16_bits_to_double(
                q[b * qs[0] + i * qs[1] + h * qs[2] + dd * qs[3]]);

        int64_t n = 0;
        if (mode == 0) {
            int64_t L = kv_lengths[b];
            if (L < 0) L = 0;
            if (L > cap) L = cap;
            int64_t last = causal ? L - n_q + i : L - 1; /* inclusive */
            for (int64_t j = 0; j <= last; ++j)
                vis[n++] = j;
        } else {
            const int32_t *list = idx + (b * n_q + i) * K;
            const float *brow = bias ? bias + (b * n_q + i) * K : NULL;
            for (int64_t t = 0; t < K; ++t)
                if (list[t] >= 0 && (int64_t)list[t] < cap &&
                    !(brow && isinf(brow[t]) && brow[t] < 0)) {
                    if (brow)
                        add[n] = (double)brow[t];
                    vis[n++] = list[t];
                }
        }
        attend_row(src, b, hk, qrow, d, scale, vis, add, n, score, orow);
        free(vis); free(score); free(qrow); free(add);
    }
    return err;
}

int fdo_dense(const uint16_t *q, const int64_t *q_strides,
              const void *k, const int64_t *k_strides,
              const void *v, const int64_t *v_strides, int kv_int8,
              const float *k_scale, const float *v_scale,
              const int64_t *scale_strides, const int32_t *kv_lengths,
              int B, int n_q, int Hq, int Hkv, int d, int64_t cap,
              int causal, double scale, double *out)
{
    kv_src src = {k, v, kv_int8, k_strides, v_strides, k_scale, v_scale,
                  scale_strides};
    return run(0, q, q_strides, &src, kv_lengths, NULL, NULL, 0, B, n_q, Hq, Hkv,
               d, cap, causal, scale, out);
}

int fdo_gather(const uint16_t *q, const int64_t *q_strides,
               const void *k, const int64_t *k_strides,
               const void *v, const int64_t *v_strides, int kv_int8,
               const float *k_scale, const float *v_scale,
               const int64_t *scale_strides, const int32_t *idx, int64_t K,
               int B, int n_q, int Hq, int Hkv, int d, int64_t cap,
               double scale, double *out)
{
    kv_src src = {k, v, kv_int8, k_strides, v_strides, k_scale, v_scale,
                  scale_strides};
    return run(1, q, q_strides, &src, NULL, idx, NULL, K, B, n_q, Hq, Hkv, d, cap,
               0, scale, out);
}

/* Index gather with one additive fp32 bias per list entry, bias [B, n_q, K]
 * contiguous, aligned with idx. */
int fdo_gather_bias(const uint16_t *q, const int64_t *q_strides,
                    const void *k, const int64_t *k_strides,
                    const void *v, const int64_t *v_strides, int kv_int8,
                    const float *k_scale, const float *v_scale,
                    const int64_t *scale_strides, const int32_t *idx,
                    const float *bias, int64_t K, int B, int n_q, int Hq,
                    int Hkv, int d, int64_t cap, double scale, double *out)
{
    kv_src src = {k, v, kv_int8, k_strides, v_strides, k_scale, v_scale,
                  scale_strides};
    return run(1, q, q_strides, &src, NULL, idx, bias, K, B, n_q, Hq, Hkv, d,
               cap, 0, scale, out);
}

void fdo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int fdo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
