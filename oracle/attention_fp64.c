/*
 * fp64 full-softmax attention -- the CPU oracle for the attention outputs.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code with the CUDA path.
 *
 * What it computes (the plain definition, no blocking or online steps):
 *   "From Ring Attention to DeepSpeed Ulysses to USP" (jsqmd.com/news/734632),
 *   §2 "The quadratic curse of attention":
 *       Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
 *   restricted, per query, to the keys the causal mask allows
 *   (same article, §3.4: token t sees tokens t' <= t), and the
 *   log-sum-exp of the scores in natural log, the quantity the LSE merge of
 *   §6.3 combines.
 *
 * For every query row iq and head h:
 *     s[ik] = scale * sum_e q[iq,h,e] * k[ik,h,e]       for each allowed key ik
 *     m     = max_ik s[ik]
 *     O     = sum_ik exp(s[ik] - m) v[ik,h,:] / sum_ik exp(s[ik] - m)
 *     LSE   = m + log(sum_ik exp(s[ik] - m))
 * A key is allowed when the call is non-causal, or when its global position
 * is not after the query's.  A row with no allowed key gets LSE = -inf, O = 0.
 *
 * Grouped-query attention (same article, §5.3 on GQA, where K and V have
 * fewer heads than Q): with Hkv key/value heads, query head h reads key/value
 * head h / (H / Hkv); Hkv = H is ordinary multi-head attention.
 *
 * Packed variable-length sequences (same article, §6 and §8: Megatron's
 * varlen kernel, and variable-length support as a ring weak spot): when
 * segment ids are given, a key is allowed only if it belongs to the query's
 * own sequence (and, causal, is not after it).
 *
 * Inputs are bf16 bit patterns; each is widened to float exactly (bf16 is the
 * top half of an IEEE float) and every product and sum is taken in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static inline double bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/*
 * q:    [nq, H, d] bf16 bits, row iq at q + iq*q_stride (q_stride in elements)
 * k, v: [nk, Hkv, d] bf16 bits, row ik at k + ik*kv_stride
 * q_pos[nq], k_pos[nk]: global token positions (used only when causal != 0)
 * q_seg[nq], k_seg[nk]: sequence ids of packed sequences, or both NULL
 * o:    [nq, H, d] double;  lse: [nq, H] double
 * Returns 0, -1 when a scratch allocation fails, -2 when Hkv does not divide H.
 */
int oracle_attention_fp64(const uint16_t *q, int64_t q_stride, const int64_t *q_pos, int64_t nq,
                          const uint16_t *k, const uint16_t *v, int64_t kv_stride,
                          const int64_t *k_pos, int64_t nk,
                          const int64_t *q_seg, const int64_t *k_seg,
                          int H, int Hkv, int d, double scale, int causal,
                          double *o, double *lse, int nthreads) {
    int failed = 0;
    if (Hkv <= 0 || H % Hkv != 0) return -2;
    const int group = H / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel reduction(| : failed)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        int have_scratch = (s && qrow && acc);
        if (!have_scratch) failed = 1;
        /* every thread reaches the work-sharing loop, scratch or not */
#pragma omp for schedule(dynamic, 4)
            for (int64_t row = 0; row < nq * (int64_t)H; ++row) {
                if (!have_scratch) continue;
                int64_t iq = row / H;
                int h = (int)(row % H);
                const uint16_t *qp = q + iq * q_stride + (int64_t)h * d;
                for (int e = 0; e < d; ++e) qrow[e] = bf16_to_double(qp[e]);

                /* every allowed score, then the max */
                double m = -INFINITY;
                int64_t n_allowed = 0;
                for (int64_t ik = 0; ik < nk; ++ik) {
                    if (causal && k_pos[ik] > q_pos[iq]) { s[ik] = -INFINITY; continue; }
                    if (q_seg && k_seg[ik] != q_seg[iq]) { s[ik] = -INFINITY; continue; }
                    const uint16_t *kp = k + ik * kv_stride + (int64_t)(h / group) * d;
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e) dot += qrow[e] * bf16_to_double(kp[e]);
                    s[ik] = scale * dot;
                    if (s[ik] > m) m = s[ik];
                    ++n_allowed;
                }
                double *orow = o + (iq * (int64_t)H + h) * d;
                if (n_allowed == 0) {
                    for (int e = 0; e < d; ++e) orow[e] = 0.0;
                    lse[iq * (int64_t)H + h] = -INFINITY;
                    continue;
                }
                /* normaliser and weighted sum of V */
                double l = 0.0;
                for (int e = 0; e < d; ++e) acc[e] = 0.0;
                for (int64_t ik = 0; ik < nk; ++ik) {
                    if (s[ik] == -INFINITY) continue;
                    double p = exp(s[ik] - m);
                    l += p;
                    const uint16_t *vp = v + ik * kv_stride + (int64_t)(h / group) * d;
                    for (int e = 0; e < d; ++e) acc[e] += p * bf16_to_double(vp[e]);
                }
                for (int e = 0; e < d; ++e) orow[e] = acc[e] / l;
                lse[iq * (int64_t)H + h] = m + log(l);
            }
        free(s);
        free(qrow);
        free(acc);
    }
    return failed ? -1 : 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
