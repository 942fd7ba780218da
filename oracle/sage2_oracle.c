/*
 * sage2_oracle.c -- plain, slow CPU oracle for the SageAttention2 quantized
 * exact-attention forward pass.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library. It shares no
 * code with the CUDA library: no headers, helpers, tables or constants.
 *
 * Sources (web pages on SageAttention2, Zhang et al., ICML 2025):
 *   [P2]  "SageAttention2 and Fast Exact INT4 Attention" visual companion
 *         (podcast.do-not-panic.com), sections "Visual Thesis",
 *         "Numerical Repair Stack", "Channel Outlier Smoothing",
 *         "Per-Thread INT4 Geometry".
 *   [P3]  "SageAttention2: Efficient Attention with Thorough Outlier Smoothing
 *         and Per-thread INT4 Quantization" research note
 *         (phantomic12.github.io), the three-component summary.
 *   [P4]  PMLR v267 zhang25ae, Abstract.
 *
 * Two modes:
 *   Mode E  (oracle_attention_exact): textbook softmax(Q K^T * scale) V in
 *           FP64 -- the exact attention rule, which the method keeps
 *           unchanged ([P2] opening paragraph; [P4] Abstract).
 *   Mode Q  (oracle_attention_emulated): the quantized pipeline step by step:
 *           K channel-mean smoothing, Q block-mean smoothing with the
 *           Delta-S logit correction ([P3] component 1, [P4] Abstract,
 *           [P2] Visual Thesis, the numerical-patch panel), INT4-grid codes
 *           with one scale per thread-owned group ([P3] component 2,
 *           [P2] Per-Thread INT4 Geometry), P~ and V in FP8 e4m3
 *           ([P4] Abstract), and two-level accumulation of P~V: a fresh
 *           partial per KV block folded into an FP32 accumulator
 *           ([P3] component 3, [P2] Numerical Repair Stack).
 *
 * The pages give no equations, group shapes, rounding modes or constants.
 * Each reading taken here is marked [R] and listed with its reason in the
 * repository's design notes. Where floating point decides an integer (an
 * INT4 code, an e4m3 code of P~) this oracle takes the decision in FP32
 * with the operation order spelled out below, because the kernel takes it in
 * FP32; everything else is FP64.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fno-fast-math -shared -fPIC.
 * -ffp-contract=off matters: no multiply-add may be fused unless written
 * as fmaf() below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define O_F16 0
#define O_BF16 1

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 1024), e - 25);
  return s ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t h) {
  int s = h >> 15, e = (h >> 7) & 255, m = h & 127;
  double v;
  if (e == 0)
    v = ldexp((double)m, -133);
  else if (e == 255)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 128), e - 134);
  return s ? -v : v;
}

static double in_val(const uint16_t *p, size_t i, int dtype) {
  return dtype == O_BF16 ? oracle_bf16_to_f64(p[i]) : oracle_f16_to_f64(p[i]);
}

/* Decode a whole fp16/bf16 tensor of n elements to FP64 (exact). */
static double *decode_all(const uint16_t *p, size_t n, int dtype) {
  double *x = (double *)malloc(sizeof(double) * (n ? n : 1));
  for (size_t i = 0; i < n; i++) x[i] = in_val(p, i, dtype);
  return x;
}

/* Round x to a binary format with p significand bits (hidden bit included),
 * smallest normal exponent emin and largest finite magnitude maxv; round to
 * nearest, ties to even. Beyond maxv: saturate (sat=1) or infinity. */
static double round_to_format(double x, int p, int emin, double maxv, int sat) {
  if (x != x || x == 0.0 || isinf(x)) {
    if (isinf(x) && sat) return copysign(maxv, x);
    return x;
  }
  double ax = fabs(x);
  int e2;
  (void)frexp(ax, &e2); /* ax = f * 2^e2 with f in [0.5, 1) */
  int lead = e2 - 1;    /* weight of the leading bit */
  if (lead < emin) lead = emin;
  double quantum = ldexp(1.0, lead - (p - 1));
  double r = nearbyint(ax / quantum) * quantum; /* default mode: ties-to-even */
  if (r > maxv) r = sat ? maxv : INFINITY;
  return copysign(r, x);
}

/* OCP 8-bit floating point, E4M3 ("fn" variant): bias 7, 3 fraction bits,
 * subnormal step 2^-9, largest finite 448, no infinities, one NaN pattern
 * per sign (S.1111.111). Encoding rounds to nearest-even and saturates to
 * +-448 ([P4] Abstract: P~ and V in FP8; the variant is the reading [R]). */
uint8_t oracle_e4m3_encode(double x) {
  if (x != x) return 0x7F;
  double r = round_to_format(x, 4, -6, 448.0, 1);
  uint8_t s = signbit(r) ? 0x80 : 0x00;
  double a = fabs(r);
  if (a == 0.0) return s;
  int e2;
  (void)frexp(a, &e2);
  int lead = e2 - 1;
  if (lead < -6) return (uint8_t)(s | (int)(a * 512.0)); /* subnormal: m * 2^-9 */
  int mant = (int)(ldexp(a, -lead) * 8.0) - 8;           /* a = (1 + m/8) 2^lead */
  return (uint8_t)(s | ((lead + 7) << 3) | mant);
}

double oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 | m), e - 10);
  return s ? -v : v;
}

/* Round FP64 results to the output dtype (fp16 or bf16), nearest-even. */
void oracle_round_output(const double *x, size_t n, int dtype, uint16_t *out) {
  for (size_t i = 0; i < n; i++) {
    double r;
    uint16_t bits;
    if (dtype == O_BF16) {
      r = round_to_format(x[i], 8, -126, 3.3895313892515355e38, 0);
      float f = (float)r; /* exact: r has 8 significant bits */
      uint32_t u;
      memcpy(&u, &f, 4);
      bits = (uint16_t)(u >> 16);
    } else {
      r = round_to_format(x[i], 11, -14, 65504.0, 0);
      uint16_t s = signbit(r) ? 0x8000 : 0;
      double a = fabs(r);
      if (isinf(a)) {
        bits = s | 0x7C00;
      } else if (a != a) {
        bits = 0x7E00;
      } else if (a == 0.0) {
        bits = s;
      } else {
        int e2;
        (void)frexp(a, &e2);
        int lead = e2 - 1;
        if (lead < -14)
          bits = (uint16_t)(s | (int)ldexp(a, 24));
        else
          bits = (uint16_t)(s | ((lead + 15) << 10) | ((int)ldexp(a, 10 - lead) - 1024));
      }
    }
    out[i] = bits;
  }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Shapes                                                                    */
/* ------------------------------------------------------------------------ */
/* Tensors are token-major and packed over the batch: Q is [total_q][Hq][D0],
 * K and V are [total_kv][Hkv][D0]; sequence b owns tokens cu[b] .. cu[b+1]-1.
 * Dp is the padded head dim (64 or 128; [P2] Visual Thesis constraint panel);
 * padded channels hold zero. */

static inline size_t tix(int tok, int h, int H, int D) { return ((size_t)tok * H + h) * D; }

/* Causal mask, bottom-right aligned [R]: key j is visible to query i of a
 * sequence with lengths (nq, nkv) iff j <= i + nkv - nq. */
static inline int visible(int causal, int i, int j, int nq, int nkv) {
  return !causal || j <= i + (nkv - nq);
}

/* ------------------------------------------------------------------------ */
/* Mode E: exact attention                                                   */
/* ------------------------------------------------------------------------ */
/* out[total_q][Hq][D0] (FP64). units: n_units triples (b, hq, qblock of bq
 * rows); n_units < 0 computes every row. Rows with no visible key are 0. */
void oracle_attention_exact(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                            int B, const int *cu_q, const int *cu_kv, int Hq, int Hkv, int D0,
                            int causal, float sm_scale, int bq, const int *units, int n_units,
                            double *out) {
  const int g = Hq / Hkv;
  double scale = (double)(sm_scale > 0.f ? sm_scale : (float)(1.0 / sqrt((double)D0)));
  int max_nq = 0;
  for (int b = 0; b < B; b++)
    if (cu_q[b + 1] - cu_q[b] > max_nq) max_nq = cu_q[b + 1] - cu_q[b];
  int nqb = (max_nq + bq - 1) / bq;
  long total_units = n_units >= 0 ? n_units : (long)B * Hq * nqb;
  double *qd = decode_all(q, (size_t)cu_q[B] * Hq * D0, dtype);
  double *kd = decode_all(k, (size_t)cu_kv[B] * Hkv * D0, dtype);
  double *vd = decode_all(v, (size_t)cu_kv[B] * Hkv * D0, dtype);

#pragma omp parallel for schedule(dynamic, 1)
  for (long u = 0; u < total_units; u++) {
    int b, h, qb;
    if (n_units >= 0) {
      b = units[3 * u];
      h = units[3 * u + 1];
      qb = units[3 * u + 2];
    } else {
      b = (int)(u / ((long)Hq * nqb));
      h = (int)((u / nqb) % Hq);
      qb = (int)(u % nqb);
    }
    const int nq = cu_q[b + 1] - cu_q[b], nkv = cu_kv[b + 1] - cu_kv[b];
    const int hk = h / g;
    double *s = (double *)malloc(sizeof(double) * (nkv > 0 ? nkv : 1));
    for (int i = qb * bq; i < nq && i < (qb + 1) * bq; i++) {
      const size_t qo = tix(cu_q[b] + i, h, Hq, D0);
      const double *qi = qd + qo;
      double m = -INFINITY;
      for (int j = 0; j < nkv; j++) {
        if (!visible(causal, i, j, nq, nkv)) {
          s[j] = -INFINITY;
          continue;
        }
        const double *kj = kd + tix(cu_kv[b] + j, hk, Hkv, D0);
        double acc = 0.0;
        for (int d = 0; d < D0; d++) acc += qi[d] * kj[d];
        s[j] = acc * scale;
        if (s[j] > m) m = s[j];
      }
      double *o = out + qo;
      for (int d = 0; d < D0; d++) o[d] = 0.0;
      if (m == -INFINITY) continue;
      double l = 0.0;
      for (int j = 0; j < nkv; j++) {
        if (s[j] == -INFINITY) continue;
        double p = exp(s[j] - m);
        l += p;
        const double *vj = vd + tix(cu_kv[b] + j, hk, Hkv, D0);
        for (int d = 0; d < D0; d++) o[d] += p * vj[d];
      }
      for (int d = 0; d < D0; d++) o[d] /= l;
    }
    free(s);
  }
  free(qd);
  free(kd);
  free(vd);
}

/* ------------------------------------------------------------------------ */
/* Mode Q, step 1: K channel means and V channel absolute maxima             */
/* ------------------------------------------------------------------------ */
/* Per (batch, kv head, channel) [R: per-head channel mean, per-channel V]:
 *   kmean = fl32( (sum_n K[n,d]) / nkv ),  the sum carried in FP64 (exact for
 *           fp16/bf16 data whose exponent spread fits 53 bits),
 *   vamax = max_n |V[n,d]|.
 * kmean, vamax: [B][Hkv][Dp]; padded channels and empty sequences give 0. */
void oracle_kv_stats(const uint16_t *k, const uint16_t *v, int dtype, int B, const int *cu_kv,
                     int Hkv, int D0, int Dp, float *kmean, float *vamax) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; b++)
    for (int h = 0; h < Hkv; h++) {
      const int n = cu_kv[b + 1] - cu_kv[b];
      double *sum = (double *)calloc(Dp, sizeof(double));
      double *amax = (double *)calloc(Dp, sizeof(double));
      for (int t = 0; t < n; t++) /* tokens in order: the FP64 sum is sequential */
        for (int d = 0; d < D0; d++) {
          const size_t o = tix(cu_kv[b] + t, h, Hkv, D0) + d;
          sum[d] += in_val(k, o, dtype);
          double a = fabs(in_val(v, o, dtype));
          if (a > amax[d]) amax[d] = a;
        }
      for (int d = 0; d < Dp; d++) {
        size_t o = ((size_t)b * Hkv + h) * Dp + d;
        kmean[o] = n > 0 ? (float)(sum[d] / (double)n) : 0.f;
        vamax[o] = (float)amax[d]; /* exact: amax is an fp16/bf16 value */
      }
      free(sum);
      free(amax);
    }
}

/* ------------------------------------------------------------------------ */
/* Symmetric integer-grid quantizer [R]                                      */
/* ------------------------------------------------------------------------ */
/* One group of n FP32 values (already smoothed), stride-addressed, onto the
 * grid [-G, G] (G = qmax):
 *   a = max |x|;  a == 0 -> codes 0, scale 0;
 *   inv = fl32(G / a);  code = clamp(round_half_even(fl32(x * inv)), -G, G);
 *   scale = fl32(a / G).
 * G = 7 is the symmetric INT4 grid of the method ([P3] component 2); G = 127
 * the INT8 grid of the SageAttention (v1) path the research note contrasts it
 * with ([P3] opening paragraph). */
static void quant_group(const float *x, const size_t *idx, int n, int qmax, int8_t *codes,
                        float *scale) {
  float a = 0.f;
  for (int i = 0; i < n; i++) {
    float t = fabsf(x[idx[i]]);
    if (t > a) a = t;
  }
  if (a == 0.f) {
    for (int i = 0; i < n; i++) codes[idx[i]] = 0;
    *scale = 0.f;
    return;
  }
  const float g = (float)qmax;
  const float inv = g / a;
  for (int i = 0; i < n; i++) {
    float t = x[idx[i]] * inv;
    float r = nearbyintf(t);
    if (r > g) r = g;
    if (r < -g) r = -g;
    codes[idx[i]] = (int8_t)r;
  }
  *scale = a / g;
}

/* ------------------------------------------------------------------------ */
/* Mode Q, step 2: Q block means and per-row INT4 codes                      */
/* ------------------------------------------------------------------------ */
/* Q is smoothed by the mean of its block of bq consecutive rows of one
 * (sequence, head) ([P3] component 1; [P4] Abstract): over the valid rows
 * of the block, qmean[d] = fl32(sum_rows Q[r,d] / n_rows) (FP64 sum).
 * Q~ = fl32(Q - qmean); each row (token, head) gets one scale over its Dp
 * channels -- one accumulator row per thread in the tensor-memory layout,
 * the analogue of the per-thread scale ([P2] Per-Thread INT4 Geometry) [R].
 * smooth_q = 0 skips the smoothing (qmean = 0; ablation only).
 * q_per_block = 1 replaces the per-row scale by one scale over all valid rows
 * and channels of the block (the coarser per-block granularity that the
 * per-thread scheme improves on, [P3] component 2; ablation only).
 * qmean [B][Hq][nqb_max][Dp], qcodes [total_q][Hq][Dp], sq [total_q][Hq]. */
void oracle_quant_q(const uint16_t *q, int dtype, int B, const int *cu_q, int Hq, int D0, int Dp,
                    int bq, int smooth_q, int q_per_block, int qmax, float *qmean, int8_t *qcodes,
                    float *sq) {
  int max_nq = 0;
  for (int b = 0; b < B; b++)
    if (cu_q[b + 1] - cu_q[b] > max_nq) max_nq = cu_q[b + 1] - cu_q[b];
  const int nqb = (max_nq + bq - 1) / bq;
#pragma omp parallel for collapse(3) schedule(dynamic, 4)
  for (int b = 0; b < B; b++)
    for (int h = 0; h < Hq; h++)
      for (int qb = 0; qb < nqb; qb++) {
        const int nq = cu_q[b + 1] - cu_q[b];
        float *mean = qmean + (((size_t)b * Hq + h) * nqb + qb) * Dp;
        const int r0 = qb * bq, r1 = (qb + 1) * bq < nq ? (qb + 1) * bq : nq;
        if (r1 <= r0) {
          for (int d = 0; d < Dp; d++) mean[d] = 0.f;
          continue;
        }
        const int nr = r1 - r0;
        /* the smoothed block, rows in order; idx addresses it row-major */
        float *xt = (float *)malloc(sizeof(float) * (size_t)nr * Dp);
        size_t *idx = (size_t *)malloc(sizeof(size_t) * (size_t)nr * Dp);
        int8_t *ct = (int8_t *)malloc((size_t)nr * Dp);
        for (int d = 0; d < Dp; d++) {
          double sum = 0.0;
          if (d < D0)
            for (int r = r0; r < r1; r++) sum += in_val(q, tix(cu_q[b] + r, h, Hq, D0) + d, dtype);
          mean[d] = (smooth_q && d < D0) ? (float)(sum / (double)nr) : 0.f;
        }
        for (int r = 0; r < nr; r++) {
          const size_t row = (size_t)(cu_q[b] + r0 + r) * Hq + h;
          for (int d = 0; d < Dp; d++) {
            xt[(size_t)r * Dp + d] = d < D0 ? (float)in_val(q, row * D0 + d, dtype) - mean[d] : 0.f;
            idx[(size_t)r * Dp + d] = (size_t)r * Dp + d;
          }
        }
        if (q_per_block) {
          float sc;
          quant_group(xt, idx, nr * Dp, qmax, ct, &sc);
          for (int r = 0; r < nr; r++) {
            const size_t row = (size_t)(cu_q[b] + r0 + r) * Hq + h;
            memcpy(qcodes + row * Dp, ct + (size_t)r * Dp, Dp);
            sq[row] = sc;
          }
        } else {
          for (int r = 0; r < nr; r++) {
            const size_t row = (size_t)(cu_q[b] + r0 + r) * Hq + h;
            quant_group(xt, idx + (size_t)r * Dp, Dp, qmax, ct, sq + row);
            memcpy(qcodes + row * Dp, ct + (size_t)r * Dp, Dp);
          }
        }
        free(xt);
        free(idx);
        free(ct);
      }
}

/* ------------------------------------------------------------------------ */
/* Mode Q, step 2b: K codes, one scale per gk consecutive tokens             */
/* ------------------------------------------------------------------------ */
/* K~ = fl32(K - kmean) (kmean may be NULL: no smoothing, ablation only).
 * Groups: gk consecutive tokens of one (sequence, kv head) over all Dp
 * channels; each thread of the accumulator-load layout multiplies a gk-column
 * chunk by one constant [R]. kcodes [total_kv][Hkv][Dp]; sk [total_kv][Hkv]
 * holds, for every token, the scale of its group. */
void oracle_quant_k(const uint16_t *k, int dtype, int B, const int *cu_kv, int Hkv, int D0, int Dp,
                    int gk, const float *kmean, int qmax, int8_t *kcodes, float *sk) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; b++)
    for (int h = 0; h < Hkv; h++) {
      const int n = cu_kv[b + 1] - cu_kv[b];
      const float *mu = kmean ? kmean + ((size_t)b * Hkv + h) * Dp : NULL;
      float *xt = (float *)malloc(sizeof(float) * (size_t)gk * Dp);
      int8_t *ct = (int8_t *)malloc((size_t)gk * Dp);
      size_t *idx = (size_t *)malloc(sizeof(size_t) * (size_t)gk * Dp);
      for (int t0 = 0; t0 < n; t0 += gk) {
        const int cnt = t0 + gk <= n ? gk : n - t0;
        for (int t = 0; t < cnt; t++)
          for (int d = 0; d < Dp; d++) {
            float x = d < D0 ? (float)in_val(k, tix(cu_kv[b] + t0 + t, h, Hkv, D0) + d, dtype) : 0.f;
            xt[t * Dp + d] = (d < D0 && mu) ? x - mu[d] : x;
            idx[t * Dp + d] = (size_t)t * Dp + d;
          }
        float sc;
        quant_group(xt, idx, cnt * Dp, qmax, ct, &sc);
        for (int t = 0; t < cnt; t++) {
          const size_t row = (size_t)(cu_kv[b] + t0 + t) * Hkv + h;
          memcpy(kcodes + row * Dp, ct + (size_t)t * Dp, Dp);
          sk[row] = sc;
        }
      }
      free(xt);
      free(ct);
      free(idx);
    }
}

/* ------------------------------------------------------------------------ */
/* Mode Q, step 2d: V to FP8 e4m3 with one scale per channel [R]             */
/* ------------------------------------------------------------------------ */
/* inv = fl32(448 / vamax[d]); code = e4m3(fl32(V * inv)); sv = fl32(vamax/448).
 * vamax == 0 gives codes 0 and scale 0. vcodes [total_kv][Hkv][Dp] (e4m3
 * bytes), sv [B][Hkv][Dp]. */
void oracle_quant_v(const uint16_t *v, int dtype, int B, const int *cu_kv, int Hkv, int D0, int Dp,
                    const float *vamax, uint8_t *vcodes, float *sv) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; b++)
    for (int h = 0; h < Hkv; h++) {
      const float *a = vamax + ((size_t)b * Hkv + h) * Dp;
      float inv[128];
      for (int d = 0; d < Dp; d++) {
        inv[d] = a[d] > 0.f ? 448.0f / a[d] : 0.f;
        sv[((size_t)b * Hkv + h) * Dp + d] = a[d] > 0.f ? a[d] / 448.0f : 0.f;
      }
      for (int t = cu_kv[b]; t < cu_kv[b + 1]; t++) {
        const size_t row = (size_t)t * Hkv + h;
        for (int d = 0; d < Dp; d++) {
          float x = (d < D0 && a[d] > 0.f) ? (float)in_val(v, row * D0 + d, dtype) * inv[d] : 0.f;
          vcodes[row * Dp + d] = oracle_e4m3_encode((double)x);
        }
      }
    }
}

/* ------------------------------------------------------------------------ */
/* Mode Q, step 2c: Delta-S for one (sequence, q head, q block)             */
/* ------------------------------------------------------------------------ */
/* Q = Q~ + qmean gives Q K^T = Q~ K^T + qmean K^T; the second term is the
 * correction kept for the logits ([P2] Visual Thesis, numerical-patch panel;
 * [P3] component 1). With K smoothed, K^T may be replaced by K~^T: the
 * difference qmean . kmean is the same for every key, and softmax rows do not
 * change under a per-row constant. Computed from the unquantized smoothed
 * K~ = fl32(K - kmean) in full precision [R]: every product of two FP32
 * values is exact in FP64 and the sum over the channels is carried in FP64,
 * then rounded once to FP32, which gives the correctly rounded exact dot
 * product unless it lies within about 2^-46 (relative) of an FP32 rounding
 * midpoint. The e4m3 codes of P~ depend on it only through the rounding of
 * 448 P: a Delta-S a few ulp away moves a code only where 448 P sits at a
 * midpoint, the case the P~ comparisons already account for.
 * out[j] for the nkv keys of sequence b. */
void oracle_delta_s(const uint16_t *k, int dtype, const int *cu_kv, int b, int Hkv, int hk, int D0,
                    int Dp, const float *kmean, const float *qbar, float *out) {
  const int n = cu_kv[b + 1] - cu_kv[b];
  const float *mu = kmean ? kmean + ((size_t)b * Hkv + hk) * Dp : NULL;
  for (int j = 0; j < n; j++) {
    double acc = 0.0;
    for (int d = 0; d < D0; d++) {
      float x = (float)in_val(k, tix(cu_kv[b] + j, hk, Hkv, D0) + d, dtype);
      if (mu) x = x - mu[d]; /* K~ = fl32(K - kmean) */
      acc += (double)qbar[d] * (double)x;
    }
    out[j] = (float)acc;
  }
}

/* ------------------------------------------------------------------------ */
/* Mode Q: the full quantized pipeline                                       */
/* ------------------------------------------------------------------------ */
/* Per (sequence b, q head h, q block qb) unit, in this order [R]:
 *   c   = fl32(log2(e) * sm_scale);  L = fl32(log2(448));
 *   sqc = fl32(sq[i] * c) per row;   dsc[j] = fl32(DeltaS[j] * c);
 *   for each KV tile of bkv keys, in increasing order:
 *     A[i,j]  = sum_d qcode[i,d] * kcode[j,d]      (exact integer)
 *     S'[i,j] = fma(A, fl32(sqc[i] * sk[j]), dsc[j])   in FP32 (log2 units),
 *               -inf where key j is not visible to query i
 *     m_new   = max(m, max_j S');   m448 = fl32(m_new - L)
 *     P448    = fl32(2^(fl32(S' - m448)))    (= 448 P, P = 2^(S' - m_new))
 *     P~      = e4m3(P448)                   (static scale 448 [R])
 *     alpha   = 2^(m - m_new)  (FP64);  l = alpha l + sum_j P448  (FP64;
 *               l accumulates the unquantized P [R])
 *     R[i,d]  = fl32(sum_j P~[i,j] * vcode[j,d])   (the fresh per-tile
 *               partial of the two-level scheme; the FP64 sum is exact)
 *     O[i,d]  = fl32(alpha O[i,d] + R[i,d])         (FP32 fold)
 *   out[i,d] = O[i,d] * sv[d] / l   (FP64; 0 when no key is visible).
 * Flags (ablations; smooth_q = smooth_k = 1, q_per_block = acc_bits = 0,
 * qmax = 7 is the method): smooth_q, smooth_k; q_per_block (one Q scale per
 * block, see oracle_quant_q; with gk = bkv K gets one scale per block too);
 * qmax the integer grid of the Q and K codes (127: the INT8 path of the
 * SageAttention (v1) variant, run with smooth_q = 0 and per-block scales:
 * INT8 with K smoothing, [P3] opening paragraph and its comparison of the two
 * versions); acc_bits > 0 replaces the two-level fold by one-level accumulation whose accumulator is
 * rounded to acc_bits significand bits after every 32-key MMA step (an
 * emulation of a reduced-precision FP8 MMA accumulator).
 * out [total_q][Hq][D0] (FP64, rows outside `units` untouched).
 * dump_p448 (may be NULL; then `units` names exactly one unit): receives the
 * fl32 P448 of every (row, key) of KV tile dump_kt of that unit, [bq][bkv]
 * row-major; keys that are not visible are left untouched (test hook). */
static double round_bits(double x, int bits) {
  if (x == 0.0 || bits <= 0) return x;
  int e2;
  (void)frexp(x, &e2);
  double q = ldexp(1.0, e2 - bits);
  return nearbyint(x / q) * q;
}

void oracle_attention_emulated(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                               int B, const int *cu_q, const int *cu_kv, int Hq, int Hkv, int D0,
                               int Dp, int causal, float sm_scale, int bq, int bkv, int gk,
                               int smooth_q, int smooth_k, int q_per_block, int qmax,
                               int acc_bits, const int *units, int n_units, double *out,
                               int dump_kt, float *dump_p448) {
  const int g = Hq / Hkv;
  const float scale32 = sm_scale > 0.f ? sm_scale : (float)(1.0 / sqrt((double)D0));
  const float c32 = (float)(1.4426950408889634074 * (double)scale32);
  const float L32 = (float)log2(448.0);
  const size_t tq = (size_t)cu_q[B], tkv = (size_t)cu_kv[B];
  int max_nq = 0;
  for (int b = 0; b < B; b++)
    if (cu_q[b + 1] - cu_q[b] > max_nq) max_nq = cu_q[b + 1] - cu_q[b];
  const int nqb = (max_nq + bq - 1) / bq;

  float *kmean = (float *)calloc((size_t)B * Hkv * Dp, sizeof(float));
  float *vamax = (float *)calloc((size_t)B * Hkv * Dp, sizeof(float));
  float *qmean = (float *)calloc((size_t)B * Hq * (nqb > 0 ? nqb : 1) * Dp, sizeof(float));
  int8_t *qc = (int8_t *)calloc(tq * Hq * Dp + 1, 1);
  float *sq = (float *)calloc(tq * Hq + 1, sizeof(float));
  int8_t *kc = (int8_t *)calloc(tkv * Hkv * Dp + 1, 1);
  float *sk = (float *)calloc(tkv * Hkv + 1, sizeof(float));
  uint8_t *vc = (uint8_t *)calloc(tkv * Hkv * Dp + 1, 1);
  float *sv = (float *)calloc((size_t)B * Hkv * Dp, sizeof(float));

  double e4m3_val[256]; /* value of every e4m3 byte, from the decoder above */
  for (int c = 0; c < 256; c++) e4m3_val[c] = oracle_e4m3_decode((uint8_t)c);
  oracle_kv_stats(k, v, dtype, B, cu_kv, Hkv, D0, Dp, kmean, vamax);
  oracle_quant_q(q, dtype, B, cu_q, Hq, D0, Dp, bq, smooth_q, q_per_block, qmax, qmean, qc, sq);
  oracle_quant_k(k, dtype, B, cu_kv, Hkv, D0, Dp, gk, smooth_k ? kmean : NULL, qmax, kc, sk);
  oracle_quant_v(v, dtype, B, cu_kv, Hkv, D0, Dp, vamax, vc, sv);

  long total_units = n_units >= 0 ? n_units : (long)B * Hq * nqb;
#pragma omp parallel for schedule(dynamic, 1)
  for (long u = 0; u < total_units; u++) {
    int b, h, qb;
    if (n_units >= 0) {
      b = units[3 * u];
      h = units[3 * u + 1];
      qb = units[3 * u + 2];
    } else {
      b = (int)(u / ((long)Hq * nqb));
      h = (int)((u / nqb) % Hq);
      qb = (int)(u % nqb);
    }
    const int nq = cu_q[b + 1] - cu_q[b], nkv = cu_kv[b + 1] - cu_kv[b];
    const int hk = h / g;
    const int r0 = qb * bq, r1 = (qb + 1) * bq < nq ? (qb + 1) * bq : nq;
    if (r1 <= r0) continue;
    const float *qbar = qmean + (((size_t)b * Hq + h) * nqb + qb) * Dp;
    float *dS = (float *)malloc(sizeof(float) * (nkv > 0 ? nkv : 1));
    oracle_delta_s(k, dtype, cu_kv, b, Hkv, hk, D0, Dp, smooth_k ? kmean : NULL, qbar, dS);
    float *sp = (float *)malloc(sizeof(float) * bkv);
    float *O = (float *)malloc(sizeof(float) * Dp);
    double *Oacc = (double *)malloc(sizeof(double) * Dp);
    double *R = (double *)malloc(sizeof(double) * Dp);
    const float *svh = sv + ((size_t)b * Hkv + hk) * Dp;

    for (int i = r0; i < r1; i++) {
      const size_t qrow = (size_t)(cu_q[b] + i) * Hq + h;
      const int8_t *qi = qc + qrow * Dp;
      const float sqc = sq[qrow] * c32;
      float m = -INFINITY;
      double l = 0.0;
      for (int d = 0; d < Dp; d++) {
        O[d] = 0.f;
        Oacc[d] = 0.0;
      }
      for (int t0 = 0; t0 < nkv; t0 += bkv) {
        const int cnt = t0 + bkv <= nkv ? bkv : nkv - t0;
        float mx = -INFINITY;
        for (int jj = 0; jj < cnt; jj++) {
          const int j = t0 + jj;
          if (!visible(causal, i, j, nq, nkv)) {
            sp[jj] = -INFINITY;
            continue;
          }
          const size_t krow = (size_t)(cu_kv[b] + j) * Hkv + hk;
          const int8_t *kj = kc + krow * Dp;
          int32_t A = 0; /* exact: |A| <= qmax^2 * 128 <= 127^2 * 128 */
          for (int d = 0; d < Dp; d++) A += (int32_t)qi[d] * (int32_t)kj[d];
          const float mult = sqc * sk[krow];
          const float dsc = dS[j] * c32;
          sp[jj] = fmaf((float)A, mult, dsc);
          if (sp[jj] > mx) mx = sp[jj];
        }
        const float m_new = mx > m ? mx : m;
        if (m_new == -INFINITY) continue; /* nothing visible yet */
        const double alpha = (m == -INFINITY) ? 0.0 : exp2((double)m - (double)m_new);
        const float m448 = m_new - L32;
        double lsum = 0.0;
        for (int d = 0; d < Dp; d++) R[d] = 0.0;
        if (acc_bits > 0)
          for (int d = 0; d < Dp; d++) Oacc[d] = round_bits(alpha * Oacc[d], acc_bits);
        for (int jj = 0; jj < cnt; jj++) {
          if (sp[jj] != -INFINITY) {
            const float arg = sp[jj] - m448;
            const float p448 = (float)exp2((double)arg);
            if (dump_p448 && t0 / bkv == dump_kt) dump_p448[(size_t)(i - r0) * bkv + jj] = p448;
            lsum += (double)p448;
            const double pt = round_to_format((double)p448, 4, -6, 448.0, 1); /* e4m3 value */
            const uint8_t *vj = vc + ((size_t)(cu_kv[b] + t0 + jj) * Hkv + hk) * Dp;
            if (pt != 0.0)
              for (int d = 0; d < Dp; d++) R[d] += pt * e4m3_val[vj[d]];
          }
          if (acc_bits > 0 && (((jj + 1) & 31) == 0 || jj == cnt - 1))
            for (int d = 0; d < Dp; d++) {
              Oacc[d] = round_bits(Oacc[d] + R[d], acc_bits);
              R[d] = 0.0;
            }
        }
        l = alpha * l + lsum;
        if (acc_bits <= 0)
          for (int d = 0; d < Dp; d++) O[d] = (float)(alpha * (double)O[d] + (double)(float)R[d]);
        m = m_new;
      }
      double *o = out + qrow * D0;
      for (int d = 0; d < D0; d++) {
        double od = acc_bits > 0 ? Oacc[d] : (double)O[d];
        o[d] = l > 0.0 ? od * (double)svh[d] / l : 0.0;
      }
    }
    free(dS);
    free(sp);
    free(O);
    free(Oacc);
    free(R);
  }
  free(kmean);
  free(vamax);
  free(qmean);
  free(qc);
  free(sq);
  free(kc);
  free(sk);
  free(vc);
  free(sv);
}
