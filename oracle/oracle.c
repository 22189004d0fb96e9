/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.  A plain, slow, single-threaded CPU
 * restatement of one decode step of a Llama-style decoder, used to check the
 * CUDA megakernel.  Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline leg may load it; the CUDA library never does, and this file
 * shares no code, header, table or helper with it.
 *
 * What the pages fix.  « 2 · Définition et généalogie », §2.1 defines a
 * megakernel as one persistent launch that runs a whole model forward pass;
 * §2.6 ("Le dispatch d'instructions") names its instructions RMSNORM_QKV_ROPE,
 * ATTENTION and O_PROJ, and « Résumé exécutif » ("Le problème") places it on
 * batch-1 decode of Llama-1B.  The pages give no formula for any of these
 * operations.  Every function below therefore restates the standard Llama
 * decoder definition (RMSNorm, rotate-half RoPE, grouped-query attention,
 * SwiGLU MLP, tied or separate LM head), each a reading of the pages where
 * they leave the formula open.
 *
 * Precision: every intermediate is an IEEE double.  Weights and the KV cache
 * are bf16 (their storage type); a key or value written to the cache is
 * rounded to bf16 (round to nearest even) and read back rounded, as the
 * storage type dictates.  The FP8 form of the weights (« Résumé exécutif »,
 * "Les six leviers", names lower precision as a lever but no format) is read
 * as E4M3 codes with one float scale per output row; or_quantize_rows
 * derives it from the bf16 weights and or_matvec_q8 multiplies with it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

/* bf16 bit pattern -> double (exact). */
double or_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* double -> bf16, round to nearest, ties to even, taken directly from the
   double (no intermediate float).  bf16 keeps 8 significant bits. */
uint16_t or_bf16_rne(double v) {
  if (v == 0.0) return signbit(v) ? 0x8000 : 0;
  int e;
  double m = frexp(v, &e);          /* v = m * 2^e, 0.5 <= |m| < 1 */
  double r = nearbyint(m * 256.0);  /* 8 significant bits; default mode = nearest-even */
  double q = ldexp(r, e - 8);
  float f = (float)q;               /* exact: q has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* RMSNorm (standard Llama): y_i = x_i / sqrt(mean_j x_j^2 + eps) * g_i. */
void or_rmsnorm(int n, const double *x, const uint16_t *g, double eps, double *y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * r * or_bf16_to_double(g[i]);
}

/* y = W x for W [M][K] bf16, row-major (PyTorch Linear layout [out, in]). */
void or_matvec(int M, int K, const uint16_t *W, const double *x, double *y) {
  for (int r = 0; r < M; ++r) {
    const uint16_t *w = W + (size_t)r * K;
    double acc = 0.0;
    for (int k = 0; k < K; ++k) acc += or_bf16_to_double(w[k]) * x[k];
    y[r] = acc;
  }
}

/* FP8 E4M3 (the OCP 8-bit floating-point format, variant without
   infinities): sign, 4 exponent bits with bias 7, 3 mantissa bits.  Exponent
   field 0 holds the subnormals m/8 * 2^-6; fields 1..15 hold
   (1 + m/8) * 2^(e-7), except field 15 with mantissa 7, which is NaN, so the
   largest finite magnitude is 1.75 * 2^8 = 448.  Code -> value, exact. */
double or_e4m3_to_double(uint8_t c) {
  int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double a;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    a = ldexp((double)m, -9);
  else
    a = ldexp(8.0 + (double)m, e - 10);
  return sgn ? -a : a;
}

/* Value -> code: round to nearest, ties to even, magnitudes past the
   largest finite one saturate to +-448 (no NaN is produced for a finite
   input).  The grid spacing is 2^-9 below 2^-6 (subnormals) and 2^(e-3)
   in the binade [2^e, 2^(e+1)). */
uint8_t or_e4m3_rne(double v) {
  uint8_t sgn = signbit(v) ? 0x80 : 0;
  double a = fabs(v);
  if (isnan(v)) return 0x7F;
  if (a >= 448.0) return sgn | 0x7E;
  if (a < ldexp(1.0, -6)) {
    double q = nearbyint(ldexp(a, 9)); /* multiples of 2^-9; 8 -> smallest normal */
    return sgn | (uint8_t)q;
  }
  int E;
  frexp(a, &E);           /* a = f 2^E, 0.5 <= f < 1: binade e = E - 1 */
  int e = E - 1;
  double q = nearbyint(ldexp(a, 3 - e)); /* 8 .. 16 */
  if (q >= 16.0) {
    q = 8.0;
    e += 1;
  }
  return sgn | (uint8_t)(((e + 7) << 3) | ((int)q - 8));
}

/* Per-row scaled FP8 quantisation of W [M][K] (bf16): scale_r = amax_r / 448
   in float (1 when the row is zero), code_rk = e4m3(w_rk / scale_r) with the
   division in float, so the largest magnitude of each row maps to +-448. */
void or_quantize_rows(int M, int K, const uint16_t *W, uint8_t *Q, float *scale) {
  for (int r = 0; r < M; ++r) {
    const uint16_t *w = W + (size_t)r * K;
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) {
      float a = (float)fabs(or_bf16_to_double(w[k]));
      if (a > amax) amax = a;
    }
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    scale[r] = s;
    for (int k = 0; k < K; ++k) {
      float v = (float)or_bf16_to_double(w[k]) / s;
      Q[(size_t)r * K + k] = or_e4m3_rne((double)v);
    }
  }
}

/* y = W x for the FP8 weights W_rk = e4m3(Q_rk) * scale_r. */
void or_matvec_q8(int M, int K, const uint8_t *Q, const float *scale, const double *x,
                  double *y) {
  for (int r = 0; r < M; ++r) {
    const uint8_t *q = Q + (size_t)r * K;
    double acc = 0.0;
    for (int k = 0; k < K; ++k) acc += or_e4m3_to_double(q[k]) * (double)scale[r] * x[k];
    y[r] = acc;
  }
}

/* Rotary position embedding, rotate-half convention (HF Llama): for
   i < d/2 the pair (z_i, z_{i+d/2}) is rotated by the angle
   pos * theta^(-2i/d). */
void or_rope(int d, double pos, double theta, double *z) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double inv = pow(theta, -2.0 * (double)i / (double)d);
    double a = pos * inv;
    double c = cos(a), s = sin(a);
    double u = z[i], w = z[i + half];
    z[i] = u * c - w * s;
    z[i + half] = u * s + w * c;
  }
}

/* SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)). */
double or_silu(double z) { return z / (1.0 + exp(-z)); }

/* One query head against n cached positions (rows of K and V, each d bf16):
   s_j = q.k_j / sqrt(d); p = softmax(s) (max-subtracted); o = sum_j p_j v_j. */
void or_attention(int d, int n, const double *q, const uint16_t *K, const uint16_t *V,
                  double *o) {
  double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int k = 0; k < d; ++k) acc += q[k] * or_bf16_to_double(K[(size_t)j * d + k]);
    s[j] = acc * scale;
    if (s[j] > mx) mx = s[j];
  }
  double den = 0.0;
  for (int j = 0; j < n; ++j) {
    s[j] = exp(s[j] - mx);
    den += s[j];
  }
  for (int k = 0; k < d; ++k) o[k] = 0.0;
  for (int j = 0; j < n; ++j)
    for (int k = 0; k < d; ++k) o[k] += s[j] * or_bf16_to_double(V[(size_t)j * d + k]);
  for (int k = 0; k < d; ++k) o[k] /= den;
  free(s);
}

/* Index of the largest value; ties go to the lowest index. */
int or_argmax(int n, const double *v) {
  int best = 0;
  for (int i = 1; i < n; ++i)
    if (v[i] > v[best]) best = i;
  return best;
}

/* One decode step for B independent sequences.
 *   tokens[b]    token fed at this step
 *   positions[b] its position p; the step writes K/V at p and attends to 0..p
 *   kc, vc       caches [L][B][nkv][max_ctx][d] bf16, updated in place
 *   logits       [B][V] doubles
 * Per sequence: x = E[t]; per layer: y = RMSNorm(x) g1; q,k,v = W{q,k,v} y;
 * RoPE on q and k at p; store bf16(k), bf16(v) at p; for every q head h of
 * group g = h / (nq/nkv): o_h = attention(q_h, K[g][0..p], V[g][0..p]);
 * x += Wo concat(o); y = RMSNorm(x) g2; x += Wd (silu(Wg y) * (Wu y));
 * finally logits = W_lm (RMSNorm(x) g_f), W_lm = E when tied.  With m->q8
 * every projection (and W_lm) is its FP8 form instead (or_matvec_q8).
 * Returns 0, or -1 on a bad argument. */
/* projection `w` of layer l: bf16, or FP8 codes with row scales `sc` */
#define MV(M_, K_, w, sc, x_, y_)                                              \
  do {                                                                         \
    if (m->q8)                                                                 \
      or_matvec_q8((M_), (K_), m->q8->w[l], m->q8->sc[l], (x_), (y_));         \
    else                                                                       \
      or_matvec((M_), (K_), m->w[l], (x_), (y_));                              \
  } while (0)

int or_decode_step(const or_model *m, int B, int max_ctx, uint16_t *kc, uint16_t *vc,
                   const int32_t *tokens, const int32_t *positions, double *logits) {
  const int H = m->H, nq = m->nq, nkv = m->nkv, d = m->d, F = m->F, V = m->V, L = m->L;
  const int qpg = nq / nkv;
  if (nq % nkv != 0 || d % 2 != 0) return -1;
  double *x = (double *)malloc(sizeof(double) * H);
  double *y = (double *)malloc(sizeof(double) * H);
  double *q = (double *)malloc(sizeof(double) * (size_t)nq * d);
  double *k = (double *)malloc(sizeof(double) * (size_t)nkv * d);
  double *v = (double *)malloc(sizeof(double) * (size_t)nkv * d);
  double *o = (double *)malloc(sizeof(double) * (size_t)nq * d);
  double *t = (double *)malloc(sizeof(double) * (size_t)(H > F ? H : F));
  double *gt = (double *)malloc(sizeof(double) * F);
  double *up = (double *)malloc(sizeof(double) * F);
  int rc = 0;
  for (int b = 0; b < B && rc == 0; ++b) {
    int tok = tokens[b], p = positions[b];
    if (tok < 0 || tok >= V || p < 0 || p >= max_ctx) {
      rc = -1;
      break;
    }
    for (int i = 0; i < H; ++i) x[i] = or_bf16_to_double(m->embed[(size_t)tok * H + i]);
    for (int l = 0; l < L; ++l) {
      or_rmsnorm(H, x, m->attn_norm[l], m->eps, y);
      MV(nq * d, H, wq, sq, y, q);
      MV(nkv * d, H, wk, sk, y, k);
      MV(nkv * d, H, wv, sv, y, v);
      for (int h = 0; h < nq; ++h) or_rope(d, (double)p, m->theta, q + (size_t)h * d);
      for (int g = 0; g < nkv; ++g) or_rope(d, (double)p, m->theta, k + (size_t)g * d);
      for (int g = 0; g < nkv; ++g) {
        size_t base = ((((size_t)l * B + b) * nkv + g) * max_ctx + p) * d;
        for (int i = 0; i < d; ++i) {
          kc[base + i] = or_bf16_rne(k[(size_t)g * d + i]);
          vc[base + i] = or_bf16_rne(v[(size_t)g * d + i]);
        }
      }
      for (int h = 0; h < nq; ++h) {
        int g = h / qpg;
        size_t base = (((size_t)l * B + b) * nkv + g) * (size_t)max_ctx * d;
        or_attention(d, p + 1, q + (size_t)h * d, kc + base, vc + base, o + (size_t)h * d);
      }
      MV(H, nq * d, wo, so, o, t);
      for (int i = 0; i < H; ++i) x[i] += t[i];
      or_rmsnorm(H, x, m->mlp_norm[l], m->eps, y);
      MV(F, H, w_gate, s_gate, y, gt);
      MV(F, H, w_up, s_up, y, up);
      for (int i = 0; i < F; ++i) gt[i] = or_silu(gt[i]) * up[i];
      MV(H, F, w_down, s_down, gt, t);
      for (int i = 0; i < H; ++i) x[i] += t[i];
    }
    or_rmsnorm(H, x, m->final_norm, m->eps, y);
    if (m->q8)
      or_matvec_q8(V, H, m->q8->lm, m->q8->s_lm, y, logits + (size_t)b * V);
    else
      or_matvec(V, H, m->lm_head ? m->lm_head : m->embed, y, logits + (size_t)b * V);
  }
  free(x);
  free(y);
  free(q);
  free(k);
  free(v);
  free(o);
  free(t);
  free(gt);
  free(up);
  return rc;
}
