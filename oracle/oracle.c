/*
 * ORACLE — test infrastructure only. Nothing on the product path may call it:
 * only the tests, the smoke check and the CPU-baseline leg of the benchmark.
 *
 * A plain, slow CPU restatement of the single-GPU MegaMoE expert path as the
 * DeepGEMM MegaMoE pages describe it:
 *   route (expert counts, prefix offsets, expert-sorted slot permutation)
 *   -> L1 grouped GEMM over [gate | up]            ("MegaMoE on SM100/SM90", sec. 4.1, Linear1 phase)
 *   -> SwiGLU (optional clamp) x top-k weight       ("MEGAMOE_SM90_DESIGN", sec. 10.1, steps 2-3)
 *   -> per-32 amax, UE8M0 scale, E4M3 requantise    (sec. 4.1 "amax, UE8M0 L2 act SF"; sec. 10.1 steps 4-5)
 *   -> L2 grouped GEMM, BF16 per slot row           (sec. 4.1, Linear2 phase; sec. 11.1)
 *   -> per-token FP32 sum of the slot rows -> BF16  (sec. 11.2, combine reduce)
 * Operands are FP8 E4M3 activations and MXFP4 weights (E2M1 + UE8M0 per 32
 * along K), accumulation in FP32 (the design's FP32 accumulator), every sum
 * taken in ascending index order. No blocking, fusion or reordering.
 *
 * Readings where the pages are silent or disagree:
 *  - the top-k weight multiplies the SwiGLU output before the amax (the
 *    kernels' order); the combine is then an unweighted sum;
 *  - the L2-activation scale is UE8M0, one per 32 along I, equal to the
 *    smallest power of two >= amax/448 (so nothing saturates), code 127 for
 *    amax == 0, clamped to [1, 254];
 *  - the E4M3 cast rounds to nearest even and saturates at +-448;
 *  - the clamp is symmetric on both gate and up, before the SiLU;
 *  - W1 rows [0, I) are gate and [I, 2I) are up; E2M1 codes are packed two per
 *    byte with the even K index in the low nibble; E4M3 weights (the FP8
 *    weight variant) are one byte per element; both carry one UE8M0 scale per
 *    32 along K (OCP MX: MXFP4 / MXFP8);
 *  - within one expert, rows are in ascending source-slot order;
 *  - shared experts sit at expert indices E..E+S-1, slot k+s of every token,
 *    with weight 1; a topk_idx of -1 disables its slot.
 *
 * The float-scale FP8 recipe (w_fmt 2; "MEGAMOE_SM90_DESIGN" sec. 5.3 scale
 * application, sec. 10.1 steps 4-5 exact float L2-activation scale, sec. 15.2
 * weight scale layout (E, N/128, K/128)): every weight and activation element
 * is E4M3 with a float32 scale per 128 along K (weights: per 128 x 128 block).
 * Readings: each 128-long K block's partial sum is taken in FP32 over the
 * unscaled E4M3 products, multiplied by (activation scale x weight scale) and
 * added to the FP32 accumulator in ascending block order; the L2-activation
 * scale is one float32 per (row, 128 along I), amax / 448 by one IEEE
 * division (1 when amax is 0), and the E4M3 code is the nearest-even
 * saturating encoding of y / scale.
 *
 * Build with -ffp-contract=off. Defining ORC_MUTANT to a non-zero value plants
 * one deliberate mistake (used only to show that the pin tests catch it).
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif
#define MUT(n) (ORC_MUTANT == (n))

/* ------------------------------------------------------------------ formats */

/* OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent
 * field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity. */
float orc_e4m3_to_float(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  float v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexpf((float)m, -9);
  else v = ldexpf((float)(8 + m), e - 10);
  return s ? -v : v;
}

/* OCP FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit;
 * exponent field 0 is subnormal (m * 0.5). */
float orc_e2m1_to_float(uint8_t c) {
  int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  float v = (e == 0) ? 0.5f * (float)m : ldexpf((float)(2 + m), e - 2);
  return s ? -v : v;
}

/* OCP UE8M0 scale: 2^(b - 127); 0xFF is NaN. */
float orc_ue8m0_to_float(uint8_t b) {
  if (b == 255) return NAN;
  return ldexpf(1.0f, (int)b - 127);
}

/* Nearest E4M3 value, ties to the even code, saturating at +-448: a search over
 * the 127 finite non-negative codes, which are monotone in value. */
uint8_t orc_float_to_e4m3(float v) {
  float a = fabsf(v);
  int c;
  if (a >= 448.0f) {
    c = 126;
  } else {
    int lo = 0, hi = 126; /* invariant: value(lo) <= a < value(hi + 1) */
    while (lo < hi) {
      int mid = (lo + hi + 1) / 2;
      if (orc_e4m3_to_float((uint8_t)mid) <= a) lo = mid;
      else hi = mid - 1;
    }
    c = lo;
    float vlo = orc_e4m3_to_float((uint8_t)c);
    if (vlo != a && c < 126) {
      float vhi = orc_e4m3_to_float((uint8_t)(c + 1));
      float dlo = a - vlo, dhi = vhi - a;
#if MUT(12)
      (void)dhi; /* mistake: truncation toward zero */
#else
      if (dhi < dlo || (dhi == dlo && (c & 1))) c = c + 1;
#endif
    }
  }
  if (c == 0) return 0;
  return (uint8_t)(v < 0.0f ? (c | 0x80) : c);
}

float orc_bf16_to_float(uint16_t h) {
  uint32_t b = (uint32_t)h << 16;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

/* bfloat16 = upper half of the float32 pattern, rounded to nearest even. */
uint16_t orc_float_to_bf16(float v) {
  uint32_t b;
  memcpy(&b, &v, 4);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((b >> 16) | 0x40u);
  uint32_t upper = b >> 16, lower = b & 0xFFFFu;
#if MUT(11)
  (void)lower; /* mistake: truncation */
#else
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
#endif
  return (uint16_t)upper;
}

/* UE8M0 code of the smallest power of two p with amax/448 <= p (amax/448 taken
 * in float32); 127 for amax == 0; clamped to [1, 254]. */
uint8_t orc_requant_code(float amax) {
  if (!(amax > 0.0f)) return 127;
  float r = amax / 448.0f;
  int ex;
  float m = frexpf(r, &ex); /* r = m * 2^ex, 0.5 <= m < 1 */
  int p = (m == 0.5f) ? ex - 1 : ex;
#if MUT(3)
  p = ex - 1; /* mistake: round the scale down */
#endif
  int code = 127 + p;
  if (code < 1) code = 1;
  if (code > 254) code = 254;
  return (uint8_t)code;
}

void orc_decode_e4m3(const uint8_t* in, float* out, long n) { for (long i = 0; i < n; ++i) out[i] = orc_e4m3_to_float(in[i]); }
void orc_decode_e2m1(const uint8_t* in, float* out, long n) { for (long i = 0; i < n; ++i) out[i] = orc_e2m1_to_float(in[i]); }
void orc_decode_ue8m0(const uint8_t* in, float* out, long n) { for (long i = 0; i < n; ++i) out[i] = orc_ue8m0_to_float(in[i]); }
void orc_encode_e4m3(const float* in, uint8_t* out, long n) { for (long i = 0; i < n; ++i) out[i] = orc_float_to_e4m3(in[i]); }
void orc_encode_bf16(const float* in, uint16_t* out, long n) { for (long i = 0; i < n; ++i) out[i] = orc_float_to_bf16(in[i]); }
void orc_requant_codes(const float* amax, uint8_t* out, long n) { for (long i = 0; i < n; ++i) out[i] = orc_requant_code(amax[i]); }

/* E2M1 code of element kk of a packed row (even index in the low nibble). */
static uint8_t orc_nibble(const uint8_t* row, long kk) {
  uint8_t byte = row[kk / 2];
#if MUT(1)
  return (kk & 1) ? (byte & 15) : (byte >> 4); /* mistake: nibble order */
#else
  return (kk & 1) ? (byte >> 4) : (byte & 15);
#endif
}

/* Scale index of element kk: one scale per 32 along K. */
static long orc_sf_index(long kk) {
#if MUT(10)
  return (kk / 128) * 4; /* mistake: per-128 granularity */
#else
  return kk / 32;
#endif
}

/* Element kk of a weight row (format fmt), before its block scale. Rows are
 * K/2 bytes for E2M1 and K bytes for E4M3. */
static float orc_weight(const uint8_t* row, long kk, int fmt) {
#if MUT(13)
  (void)fmt;
  return orc_e2m1_to_float(orc_nibble(row, kk)); /* mistake: every weight read as E2M1 */
#else
  return fmt ? orc_e4m3_to_float(row[kk]) : orc_e2m1_to_float(orc_nibble(row, kk));
#endif
}

/* Bytes per weight row of K elements. */
static long orc_row_bytes(long K, int fmt) { return fmt ? K : K / 2; }

/* ------------------------------------------------------------------ routing */

static int orc_slot_expert(int T, int k, int S, int E, const int32_t* topk_idx, long s, int* bad) {
  int Kp = k + S;
  long t = s / Kp;
  int j = (int)(s % Kp);
  (void)T;
  if (j >= k) return E + (j - k);
  int e = topk_idx[t * k + j];
  if (e == -1) return -1;
  if (e < 0 || e >= E) { ++*bad; return -1; }
  return e;
}

int orc_route(int T, int k, int S, int E, const int32_t* topk_idx,
              int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos) {
  int Ep = E + S, bad = 0;
  long R = (long)T * (k + S);
  for (int e = 0; e < Ep; ++e) counts[e] = 0;
  for (long s = 0; s < R; ++s) {
    int e = orc_slot_expert(T, k, S, E, topk_idx, s, &bad);
    if (e >= 0) counts[e]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < Ep; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)calloc((size_t)Ep + 1, sizeof(int32_t));
  int dummy = 0;
#if MUT(9)
  for (long s = R - 1; s >= 0; --s) { /* mistake: unstable (descending) order */
#else
  for (long s = 0; s < R; ++s) {
#endif
    int e = orc_slot_expert(T, k, S, E, topk_idx, s, &dummy);
    if (e < 0) { pos[s] = -1; continue; }
    int r = offsets[e] + fill[e]++;
    perm[r] = (int32_t)s;
    pos[s] = r;
  }
  free(fill);
  return bad;
}

/* ------------------------------------------------------------------ the path */

typedef struct {
  const orc_dims* d;
  const uint8_t *x, *x_sf, *w1, *w1_sf, *w2, *w2_sf;
  const int32_t* topk_idx;
  const float* topk_w;
  const int32_t* perm;
  int nrows;
  float* acc1;
  uint8_t *q, *qsf;
  uint16_t* z;
  int th, nth;
} orc_job;

/* One pool row: L1, SwiGLU x weight, requantise, L2, BF16. */
static void orc_one_row(const orc_job* J, long r, float* xh, float* a1, float* y, float* qh) {
  const orc_dims* d = J->d;
  const int H = d->H, I = d->I, k = d->k, Kp = d->k + d->S;
  long s = J->perm[r], t = s / Kp;
  int j = (int)(s % Kp);
  int e = (j < k) ? J->topk_idx[t * k + j] : d->E + (j - k);
  float wgt = (j < k) ? J->topk_w[t * k + j] : 1.0f;

  /* dequantised activation row: E4M3 value x UE8M0 scale of its 32-group */
  for (long kk = 0; kk < H; ++kk) {
#if MUT(6)
    xh[kk] = orc_e4m3_to_float(J->x[t * H + kk]); /* mistake: activation scale dropped */
#else
    xh[kk] = orc_e4m3_to_float(J->x[t * H + kk]) * orc_ue8m0_to_float(J->x_sf[t * (H / 32) + orc_sf_index(kk)]);
#endif
  }
  /* L1: acc1[n] = sum_k x[k] * W1[e][n][k], FP32, ascending k */
  for (long n = 0; n < 2L * I; ++n) {
    const uint8_t* wr = J->w1 + ((long)e * 2 * I + n) * orc_row_bytes(H, d->w_fmt);
    const uint8_t* sr = J->w1_sf + ((long)e * 2 * I + n) * (H / 32);
    float acc = 0.0f;
    for (long kk = 0; kk < H; ++kk) {
      float wv = orc_weight(wr, kk, d->w_fmt) * orc_ue8m0_to_float(sr[orc_sf_index(kk)]);
      acc += xh[kk] * wv;
    }
    a1[n] = acc;
  }
  if (J->acc1) memcpy(J->acc1 + r * 2L * I, a1, sizeof(float) * 2 * (size_t)I);

  /* SwiGLU: y = silu(clamp(g)) * clamp(u) * w */
  for (long n = 0; n < I; ++n) {
#if MUT(2)
    float g = a1[I + n], u = a1[n]; /* mistake: gate and up swapped */
#else
    float g = a1[n], u = a1[I + n];
#endif
    if (d->clamp > 0.0f) {
      g = fminf(fmaxf(g, -d->clamp), d->clamp);
      u = fminf(fmaxf(u, -d->clamp), d->clamp);
    }
#if MUT(8)
    float silu = g / (1.0f + expf(g)); /* mistake: sign in the sigmoid */
#else
    float silu = g / (1.0f + expf(-g));
#endif
    float v = silu * u;
#if MUT(4)
    (void)wgt; /* mistake: top-k weight dropped */
#else
    if (!d->weight_in_combine) v = v * wgt;
#endif
    y[n] = v;
  }
  /* requantise per 32 along I: UE8M0 scale, E4M3 element */
  for (long b = 0; b < I / 32; ++b) {
    float amax = 0.0f;
    for (long n = 32 * b; n < 32 * b + 32; ++n) amax = fmaxf(amax, fabsf(y[n]));
    uint8_t code = orc_requant_code(amax);
    float sc = orc_ue8m0_to_float(code);
    for (long n = 32 * b; n < 32 * b + 32; ++n) {
      uint8_t qq = orc_float_to_e4m3(y[n] / sc);
      if (J->q) J->q[r * I + n] = qq;
      qh[n] = orc_e4m3_to_float(qq) * sc;
    }
    if (J->qsf) J->qsf[r * (I / 32) + b] = code;
  }
  /* L2: z[h] = bf16(sum_i q[i] * W2[e][h][i]), FP32, ascending i */
  for (long h = 0; h < H; ++h) {
    const uint8_t* wr = J->w2 + ((long)e * H + h) * orc_row_bytes(I, d->w_fmt);
    const uint8_t* sr = J->w2_sf + ((long)e * H + h) * (I / 32);
    float acc = 0.0f;
    for (long i = 0; i < I; ++i) {
#if MUT(5)
      /* mistake: W2 read transposed ([I][H] instead of [H][I]) */
      long flat = i * H + h;
      const uint8_t* wt = J->w2 + (long)e * H * orc_row_bytes(I, d->w_fmt);
      const uint8_t* st = J->w2_sf + (long)e * H * (I / 32);
      float wv = orc_weight(wt, flat, d->w_fmt) * orc_ue8m0_to_float(st[flat / 32]);
      (void)wr; (void)sr;
#else
      float wv = orc_weight(wr, i, d->w_fmt) * orc_ue8m0_to_float(sr[orc_sf_index(i)]);
#endif
      acc += qh[i] * wv;
    }
    J->z[r * H + h] = orc_float_to_bf16(acc);
  }
}

/* Float scale of a 128-long block: the float32 stored at element i of a
 * float32 array passed as bytes. */
static float orc_f32_at(const uint8_t* base, long i) {
  float v;
  memcpy(&v, base + 4 * i, 4);
  return v;
}

/* One pool row under the float-scale FP8 recipe (w_fmt 2): L1 per 128-K
 * block with float scales, SwiGLU x weight, float per-128 requantise, L2 per
 * 128-K block, BF16. */
static void orc_one_row_f128(const orc_job* J, long r, float* xh, float* a1, float* y, float* qh) {
  const orc_dims* d = J->d;
  const int H = d->H, I = d->I, k = d->k, Kp = d->k + d->S;
  const long HB = H / 128, IB = I / 128;
  long s = J->perm[r], t = s / Kp;
  int j = (int)(s % Kp);
  int e = (j < k) ? J->topk_idx[t * k + j] : d->E + (j - k);
  float wgt = (j < k) ? J->topk_w[t * k + j] : 1.0f;

  /* unscaled E4M3 activation row; its scales stay per block */
  for (long kk = 0; kk < H; ++kk) xh[kk] = orc_e4m3_to_float(J->x[t * H + kk]);
  /* L1: acc1[n] = sum_b (sx[t][b] * sw1[e][n/128][b]) * sum_{k in b} x[k] * W1[e][n][k] */
  for (long n = 0; n < 2L * I; ++n) {
    const uint8_t* wr = J->w1 + ((long)e * 2 * I + n) * H;
    float acc = 0.0f;
    for (long b = 0; b < HB; ++b) {
      float part = 0.0f;
      for (long kk = 128 * b; kk < 128 * b + 128; ++kk) part += xh[kk] * orc_e4m3_to_float(wr[kk]);
#if MUT(15)
      float sc = orc_f32_at(J->x_sf, t * HB + b); /* mistake: weight block scale dropped */
#else
      float sc = orc_f32_at(J->x_sf, t * HB + b) * orc_f32_at(J->w1_sf, ((long)e * (2 * I / 128) + n / 128) * HB + b);
#endif
      acc += part * sc;
    }
    a1[n] = acc;
  }
  if (J->acc1) memcpy(J->acc1 + r * 2L * I, a1, sizeof(float) * 2 * (size_t)I);

  /* SwiGLU: y = silu(clamp(g)) * clamp(u) * w */
  for (long n = 0; n < I; ++n) {
    float g = a1[n], u = a1[I + n];
    if (d->clamp > 0.0f) {
      g = fminf(fmaxf(g, -d->clamp), d->clamp);
      u = fminf(fmaxf(u, -d->clamp), d->clamp);
    }
    float silu = g / (1.0f + expf(-g));
    float v = silu * u;
    if (!d->weight_in_combine) v = v * wgt;
    y[n] = v;
  }
  /* requantise per 128 along I: float scale amax / 448, E4M3 of y / scale */
  float qs[128]; /* the row's L2-activation scales (I / 128 <= 128) */
  for (long b = 0; b < IB; ++b) {
    float amax = 0.0f;
    for (long n = 128 * b; n < 128 * b + 128; ++n) amax = fmaxf(amax, fabsf(y[n]));
    float sc = amax / 448.0f;
    if (!(sc > 0.0f)) sc = 1.0f;
#if MUT(16)
    sc = amax / 256.0f; /* mistake: scale from the wrong format maximum */
    if (!(sc > 0.0f)) sc = 1.0f;
#endif
    for (long n = 128 * b; n < 128 * b + 128; ++n) {
      uint8_t qq = orc_float_to_e4m3(y[n] / sc);
      if (J->q) J->q[r * I + n] = qq;
      qh[n] = orc_e4m3_to_float(qq);
    }
    if (J->qsf) memcpy(J->qsf + 4 * (r * IB + b), &sc, 4);
    qs[b] = sc;
  }
  /* L2: z[h] = bf16(sum_b (sq[b] * sw2[e][h/128][b]) * sum_{i in b} q[i] * W2[e][h][i]) */
  for (long h = 0; h < H; ++h) {
    const uint8_t* wr = J->w2 + ((long)e * H + h) * I;
    float acc = 0.0f;
    for (long b = 0; b < IB; ++b) {
      float part = 0.0f;
      for (long i = 128 * b; i < 128 * b + 128; ++i) part += qh[i] * orc_e4m3_to_float(wr[i]);
      float sc = qs[b] * orc_f32_at(J->w2_sf, ((long)e * HB + h / 128) * IB + b);
      acc += part * sc;
    }
    J->z[r * H + h] = orc_float_to_bf16(acc);
  }
}

static void* orc_worker(void* arg) {
  const orc_job* J = (const orc_job*)arg;
  const orc_dims* d = J->d;
  float* xh = (float*)malloc(sizeof(float) * (size_t)d->H);
  float* a1 = (float*)malloc(sizeof(float) * 2 * (size_t)d->I);
  float* y = (float*)malloc(sizeof(float) * (size_t)d->I);
  float* qh = (float*)malloc(sizeof(float) * (size_t)d->I);
  for (long r = J->th; r < J->nrows; r += J->nth) {
    if (d->w_fmt == 2) orc_one_row_f128(J, r, xh, a1, y, qh);
    else orc_one_row(J, r, xh, a1, y, qh);
  }
  free(xh); free(a1); free(y); free(qh);
  return NULL;
}

int orc_forward(const orc_dims* d, const uint8_t* x, const uint8_t* x_sf, const int32_t* topk_idx,
                const float* topk_w, const uint8_t* w1, const uint8_t* w1_sf, const uint8_t* w2,
                const uint8_t* w2_sf, uint16_t* out, float* acc1, uint8_t* q, uint8_t* qsf, uint16_t* z,
                int nthreads) {
  if (!d || d->T < 0 || d->H % 32 || d->I % 32 || d->E < 1 || d->k < 1 || d->S < 0) return -1;
  if (d->w_fmt != 0 && d->w_fmt != 1 && d->w_fmt != 2) return -1;
  if (d->w_fmt == 2 && (d->H % 128 || d->I % 128 || d->I > 16384)) return -1;
  const int T = d->T, H = d->H, k = d->k, Kp = d->k + d->S, Ep = d->E + d->S;
  long R = (long)T * Kp;
  int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * ((size_t)Ep + 1));
  int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * ((size_t)Ep + 1));
  int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * ((size_t)R + 1));
  int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * ((size_t)R + 1));
  uint16_t* zz = z ? z : (uint16_t*)malloc(sizeof(uint16_t) * ((size_t)R * H + 1));
  int bad = orc_route(T, d->k, d->S, d->E, topk_idx, counts, offsets, perm, pos);
  int nrows = offsets[Ep];

  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  orc_job jobs[512];
  pthread_t tid[512];
  for (int i = 0; i < nthreads; ++i) {
    orc_job J = {d, x, x_sf, w1, w1_sf, w2, w2_sf, topk_idx, topk_w, perm, nrows, acc1, q, qsf, zz, i, nthreads};
    jobs[i] = J;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&tid[i], NULL, orc_worker, &jobs[i]);
  orc_worker(&jobs[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(tid[i], NULL);

  /* combine: out[t][h] = bf16(sum over valid slots j ascending of z[pos[t,j]][h]) */
  for (long t = 0; t < T; ++t) {
    int last = -1;
    for (int j = 0; j < Kp; ++j) if (pos[t * Kp + j] >= 0) last = j;
    for (long h = 0; h < H; ++h) {
      float sum = 0.0f;
      for (int j = 0; j < Kp; ++j) {
        long r = pos[t * Kp + j];
        if (r < 0) continue;
#if MUT(7)
        if (j == last) continue; /* mistake: last slot dropped */
#endif
        float v = orc_bf16_to_float(zz[r * H + h]);
        if (d->weight_in_combine) v *= (j < k) ? topk_w[t * k + j] : 1.0f;
        sum += v;
      }
      out[t * H + h] = orc_float_to_bf16(sum);
    }
    (void)last;
  }
  free(counts); free(offsets); free(perm); free(pos);
  if (!z) free(zz);
  return bad;
}

void orc_l2_rows(int R, int H, int I, int w_fmt, const int32_t* expert_of_row, const uint8_t* q,
                 const uint8_t* qsf, const uint8_t* w2, const uint8_t* w2_sf, float* acc2) {
  if (w_fmt == 2) {
    const long HB = H / 128, IB = I / 128;
    for (long r = 0; r < R; ++r) {
      long e = expert_of_row[r];
      for (long h = 0; h < H; ++h) {
        const uint8_t* wr = w2 + (e * H + h) * I;
        float acc = 0.0f;
        for (long b = 0; b < IB; ++b) {
          float part = 0.0f;
          for (long i = 128 * b; i < 128 * b + 128; ++i)
            part += orc_e4m3_to_float(q[r * I + i]) * orc_e4m3_to_float(wr[i]);
          acc += part * (orc_f32_at(qsf, r * IB + b) * orc_f32_at(w2_sf, (e * HB + h / 128) * IB + b));
        }
        acc2[r * H + h] = acc;
      }
    }
    return;
  }
  for (long r = 0; r < R; ++r) {
    long e = expert_of_row[r];
    for (long h = 0; h < H; ++h) {
      const uint8_t* wr = w2 + (e * H + h) * orc_row_bytes(I, w_fmt);
      const uint8_t* sr = w2_sf + (e * H + h) * (I / 32);
      float acc = 0.0f;
      for (long i = 0; i < I; ++i) {
#if MUT(14)
        float a = orc_e4m3_to_float(q[r * I + i]); /* mistake: activation scale dropped in the L2-only path */
        (void)qsf;
#else
        float a = orc_e4m3_to_float(q[r * I + i]) * orc_ue8m0_to_float(qsf[r * (I / 32) + i / 32]);
#endif
        acc += a * (orc_weight(wr, i, w_fmt) * orc_ue8m0_to_float(sr[orc_sf_index(i)]));
      }
      acc2[r * H + h] = acc;
    }
  }
}
