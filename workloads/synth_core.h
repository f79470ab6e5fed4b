/*
 * Seeded synthetic inputs for the MoE expert path (input preparation only).
 *
 * This header is compiled twice: as host C (libsynth, used by the tests, the
 * oracle side and the CPU baseline) and as CUDA device code (libsynth_cuda,
 * used to fill multi-GB weight tensors directly in HBM). Every operation below
 * is integer arithmetic or an IEEE-754 single-precision multiply/divide/compare,
 * so both builds produce the same bytes.
 *
 * Definitions
 *   SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *   generators", OOPSLA 2014): state advances by the golden gamma
 *   0x9E3779B97F4A7C15 and each output is the mix64 finaliser of the state.
 *   syn_u64(key, n) is the n-th output of a SplitMix64 stream started at `key`,
 *   which makes the generator counter based (any element can be drawn alone).
 *
 *   Normal draws use the Irwin-Hall approximation: the sum of twelve uniform
 *   variates minus six has mean 0 and variance 1. The twelve uniforms are the
 *   16-bit fields of three SplitMix64 outputs, each taken as (u + 1/2) / 2^16,
 *   so the sum is an integer multiple of 2^-17 and is exact in float32.
 *
 *   Block quantisation (OCP Microscaling formats v1.0): one shared UE8M0
 *   exponent per 32 consecutive elements along the reduction dimension
 *   (weights in E2M1 (MXFP4) or, for the FP8 weight variant, E4M3 (MXFP8)),
 *   chosen as the smallest power of two s with amax / qmax <= s (qmax = 448
 *   for E4M3, 6 for E2M1), elements rounded to nearest-even in the element
 *   format after division by s.
 *
 *   Float-scale FP8 recipe (weights and activations E4M3, float32 scales per
 *   128 along K): an activation group of 128 takes the scale amax / 448 (one
 *   IEEE division) and its elements the nearest-even E4M3 of v / scale; a
 *   128 x 128 weight block takes a seeded scale std * 5/448 * u, u in [1, 2)
 *   on a 2^-23 grid (within a factor of two of the amax scale of a normal
 *   block, and never a power of two by construction except for u = 1), and
 *   its elements the E4M3 of w / scale (saturating beyond 448).
 *
 * None of this is a step of the expert computation itself; it only builds the
 * FP8 / MXFP4 byte tensors that both the CUDA path and the oracle consume.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>
#include <string.h>

#ifdef __CUDACC__
#define SYN_FN __host__ __device__ static inline
#else
#define SYN_FN static inline
#endif

/* Stream tags: one independent SplitMix64 stream per synthetic tensor. */
enum {
  SYN_TAG_X = 1,        /* activations x[T][H]                      */
  SYN_TAG_W1 = 2,       /* L1 weights [E'][2I][H] (gate rows, then up rows) */
  SYN_TAG_W2 = 3,       /* L2 weights [E'][H][I]                    */
  SYN_TAG_ROUTE = 4,    /* uniform top-k draws (partial Fisher-Yates) */
  SYN_TAG_ZIPF_PERM = 5,/* permutation of experts for Zipf ranks    */
  SYN_TAG_ZIPF_DRAW = 6,/* weighted draws for Zipf routing          */
  SYN_TAG_LOGITS = 7,   /* router logits for the top-k weights      */
  SYN_TAG_BLOCK_SF = 8  /* + (which - SYN_TAG_W1): float weight block scales */
};

SYN_FN uint32_t syn_f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
SYN_FN float syn_u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

SYN_FN uint64_t syn_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* n-th output (n = 0, 1, ...) of a SplitMix64 stream whose state starts at key. */
SYN_FN uint64_t syn_u64(uint64_t key, uint64_t n) {
  return syn_mix64(key + (n + 1ULL) * 0x9E3779B97F4A7C15ULL);
}

/* Key of the stream for (seed, tag): the first output of a SplitMix64 stream
 * started at seed * 2^8 + tag. */
SYN_FN uint64_t syn_stream_key(uint64_t seed, uint64_t tag) {
  return syn_u64((seed << 8) + tag, 0);
}

/* Irwin-Hall N(0,1) approximation for element `idx` of stream `key`. */
SYN_FN float syn_normal(uint64_t key, uint64_t idx) {
  uint64_t s = 0;
  for (int w = 0; w < 3; ++w) {
    uint64_t u = syn_u64(key, idx * 3ULL + (uint64_t)w);
    s += (u & 0xFFFFULL) + ((u >> 16) & 0xFFFFULL) + ((u >> 32) & 0xFFFFULL) + (u >> 48);
  }
  /* sum_i (u_i + 1/2) / 2^16 - 6 = (2 s + 12 - 12 * 2^16) / 2^17, |numerator| < 2^20 */
  int32_t num = (int32_t)(2 * s) + 12 - 786432;
  return (float)num * (1.0f / 131072.0f);
}

/* Round a finite float to the nearest bfloat16 value, ties to even. */
SYN_FN float syn_round_bf16(float f) {
  uint32_t b = syn_f2u(f);
  uint32_t r = b + 0x7FFFu + ((b >> 16) & 1u);
  return syn_u2f(r & 0xFFFF0000u);
}

/* Exact 2^n for -149 <= n <= 127. */
SYN_FN float syn_pow2(int n) {
  if (n >= -126) return syn_u2f((uint32_t)(n + 127) << 23);
  return syn_u2f(1u << (n + 149));
}

/* UE8M0 code of the smallest power of two s with amax / qmax <= s
 * (amax / qmax evaluated as one IEEE single-precision division),
 * clamped to [1, 254]; amax == 0 gives code 127 (s = 1). */
SYN_FN uint8_t syn_scale_code(float amax, float qmax) {
  if (!(amax > 0.0f)) return 127;
  float r = amax / qmax;
  uint32_t b = syn_f2u(r);
  int e = (int)((b >> 23) & 0xFFu);
  uint32_t m = b & 0x7FFFFFu;
  int code = (e == 0) ? 1 : ((m == 0) ? e : e + 1);
  if (code < 1) code = 1;
  if (code > 254) code = 254;
  return (uint8_t)code;
}

/* Nearest integer to t (0 <= t < 2^22), ties to even. */
SYN_FN uint32_t syn_rne_uint(float t) {
  uint32_t fl = (uint32_t)t;
  float frac = t - (float)fl;
  if (frac > 0.5f || (frac == 0.5f && (fl & 1u))) fl += 1u;
  return fl;
}

/* float -> FP8 E4M3 (OCP "fn" variant: bias 7, no infinities, max 448),
 * round to nearest even, saturating to +-448. Finite input only. */
SYN_FN uint8_t syn_e4m3_encode(float v) {
  uint32_t b = syn_f2u(v);
  uint8_t sign = (uint8_t)((b >> 24) & 0x80u);
  b &= 0x7FFFFFFFu;
  float a = syn_u2f(b);
  if (b == 0) return 0;
  if (a >= 448.0f) return (uint8_t)(sign | 0x7E);
  int e = (int)(b >> 23) - 127;
  uint8_t out;
  if (e < -6) {
    /* subnormal grid: multiples of 2^-9; a code of 8 is the smallest normal */
    uint32_t qi = syn_rne_uint(a * 512.0f);
    out = (uint8_t)qi;
  } else {
    uint32_t mant = b & 0x7FFFFFu;
    uint32_t keep = mant >> 20, rest = mant & 0xFFFFFu;
    if (rest > 0x80000u || (rest == 0x80000u && (keep & 1u))) keep += 1u;
    int ef = e + 7;
    if (keep == 8u) { keep = 0u; ef += 1; }
    if (ef > 15 || (ef == 15 && keep == 7u)) out = 0x7E;
    else out = (uint8_t)((ef << 3) | (int)keep);
  }
  return out ? (uint8_t)(sign | out) : (uint8_t)0;
}

/* float -> FP4 E2M1 code (values 0, .5, 1, 1.5, 2, 3, 4, 6), nearest even,
 * saturating to +-6. Finite input only. */
SYN_FN uint8_t syn_e2m1_encode(float v) {
  float a = v < 0.0f ? -v : v;
  uint8_t c;
  if (a <= 0.25f) c = 0;
  else if (a < 0.75f) c = 1;
  else if (a <= 1.25f) c = 2;
  else if (a < 1.75f) c = 3;
  else if (a <= 2.5f) c = 4;
  else if (a < 3.5f) c = 5;
  else if (a <= 5.0f) c = 6;
  else c = 7;
  return (c != 0 && v < 0.0f) ? (uint8_t)(c | 8) : c;
}

/* One 32-element group of activations: bf16(N(0,1)) -> E4M3 + UE8M0.
 * Element j of the group is stream element idx0 + j. */
SYN_FN void syn_group_x(uint64_t key, uint64_t idx0, uint8_t* q, uint8_t* sf) {
  float v[32];
  float amax = 0.0f;
  for (int j = 0; j < 32; ++j) {
    v[j] = syn_round_bf16(syn_normal(key, idx0 + (uint64_t)j));
    float a = v[j] < 0.0f ? -v[j] : v[j];
    if (a > amax) amax = a;
  }
  uint8_t code = syn_scale_code(amax, 448.0f);
  float inv = syn_pow2(127 - (int)code);
  for (int j = 0; j < 32; ++j) q[j] = syn_e4m3_encode(v[j] * inv);
  *sf = code;
}

/* One 32-element group of weights: N(0, std^2) -> E2M1 + UE8M0, packed two
 * per byte with the even element in the low nibble. */
SYN_FN void syn_group_w(uint64_t key, uint64_t idx0, float std_, uint8_t* packed16, uint8_t* sf) {
  float v[32];
  float amax = 0.0f;
  for (int j = 0; j < 32; ++j) {
    v[j] = syn_normal(key, idx0 + (uint64_t)j) * std_;
    float a = v[j] < 0.0f ? -v[j] : v[j];
    if (a > amax) amax = a;
  }
  uint8_t code = syn_scale_code(amax, 6.0f);
  float inv = syn_pow2(127 - (int)code);
  for (int j = 0; j < 16; ++j) {
    uint8_t lo = syn_e2m1_encode(v[2 * j] * inv);
    uint8_t hi = syn_e2m1_encode(v[2 * j + 1] * inv);
    packed16[j] = (uint8_t)(lo | (hi << 4));
  }
  *sf = code;
}

/* One 32-element group of FP8 weights: N(0, std^2) -> E4M3 + UE8M0 (the MXFP8
 * weight variant), one byte per element. Same stream elements as syn_group_w. */
SYN_FN void syn_group_w8(uint64_t key, uint64_t idx0, float std_, uint8_t* q32, uint8_t* sf) {
  float v[32];
  float amax = 0.0f;
  for (int j = 0; j < 32; ++j) {
    v[j] = syn_normal(key, idx0 + (uint64_t)j) * std_;
    float a = v[j] < 0.0f ? -v[j] : v[j];
    if (a > amax) amax = a;
  }
  uint8_t code = syn_scale_code(amax, 448.0f);
  float inv = syn_pow2(127 - (int)code);
  for (int j = 0; j < 32; ++j) q32[j] = syn_e4m3_encode(v[j] * inv);
  *sf = code;
}

/* One 128-element group of activations for the float-scale recipe:
 * bf16(N(0,1)) -> E4M3 with a float32 scale amax / 448 (1 when amax is 0).
 * Element j is stream element idx0 + j (the values of syn_group_x). */
SYN_FN void syn_group_x128(uint64_t key, uint64_t idx0, uint8_t* q, float* sf) {
  float v[128];
  float amax = 0.0f;
  for (int j = 0; j < 128; ++j) {
    v[j] = syn_round_bf16(syn_normal(key, idx0 + (uint64_t)j));
    float a = v[j] < 0.0f ? -v[j] : v[j];
    if (a > amax) amax = a;
  }
  float s = amax / 448.0f;
  if (!(s > 0.0f)) s = 1.0f;
  for (int j = 0; j < 128; ++j) q[j] = syn_e4m3_encode(v[j] / s);
  *sf = s;
}

/* Float32 scale of 128 x 128 weight block `idx` of stream `key`:
 * (std * 5/448) * u with u = 1 + m * 2^-23, m the top 23 bits of the draw. */
SYN_FN float syn_block_scale(uint64_t key, uint64_t idx, float std_) {
  uint64_t d = syn_u64(key, idx);
  float u = 1.0f + (float)(uint32_t)(d >> 41) * (1.0f / 8388608.0f);
  return (std_ * 0x1.6db6dcp-7f) * u;
}

/* One weight element of the float-scale recipe: E4M3 of (N(0,1) * std) / scale,
 * stream element idx (the values of syn_group_w / syn_group_w8). */
SYN_FN uint8_t syn_elem_w8f(uint64_t key, uint64_t idx, float std_, float scale) {
  return syn_e4m3_encode((syn_normal(key, idx) * std_) / scale);
}

#endif /* SYNTH_CORE_H */
