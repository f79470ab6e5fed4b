/*
 * Host build of the seeded synthetic-input generator (see synth_core.h).
 * Exported with C linkage for ctypes. Compile with -ffp-contract=off.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include "synth_core.h"

/* x rows [t0, t1) of a [T][H] activation tensor: E4M3 bytes + UE8M0 per 32. */
void syn_gen_x(uint64_t seed, int H, int t0, int t1, uint8_t* x, uint8_t* x_sf) {
  uint64_t key = syn_stream_key(seed, SYN_TAG_X);
  int G = H / 32;
  for (int t = t0; t < t1; ++t)
    for (int g = 0; g < G; ++g)
      syn_group_x(key, (uint64_t)t * (uint64_t)H + (uint64_t)g * 32u,
                  x + (size_t)(t - t0) * H + (size_t)g * 32, x_sf + (size_t)(t - t0) * G + g);
}

/* x rows [t0, t1) for the float-scale recipe: E4M3 bytes + float32 scale per 128. */
void syn_gen_x128(uint64_t seed, int H, int t0, int t1, uint8_t* x, float* x_sf) {
  uint64_t key = syn_stream_key(seed, SYN_TAG_X);
  int G = H / 128;
  for (int t = t0; t < t1; ++t)
    for (int g = 0; g < G; ++g)
      syn_group_x128(key, (uint64_t)t * (uint64_t)H + (uint64_t)g * 128u,
                     x + (size_t)(t - t0) * H + (size_t)g * 128, x_sf + (size_t)(t - t0) * G + g);
}

typedef struct {
  uint64_t key;
  int rows, K, e0, e1, th, nth, fp8;
  float std_;
  uint8_t *w, *w_sf;
} syn_wjob;

static void* syn_w_worker(void* arg) {
  syn_wjob* j = (syn_wjob*)arg;
  int G = j->K / 32;
  long total = (long)(j->e1 - j->e0) * j->rows;
  for (long r = j->th; r < total; r += j->nth) {
    long e = j->e0 + r / j->rows, n = r % j->rows;
    uint64_t base = ((uint64_t)e * (uint64_t)j->rows + (uint64_t)n) * (uint64_t)j->K;
    for (int g = 0; g < G; ++g) {
      if (j->fp8)
        syn_group_w8(j->key, base + (uint64_t)g * 32u, j->std_, j->w + (size_t)r * j->K + (size_t)g * 32,
                     j->w_sf + (size_t)r * G + g);
      else
        syn_group_w(j->key, base + (uint64_t)g * 32u, j->std_,
                    j->w + (size_t)r * (j->K / 2) + (size_t)g * 16, j->w_sf + (size_t)r * G + g);
    }
  }
  return NULL;
}

/* Weight tensor `which` (SYN_TAG_W1 or SYN_TAG_W2) for experts [e0, e1):
 * rows_per_expert rows of K elements each, E2M1 packed + UE8M0 per 32 along K.
 * Output buffers hold only the requested experts, expert e0 first. */
static void syn_gen_w_any(uint64_t seed, int which, int rows_per_expert, int K, int e0, int e1,
                          float std_, uint8_t* w, uint8_t* w_sf, int nthreads, int fp8) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  syn_wjob jobs[256];
  pthread_t tid[256];
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].key = syn_stream_key(seed, (uint64_t)which);
    jobs[i].rows = rows_per_expert; jobs[i].K = K; jobs[i].e0 = e0; jobs[i].e1 = e1;
    jobs[i].th = i; jobs[i].nth = nthreads; jobs[i].std_ = std_; jobs[i].w = w; jobs[i].w_sf = w_sf;
    jobs[i].fp8 = fp8;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&tid[i], NULL, syn_w_worker, &jobs[i]);
  syn_w_worker(&jobs[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(tid[i], NULL);
}

typedef struct {
  uint64_t key, skey;
  int rows, K, e0, e1, th, nth;
  float std_;
  uint8_t* w;
  float* w_sf;
} syn_w8f_job;

static void* syn_w8f_worker(void* arg) {
  syn_w8f_job* j = (syn_w8f_job*)arg;
  const int RB = j->rows / 128, KB = j->K / 128;
  long total = (long)(j->e1 - j->e0) * j->rows;
  for (long r = j->th; r < total; r += j->nth) {
    long e = j->e0 + r / j->rows, n = r % j->rows;
    uint64_t base = ((uint64_t)e * (uint64_t)j->rows + (uint64_t)n) * (uint64_t)j->K;
    for (int kb = 0; kb < KB; ++kb) {
      uint64_t bi = ((uint64_t)e * (uint64_t)RB + (uint64_t)(n / 128)) * (uint64_t)KB + (uint64_t)kb;
      float sc = syn_block_scale(j->skey, bi, j->std_);
      if (n % 128 == 0) j->w_sf[((size_t)(r / j->rows) * RB + (size_t)(n / 128)) * KB + kb] = sc;
      for (int k = 128 * kb; k < 128 * kb + 128; ++k)
        j->w[(size_t)r * j->K + k] = syn_elem_w8f(j->key, base + (uint64_t)k, j->std_, sc);
    }
  }
  return NULL;
}

/* Weights for the float-scale recipe, experts [e0, e1): E4M3 [n][rows][K] and
 * float32 block scales [n][rows/128][K/128]. */
void syn_gen_w8f(uint64_t seed, int which, int rows_per_expert, int K, int e0, int e1,
                 float std_, uint8_t* w, float* w_sf, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  syn_w8f_job jobs[256];
  pthread_t tid[256];
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].key = syn_stream_key(seed, (uint64_t)which);
    jobs[i].skey = syn_stream_key(seed, (uint64_t)(SYN_TAG_BLOCK_SF + (which - SYN_TAG_W1)));
    jobs[i].rows = rows_per_expert; jobs[i].K = K; jobs[i].e0 = e0; jobs[i].e1 = e1;
    jobs[i].th = i; jobs[i].nth = nthreads; jobs[i].std_ = std_; jobs[i].w = w; jobs[i].w_sf = w_sf;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&tid[i], NULL, syn_w8f_worker, &jobs[i]);
  syn_w8f_worker(&jobs[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(tid[i], NULL);
}

void syn_gen_w(uint64_t seed, int which, int rows_per_expert, int K, int e0, int e1,
               float std_, uint8_t* w, uint8_t* w_sf, int nthreads) {
  syn_gen_w_any(seed, which, rows_per_expert, K, e0, e1, std_, w, w_sf, nthreads, 0);
}

/* Same weights quantised to E4M3 + UE8M0 (one byte per element, K bytes per row). */
void syn_gen_w8(uint64_t seed, int which, int rows_per_expert, int K, int e0, int e1,
                float std_, uint8_t* w, uint8_t* w_sf, int nthreads) {
  syn_gen_w_any(seed, which, rows_per_expert, K, e0, e1, std_, w, w_sf, nthreads, 1);
}

/* Routing for T tokens over E experts, k distinct experts per token.
 *   zipf_s <= 0: uniform without replacement (partial Fisher-Yates over 0..E-1).
 *   zipf_s  > 0: expert pi(r) has weight (r+1)^-zipf_s for a seeded permutation
 *                pi; k sequential weighted draws without replacement.
 * Top-k weights: softmax over the k chosen of Irwin-Hall N(0,1) logits. */
int syn_gen_routing(uint64_t seed, int T, int E, int k, double zipf_s, int32_t* topk_idx, float* topk_w) {
  if (k > E || k < 1 || E < 1) return -1;
  int* perm = (int*)malloc(sizeof(int) * (size_t)E);
  double* wt = (double*)malloc(sizeof(double) * (size_t)E);
  char* used = (char*)malloc((size_t)E);
  if (!perm || !wt || !used) { free(perm); free(wt); free(used); return -2; }
  if (zipf_s > 0.0) {
    uint64_t kp = syn_stream_key(seed, SYN_TAG_ZIPF_PERM);
    for (int i = 0; i < E; ++i) perm[i] = i;
    for (int i = 0; i < E - 1; ++i) {
      int j = i + (int)(syn_u64(kp, (uint64_t)i) % (uint64_t)(E - i));
      int tmp = perm[i]; perm[i] = perm[j]; perm[j] = tmp;
    }
    for (int r = 0; r < E; ++r) wt[perm[r]] = pow((double)(r + 1), -zipf_s);
  }
  uint64_t kr = syn_stream_key(seed, SYN_TAG_ROUTE);
  uint64_t kz = syn_stream_key(seed, SYN_TAG_ZIPF_DRAW);
  uint64_t kl = syn_stream_key(seed, SYN_TAG_LOGITS);
  for (int t = 0; t < T; ++t) {
    if (zipf_s > 0.0) {
      for (int e = 0; e < E; ++e) used[e] = 0;
      for (int j = 0; j < k; ++j) {
        double total = 0.0;
        for (int e = 0; e < E; ++e) if (!used[e]) total += wt[e];
        double u = (double)(syn_u64(kz, (uint64_t)t * (uint64_t)k + (uint64_t)j) >> 11) * (1.0 / 9007199254740992.0);
        double target = u * total, acc = 0.0;
        int pick = -1, last = -1;
        for (int e = 0; e < E; ++e) {
          if (used[e]) continue;
          last = e;
          acc += wt[e];
          if (acc > target) { pick = e; break; }
        }
        if (pick < 0) pick = last;
        used[pick] = 1;
        topk_idx[(size_t)t * k + j] = pick;
      }
    } else {
      for (int i = 0; i < E; ++i) perm[i] = i;
      for (int j = 0; j < k; ++j) {
        int r = j + (int)(syn_u64(kr, (uint64_t)t * (uint64_t)E + (uint64_t)j) % (uint64_t)(E - j));
        int tmp = perm[j]; perm[j] = perm[r]; perm[r] = tmp;
        topk_idx[(size_t)t * k + j] = perm[j];
      }
    }
    double mx = -1e300, den = 0.0, lg[64];
    int kk = k < 64 ? k : 64;
    for (int j = 0; j < kk; ++j) {
      lg[j] = (double)syn_normal(kl, (uint64_t)t * (uint64_t)k + (uint64_t)j);
      if (lg[j] > mx) mx = lg[j];
    }
    for (int j = 0; j < kk; ++j) den += exp(lg[j] - mx);
    for (int j = 0; j < k; ++j) topk_w[(size_t)t * k + j] = j < kk ? (float)(exp(lg[j] - mx) / den) : 0.0f;
  }
  free(perm); free(wt); free(used);
  return 0;
}

/* Exposed for generator tests: single draws. */
uint64_t syn_u64_at(uint64_t key, uint64_t n) { return syn_u64(key, n); }
uint64_t syn_key(uint64_t seed, uint64_t tag) { return syn_stream_key(seed, tag); }
float syn_normal_at(uint64_t key, uint64_t idx) { return syn_normal(key, idx); }
