/*
 * Device build of the seeded synthetic-input generator (see synth_core.h):
 * fills FP8 activations and MXFP4 weights directly in device memory with the
 * same bytes the host build produces. Compile with -fmad=false.
 */
#include <cuda_runtime.h>
#include "synth_core.h"

__global__ void syn_x_kernel(uint64_t key, int H, long long groups, uint8_t* x, uint8_t* x_sf) {
  const int G = H / 32;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < groups;
       g += (long long)gridDim.x * blockDim.x) {
    long long t = g / G, gg = g % G;
    uint8_t q[32];
    uint8_t sf;
    syn_group_x(key, (uint64_t)t * (uint64_t)H + (uint64_t)gg * 32u, q, &sf);
    uint4* dst = reinterpret_cast<uint4*>(x + (size_t)t * H + (size_t)gg * 32);
    uint4 a, b;
    memcpy(&a, q, 16);
    memcpy(&b, q + 16, 16);
    dst[0] = a;
    dst[1] = b;
    x_sf[(size_t)t * G + gg] = sf;
  }
}

__global__ void syn_w_kernel(uint64_t key, int rows, int K, int e0, long long groups, float std_,
                             uint8_t* w, uint8_t* w_sf) {
  const int G = K / 32;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < groups;
       g += (long long)gridDim.x * blockDim.x) {
    long long r = g / G, gg = g % G;           /* r: row within the requested experts */
    long long e = e0 + r / rows, n = r % rows;
    uint64_t base = ((uint64_t)e * (uint64_t)rows + (uint64_t)n) * (uint64_t)K + (uint64_t)gg * 32u;
    uint8_t p[16];
    uint8_t sf;
    syn_group_w(key, base, std_, p, &sf);
    uint4 a;
    memcpy(&a, p, 16);
    *reinterpret_cast<uint4*>(w + (size_t)r * (K / 2) + (size_t)gg * 16) = a;
    w_sf[(size_t)r * G + gg] = sf;
  }
}

__global__ void syn_w8_kernel(uint64_t key, int rows, int K, int e0, long long groups, float std_,
                              uint8_t* w, uint8_t* w_sf) {
  const int G = K / 32;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < groups;
       g += (long long)gridDim.x * blockDim.x) {
    long long r = g / G, gg = g % G;
    long long e = e0 + r / rows, n = r % rows;
    uint64_t base = ((uint64_t)e * (uint64_t)rows + (uint64_t)n) * (uint64_t)K + (uint64_t)gg * 32u;
    uint8_t q[32];
    uint8_t sf;
    syn_group_w8(key, base, std_, q, &sf);
    uint4 a, b;
    memcpy(&a, q, 16);
    memcpy(&b, q + 16, 16);
    uint4* dst = reinterpret_cast<uint4*>(w + (size_t)r * K + (size_t)gg * 32);
    dst[0] = a;
    dst[1] = b;
    w_sf[(size_t)r * G + gg] = sf;
  }
}

__global__ void syn_x128_kernel(uint64_t key, int H, long long groups, uint8_t* x, float* x_sf) {
  const int G = H / 128;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < groups;
       g += (long long)gridDim.x * blockDim.x) {
    long long t = g / G, gg = g % G;
    uint8_t q[128];
    float sf;
    syn_group_x128(key, (uint64_t)t * (uint64_t)H + (uint64_t)gg * 128u, q, &sf);
    uint4* dst = reinterpret_cast<uint4*>(x + (size_t)t * H + (size_t)gg * 128);
    for (int c = 0; c < 8; ++c) {
      uint4 a;
      memcpy(&a, q + 16 * c, 16);
      dst[c] = a;
    }
    x_sf[(size_t)t * G + gg] = sf;
  }
}

/* One thread per 16 consecutive elements of a row within one 128-wide K block. */
__global__ void syn_w8f_kernel(uint64_t key, uint64_t skey, int rows, int K, int e0, long long chunks, float std_,
                               uint8_t* w, float* w_sf) {
  const int C = K / 16, RB = rows / 128, KB = K / 128;
  for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < chunks;
       c += (long long)gridDim.x * blockDim.x) {
    long long r = c / C, cc = c % C;            /* r: row within the requested experts */
    long long e = e0 + r / rows, n = r % rows;
    int kb = (int)(cc / 8);
    uint64_t bi = ((uint64_t)e * (uint64_t)RB + (uint64_t)(n / 128)) * (uint64_t)KB + (uint64_t)kb;
    float sc = syn_block_scale(skey, bi, std_);
    uint64_t base = ((uint64_t)e * (uint64_t)rows + (uint64_t)n) * (uint64_t)K + (uint64_t)cc * 16u;
    uint8_t q[16];
    for (int j = 0; j < 16; ++j) q[j] = syn_elem_w8f(key, base + (uint64_t)j, std_, sc);
    uint4 a;
    memcpy(&a, q, 16);
    *reinterpret_cast<uint4*>(w + (size_t)r * K + (size_t)cc * 16) = a;
    if (n % 128 == 0 && cc % 8 == 0) w_sf[((size_t)(r / rows) * RB + (size_t)(n / 128)) * KB + kb] = sc;
  }
}

static int syn_grid(long long groups) {
  long long b = (groups + 255) / 256;
  if (b > 152 * 64) b = 152 * 64;
  if (b < 1) b = 1;
  return (int)b;
}

extern "C" int syn_dev_gen_x(uint64_t seed, int T, int H, void* x, void* x_sf, void* stream) {
  if (T <= 0) return 0;
  if (H % 32) return -1;
  long long groups = (long long)T * (H / 32);
  syn_x_kernel<<<syn_grid(groups), 256, 0, (cudaStream_t)stream>>>(
      syn_stream_key(seed, SYN_TAG_X), H, groups, (uint8_t*)x, (uint8_t*)x_sf);
  return (int)cudaGetLastError();
}

extern "C" int syn_dev_gen_w(uint64_t seed, int which, int rows_per_expert, int K, int e0, int e1,
                             float std_, void* w, void* w_sf, void* stream) {
  if (e1 <= e0) return 0;
  if (K % 32) return -1;
  long long groups = (long long)(e1 - e0) * rows_per_expert * (K / 32);
  syn_w_kernel<<<syn_grid(groups), 256, 0, (cudaStream_t)stream>>>(
      syn_stream_key(seed, (uint64_t)which), rows_per_expert, K, e0, groups, std_, (uint8_t*)w, (uint8_t*)w_sf);
  return (int)cudaGetLastError();
}

extern "C" int syn_dev_gen_w8(uint64_t seed, int which, int rows_per_expert, int K, int e0, int e1,
                              float std_, void* w, void* w_sf, void* stream) {
  if (e1 <= e0) return 0;
  if (K % 32) return -1;
  long long groups = (long long)(e1 - e0) * rows_per_expert * (K / 32);
  syn_w8_kernel<<<syn_grid(groups), 256, 0, (cudaStream_t)stream>>>(
      syn_stream_key(seed, (uint64_t)which), rows_per_expert, K, e0, groups, std_, (uint8_t*)w, (uint8_t*)w_sf);
  return (int)cudaGetLastError();
}

extern "C" int syn_dev_gen_x128(uint64_t seed, int T, int H, void* x, void* x_sf, void* stream) {
  if (T <= 0) return 0;
  if (H % 128) return -1;
  long long groups = (long long)T * (H / 128);
  syn_x128_kernel<<<syn_grid(groups), 256, 0, (cudaStream_t)stream>>>(
      syn_stream_key(seed, SYN_TAG_X), H, groups, (uint8_t*)x, (float*)x_sf);
  return (int)cudaGetLastError();
}

extern "C" int syn_dev_gen_w8f(uint64_t seed, int which, int rows_per_expert, int K, int e0, int e1,
                               float std_, void* w, void* w_sf, void* stream) {
  if (e1 <= e0) return 0;
  if (K % 128 || rows_per_expert % 128) return -1;
  long long chunks = (long long)(e1 - e0) * rows_per_expert * (K / 16);
  syn_w8f_kernel<<<syn_grid(chunks), 256, 0, (cudaStream_t)stream>>>(
      syn_stream_key(seed, (uint64_t)which), syn_stream_key(seed, (uint64_t)(SYN_TAG_BLOCK_SF + (which - SYN_TAG_W1))),
      rows_per_expert, K, e0, chunks, std_, (uint8_t*)w, (float*)w_sf);
  return (int)cudaGetLastError();
}
