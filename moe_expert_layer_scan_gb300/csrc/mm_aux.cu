// Router, row gather, combine and the bounded-wait probe.
//
// Router: the pages' dispatch bookkeeping ("MegaMoE research report" sec. 4.1,
// WG0: expert counts, source metadata; "MEGAMOE_SM90_DESIGN" sec. 9.2 pool
// fill) on one GPU. Slots s = t*(k+S)+j are counted per expert, the counts
// prefix-summed into pool offsets, and every slot placed at
// offsets[e] + (number of earlier slots of the same expert) — a stable
// counting sort, so the result is unique and bit-reproducible.
// Combine: "MEGAMOE_SM90_DESIGN" sec. 11.2 — per token, the BF16 rows of its
// active slots are summed in FP32 in slot order and cast to BF16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mm_internal.h"
#include "mm_ptx.cuh"

namespace mm {

__device__ __forceinline__ int slot_expert(const RouteArgs& a, long s, bool* bad) {
  const int Kp = a.k + a.S;
  const long t = s / Kp;
  const int j = (int)(s - t * Kp);
  if (j >= a.k) return a.E + (j - a.k);
  const int e = a.topk_idx[t * a.k + j];
  if (e == -1) return -1;
  if (e < 0 || e >= a.E) {
    *bad = true;
    return -1;
  }
  return e;
}

// Exclusive prefix sum over blockDim.x (= 1024) threads; returns the
// exclusive value of this thread and writes the total to *total.
__device__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    scratch[32 + lane] = wi - w;  // exclusive warp prefix
    if (lane == 31) scratch[64] = wi;
  }
  __syncthreads();
  const int excl = incl - v + scratch[32 + warp];
  *total = scratch[64];
  __syncthreads();
  return excl;
}

// Stable placement of the slots [c0, c1) by one CTA of 1024 threads (32
// warps). hist[w][e] must hold, for every warp w and expert e, the first pool
// row warp w writes for expert e; warp w owns a contiguous sub-range and walks
// it 32 slots at a time in order, ranking equal experts with __match_any_sync.
__device__ void place_slots(const RouteArgs& a, long c0, long c1, int* hist) {
  const int Ep = a.E + a.S, Kp = a.k + a.S;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long sub = (c1 - c0 + 31) / 32;
  const long s0 = c0 + warp * sub, s1 = (s0 + sub < c1) ? s0 + sub : c1;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (long base = s0; base < s1; base += 32) {
    const long s = base + lane;
    const bool in = s < s1;
    bool dummy = false;
    const int e = in ? slot_expert(a, s, &dummy) : -2;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0) {
      const int p = hist[warp * Ep + e] + rank;
      a.perm[p] = (int32_t)s;
      a.pos[s] = p;
      const long t = s / Kp;
      const int j = (int)(s - t * Kp);
      a.row_w[p] = (j < a.k) ? a.topk_w[t * a.k + j] : 1.0f;
    } else if (in) {
      a.pos[s] = -1;
    }
    __syncwarp();
    if (e >= 0 && rank == 0) hist[warp * Ep + e] += __popc(peers);
    __syncwarp();
  }
}

// Per-warp expert histograms of the slots [c0, c1) (same split as place_slots).
__device__ bool warp_histograms(const RouteArgs& a, long c0, long c1, int* hist) {
  const int Ep = a.E + a.S;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32 * Ep; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const long sub = (c1 - c0 + 31) / 32;
  const long s0 = c0 + warp * sub, s1 = (s0 + sub < c1) ? s0 + sub : c1;
  bool bad = false;
  for (long s = s0 + lane; s < s1; s += 32) {
    const int e = slot_expert(a, s, &bad);
    if (e >= 0) atomicAdd(&hist[warp * Ep + e], 1);
  }
  __syncthreads();
  return bad;
}

// Counts -> offsets (exclusive scan) and the two GEMM tile tables; thread e
// holds expert e's total in `tot`. Called by all 1024 threads.
__device__ int offsets_and_tiles(const RouteArgs& a, int tot, int* scratch) {
  const int Ep = a.E + a.S;
  const int tid = threadIdx.x;
  int total_rows;
  const int excl = block_exclusive_scan(tid < Ep ? tot : 0, scratch, &total_rows);
  if (tid < Ep) {
    a.counts[tid] = tot;
    a.offsets[tid] = excl;
  }
  if (tid == 0) a.offsets[Ep] = total_rows;
  // Tile order. With per-expert tile widths (dual_sms > 0): the experts with
  // more than one token tile ("heavy", compute bound) first, then the rest
  // (weight-stream bound), each group in expert order, so that each class's
  // launch takes one range of tiles. Otherwise the expert order (nheavy = 0).
  __shared__ int pt1[kMaxExperts], pt2[kMaxExperts];
  int nheavy = 0, p = tid;
  bool heavy = false;
  if (a.dual_sms > 0) {
    heavy = tid < Ep && tot > a.bn_l1;
    const int hrank = block_exclusive_scan(heavy ? 1 : 0, scratch, &nheavy);
    p = heavy ? hrank : nheavy + (tid - hrank);
  }
  if (tid < Ep) {
    const int bn1 = heavy ? a.bn_heavy : a.bn_l1, bn2 = heavy ? a.bn_heavy : a.bn_l2;
    pt1[p] = (tot + bn1 - 1) / bn1 * a.fb_l1;
    pt2[p] = (tot + bn2 - 1) / bn2 * a.fb_l2;
    a.eorder[p] = tid;
  }
  __syncthreads();
  const int t1 = tid < Ep ? pt1[tid] : 0, t2 = tid < Ep ? pt2[tid] : 0;
  int n1, n2;
  const int e1 = block_exclusive_scan(t1, scratch, &n1);
  const int e2 = block_exclusive_scan(t2, scratch, &n2);
  if (tid < Ep) {
    a.tiles_l1[tid] = e1;
    a.tiles_l2[tid] = e2;
  }
  if (tid == 0) {
    a.tiles_l1[Ep] = n1;
    a.tiles_l2[Ep] = n2;
  }
  // the heavy experts' tiles: the prefix at position nheavy (all tiles when
  // every expert is heavy)
  if (tid == (nheavy < Ep ? nheavy : 0)) {
    const int h1 = nheavy < Ep ? e1 : n1;
    a.tiles_l1[Ep + 1] = h1;
    a.tiles_l2[Ep + 1] = nheavy < Ep ? e2 : n2;
    if (a.dual_sms > 0) {
      // the heavy class's share of the SMs, by the classes' weighted L1 tiles
      const long long cw = (long long)h1 * kCostHeavyTile, cl = (long long)(n1 - h1) * kCostLightTile;
      int g = cw + cl > 0 ? (int)((2 * cw * a.dual_sms + (cw + cl)) / (2 * (cw + cl))) : 0;
      if (cw > 0 && g < 1) g = 1;
      if (cl > 0 && g > a.dual_sms - 1) g = a.dual_sms - 1;
      a.sched[kSchedHeavyCtas] = g;
    }
  }
  if (tid == 0) a.sched[kSchedHeavyExperts] = nheavy;
  // Expert-parallel-ready outputs. With the routed experts split over ranks in
  // contiguous blocks, the expert-major order is also rank-major, so each
  // destination rank's rows are one range of the sorted order. The shared
  // experts (replicated on every rank) follow the last routed rank.
  const int per_rank = a.E / a.ep_ranks;
  if (tid < a.E && tid % per_rank == 0) a.rank_offsets[tid / per_rank] = excl;
  if (a.S > 0 && tid == a.E) a.rank_offsets[a.ep_ranks] = excl;
  if (a.S == 0 && tid == 0) a.rank_offsets[a.ep_ranks] = total_rows;
  // cumulative per-expert receive statistics (never cleared here)
  if (a.stats && tid < Ep && tot > 0) atomicAdd(&a.stats[tid], tot);
  return excl;
}

// Routing of at most kRouteSmallMax slots (decode-sized calls) by one CTA:
// every slot's expert is read once into shared memory and counted with
// shared atomics; a slot's rank within its expert is the number of earlier
// slots of the same expert, counted from the shared list, which keeps the
// placement stable (ascending slot order within each expert).
__global__ void __launch_bounds__(1024, 1) route_small_kernel(RouteArgs a) {
  __shared__ int es[kRouteSmallMax];
  __shared__ int cnt[kMaxExperts];
  __shared__ int first[kMaxExperts];
  __shared__ int scratch[72];
  __shared__ int bad_any;
  pdl_trigger();
  const int Ep = a.E + a.S, Kp = a.k + a.S;
  const int R = a.T * Kp;
  const int tid = threadIdx.x;
  if (tid == 0) bad_any = 0;
  if (tid < Ep) cnt[tid] = 0;
  for (int i = tid; i <= R; i += blockDim.x) a.ready[i] = 0;
  if (tid < kSchedCounters) a.sched[tid] = 0;
  __syncthreads();
  bool bad = false;
  int e = -1;
  if (tid < R) {
    e = slot_expert(a, tid, &bad);
    es[tid] = e;
    if (e >= 0) atomicAdd(&cnt[e], 1);
  }
  if (bad) bad_any = 1;
  __syncthreads();
  const int excl = offsets_and_tiles(a, tid < Ep ? cnt[tid] : 0, scratch);
  if (tid < Ep) first[tid] = excl;
  __syncthreads();
  if (tid < R) {
    if (e >= 0) {
      int rank = 0;
      for (int s2 = 0; s2 < tid; ++s2) rank += es[s2] == e ? 1 : 0;
      const int p = first[e] + rank;
      a.perm[p] = tid;
      a.pos[tid] = p;
      const int t = tid / Kp, j = tid - t * Kp;
      a.row_w[p] = (j < a.k) ? a.topk_w[t * a.k + j] : 1.0f;
    } else {
      a.pos[tid] = -1;
    }
  }
  if (tid == 0) *a.status = bad_any ? MM_DEV_BAD_ROUTING : 0u;
}

// Routing by one CTA (few slots): histograms, offsets, cursors, placement.
__global__ void __launch_bounds__(1024, 1) route_kernel(RouteArgs a) {
  extern __shared__ int sh[];
  pdl_trigger();
  const int Ep = a.E + a.S, Kp = a.k + a.S;
  const long R = (long)a.T * Kp;
  int* hist = sh;               // [32][Ep]
  int* scratch = sh + 32 * Ep;  // [72]
  __shared__ int bad_any;
  const int tid = threadIdx.x;
  if (tid == 0) bad_any = 0;
  for (long i = tid; i <= R; i += blockDim.x) a.ready[i] = 0;
  if (tid < kSchedCounters) a.sched[tid] = 0;
  const bool bad = warp_histograms(a, 0, R, hist);
  if (bad) bad_any = 1;
  int tot = 0;
  if (tid < Ep)
    for (int w = 0; w < 32; ++w) tot += hist[w * Ep + tid];
  const int excl = offsets_and_tiles(a, tot, scratch);
  if (tid < Ep) {
    int run = excl;
    for (int w = 0; w < 32; ++w) {
      const int c = hist[w * Ep + tid];
      hist[w * Ep + tid] = run;
      run += c;
    }
  }
  __syncthreads();
  place_slots(a, 0, R, hist);
  __syncthreads();
  if (tid == 0) *a.status = bad_any ? MM_DEV_BAD_ROUTING : 0u;
}

// Multi-CTA routing, pass 1: expert counts of each chunk of kRouteChunk slots.
__global__ void __launch_bounds__(1024) route_count_kernel(RouteArgs a) {
  extern __shared__ int hist[];  // [Ep]
  pdl_trigger();
  __shared__ int bad_any;
  const int Ep = a.E + a.S, Kp = a.k + a.S;
  const long R = (long)a.T * Kp;
  const long c0 = (long)blockIdx.x * kRouteChunk, c1 = (c0 + kRouteChunk < R) ? c0 + kRouteChunk : R;
  if (threadIdx.x == 0) bad_any = 0;
  for (int i = threadIdx.x; i < Ep; i += blockDim.x) hist[i] = 0;
  for (long i = c0 + threadIdx.x; i < c1; i += blockDim.x) a.ready[i] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) a.ready[R] = 0;
  if (blockIdx.x == 0 && threadIdx.x < kSchedCounters) a.sched[threadIdx.x] = 0;
  __syncthreads();
  bool bad = false;
  for (long s = c0 + threadIdx.x; s < c1; s += blockDim.x) {
    const int e = slot_expert(a, s, &bad);
    if (e >= 0) atomicAdd(&hist[e], 1);
  }
  if (bad) bad_any = 1;
  __syncthreads();
  for (int i = threadIdx.x; i < Ep; i += blockDim.x) a.chunk_cnt[(size_t)blockIdx.x * Ep + i] = hist[i];
  if (threadIdx.x == 0) a.chunk_bad[blockIdx.x] = bad_any;
}

// Pass 2 (one CTA): totals, offsets, tile tables, each chunk's first row per
// expert, and the status word.
__global__ void __launch_bounds__(1024, 1) route_scan_kernel(RouteArgs a, int G) {
  __shared__ int scratch[72];
  __shared__ int bad_any;
  pdl_trigger();
  pdl_wait();
  const int Ep = a.E + a.S;
  const int tid = threadIdx.x;
  if (tid == 0) bad_any = 0;
  __syncthreads();
  int tot = 0;
  if (tid < Ep)
    for (int g = 0; g < G; ++g) tot += a.chunk_cnt[(size_t)g * Ep + tid];
  for (int g = tid; g < G; g += blockDim.x)
    if (a.chunk_bad[g]) bad_any = 1;
  const int excl = offsets_and_tiles(a, tot, scratch);
  if (tid < Ep) {
    int run = excl;
    for (int g = 0; g < G; ++g) {
      const int c = a.chunk_cnt[(size_t)g * Ep + tid];
      a.chunk_base[(size_t)g * Ep + tid] = run;
      run += c;
    }
  }
  __syncthreads();
  if (tid == 0) *a.status = bad_any ? MM_DEV_BAD_ROUTING : 0u;
}

// Pass 3: each CTA places its chunk's slots, starting at the chunk's first row
// per expert.
__global__ void __launch_bounds__(1024, 1) route_place_kernel(RouteArgs a) {
  extern __shared__ int hist[];  // [32][Ep]
  pdl_trigger();
  pdl_wait();
  const int Ep = a.E + a.S, Kp = a.k + a.S;
  const long R = (long)a.T * Kp;
  const long c0 = (long)blockIdx.x * kRouteChunk, c1 = (c0 + kRouteChunk < R) ? c0 + kRouteChunk : R;
  warp_histograms(a, c0, c1, hist);
  if (threadIdx.x < Ep) {
    int run = a.chunk_base[(size_t)blockIdx.x * Ep + threadIdx.x];
    for (int w = 0; w < 32; ++w) {
      const int c = hist[w * Ep + threadIdx.x];
      hist[w * Ep + threadIdx.x] = run;
      run += c;
    }
  }
  __syncthreads();
  place_slots(a, c0, c1, hist);
}

// One warp per (token, column chunk of 32 x CW 16-byte pieces): the chunk of
// the token's FP8 row is read once and written to each of the token's pool
// rows in expert-sorted order (the local form of the pages' L1 pool fill);
// the first chunk's warp also copies the scale row. Disabled slots (pool row
// -1) are skipped. Long calls take 4 KB chunks per warp (CW = 8), short ones
// 1 KB chunks (CW = 2) so that enough warps run.
constexpr int kGatherRowsMin = 512;
template <int CW>
__global__ void __launch_bounds__(256) gather_kernel(GatherArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int vec = a.H / 16, sfw = a.H / 128;
  const int nch = (vec + 32 * CW - 1) / (32 * CW);
  const long items = (long)a.T * nch;
  for (long item = gw; item < items; item += nw) {
    const long t = item / nch;
    const int i0 = (int)(item - t * nch) * 32 * CW + lane;
    int dst[kMaxSlots];
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) dst[j] = j < a.Kp ? __ldg(a.pos + t * a.Kp + j) : -1;
    const uint4* __restrict__ src = reinterpret_cast<const uint4*>(a.x + t * a.H);
    uint4 v[CW];
#pragma unroll
    for (int c = 0; c < CW; ++c)
      if (i0 + 32 * c < vec) v[c] = __ldg(src + i0 + 32 * c);
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
      if (dst[j] < 0) continue;
      uint4* __restrict__ d = reinterpret_cast<uint4*>(a.pool_x + (size_t)dst[j] * a.H);
#pragma unroll
      for (int c = 0; c < CW; ++c)
        if (i0 + 32 * c < vec) d[i0 + 32 * c] = v[c];
    }
    if (i0 >= 32) continue;  // the scale row: the token's first chunk
    const uint32_t* ss = reinterpret_cast<const uint32_t*>(a.x_sf + t * (a.H / 32));
    uint32_t sv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (lane + 32 * c < sfw) sv[c] = __ldg(ss + lane + 32 * c);
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
      if (dst[j] < 0) continue;
      uint32_t* ds = reinterpret_cast<uint32_t*>(a.pool_sf + (size_t)dst[j] * (a.H / 32));
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (lane + 32 * c < sfw) ds[lane + 32 * c] = sv[c];
    }
  }
}

// Each thread owns one 16-byte column chunk (8 BF16 values) of one token: it
// issues the loads of all the token's slot rows first, then sums them in FP32
// in slot order and stores the BF16 result. MS (8, or kMaxSlots above eight
// slots per token) sizes the per-thread slot arrays, so that the common
// top-8 case keeps its registers low and more threads in flight; the slot
// rows are read once, so their loads skip L1.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
template <int MS>
__global__ void __launch_bounds__(128) combine_kernel(CombineArgs a) {
  pdl_trigger();
  pdl_wait();
  const int chunks = a.H / 8;
  const long total = (long)a.T * chunks;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const long t = i / chunks;
    const int c = (int)(i - t * chunks);
    uint4 v[MS];
    int r[MS];
#pragma unroll
    for (int j = 0; j < MS; ++j) {
      r[j] = j < a.Kp ? __ldg(a.pos + t * a.Kp + j) : -1;
      v[j] = r[j] >= 0 ? ld_stream(reinterpret_cast<const uint4*>(a.z + (size_t)r[j] * a.H) + c) : make_uint4(0, 0, 0, 0);
    }
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
    for (int j = 0; j < MS; ++j) {
      if (r[j] < 0) continue;
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] += __uint_as_float(w[e] << 16);
        acc[2 * e + 1] += __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * e]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * e + 1]));
      o[e] = lo | (hi << 16);
    }
    reinterpret_cast<uint4*>(a.out + (size_t)t * a.H)[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// splitmix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014): the i-th output of the stream `seed`.
__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Checks the SiLU division against the IEEE operations on this GPU.
// counts[0]: significands of y in [1, 2) (all 2^23) whose refined reciprocal
//            differs from __frcp_rn(y);
// counts[1]: pairs with a normal IEEE quotient where div_ge1 differs from
//            __fdiv_rn;
// counts[2]: pairs with a subnormal or zero IEEE quotient where they differ;
// counts[3]: pairs checked;
// counts[4]: pairs where they differ by more than one unit in the last place.
// x: any finite float (random sign, exponent field 0..254 and significand);
// y: half the pairs a random significand times 2^(0..127) (so [1, 2^128)),
// half 1 + e with e = a random significand times 2^(-40..129) (up to +inf).
__global__ void div_check_kernel(unsigned long long n, unsigned long long seed, unsigned long long* counts) {
  const unsigned long long tid = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  const unsigned long long nth = (unsigned long long)gridDim.x * blockDim.x;
  unsigned long long c0 = 0, c1 = 0, c2 = 0, c3 = 0, c4 = 0;
  for (unsigned long long m = tid; m < (1ull << 23); m += nth) {
    const float y = __uint_as_float(0x3F800000u | (uint32_t)m);
    if (__float_as_uint(rcp_newton(y)) != __float_as_uint(__frcp_rn(y))) ++c0;
  }
  for (unsigned long long i = tid; i < n; i += nth) {
    const uint64_t h = splitmix64(seed, i);
    const uint32_t hx = (uint32_t)h, hy = (uint32_t)(h >> 32);
    uint32_t xe = (hx >> 23) & 0xFFu;
    if (xe == 0xFFu) xe = 0xFEu;
    const float x = __uint_as_float((hx & 0x807FFFFFu) | (xe << 23));
    const float sig = __uint_as_float(0x3F800000u | (hy & 0x7FFFFFu));
    float y;
    if (hy >> 31) {
      y = ldexpf(sig, (int)((hy >> 23) & 0x7Fu));
    } else {
      const int k = (int)((hy >> 23) & 0xFFu) % 170 - 40;  // 128, 129: 1 + e = +inf
      y = __fadd_rn(1.0f, ldexpf(sig, k));
    }
    const float a = div_ge1(x, y), b = __fdiv_rn(x, y);
    const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
    ++c3;
    if (ua != ub) {
      if (fabsf(b) >= 0x1p-126f) ++c1;
      else ++c2;
      const uint32_t d = ua > ub ? ua - ub : ub - ua;
      if (((ua ^ ub) >> 31) != 0u ? (ua & 0x7FFFFFFFu) + (ub & 0x7FFFFFFFu) > 1u : d > 1u) ++c4;
    }
  }
  if (c0) atomicAdd(&counts[0], c0);
  if (c1) atomicAdd(&counts[1], c1);
  if (c2) atomicAdd(&counts[2], c2);
  atomicAdd(&counts[3], c3);
  if (c4) atomicAdd(&counts[4], c4);
}

// Waits on an mbarrier nobody arrives on, with the same bounded wait the GEMM
// pipeline uses, and records the expiry in the status word.
__global__ void timeout_probe_kernel(uint32_t* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, timeout_ns, 7);
  __syncthreads();
}

}  // namespace mm

extern "C" int mm_route_launches(int slots) { return slots <= mm::kRouteSingleMax ? 1 : 3; }

extern "C" int mm_launch_route(const mm::RouteArgs* a, void* stream) {
  const int Ep = a->E + a->S;
  const long R = (long)a->T * (a->k + a->S);
  static bool attr_set = false;
  if (!attr_set) {
    const int big = (int)(sizeof(int) * (32 * mm::kMaxExperts + 72));
    cudaError_t e = cudaFuncSetAttribute(mm::route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mm::route_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (e != cudaSuccess) return (int)e;
    attr_set = true;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (R <= mm::kRouteSmallMax) {
    // the first kernel of a forward: ordinary stream order behind the previous work
    return (int)mm::launch_kernel(mm::route_small_kernel, dim3(1), dim3(1024), 0, st, false, *a);
  }
  if (R <= mm::kRouteSingleMax) {
    // the first kernel of a forward: ordinary stream order behind the previous work
    return (int)mm::launch_kernel(mm::route_kernel, dim3(1), dim3(1024), sizeof(int) * (32 * (size_t)Ep + 72), st,
                                  false, *a);
  }
  const int G = (int)((R + mm::kRouteChunk - 1) / mm::kRouteChunk);
  cudaError_t e = mm::launch_kernel(mm::route_count_kernel, dim3(G), dim3(1024), sizeof(int) * (size_t)Ep, st, false,
                                    *a);
  if (e == cudaSuccess) e = mm::launch_kernel(mm::route_scan_kernel, dim3(1), dim3(1024), 0, st, true, *a, G);
  if (e == cudaSuccess)
    e = mm::launch_kernel(mm::route_place_kernel, dim3(G), dim3(1024), sizeof(int) * 32 * (size_t)Ep, st, true, *a);
  return (int)e;
}

namespace mm {
// Weight-scale transform (the SM100 weight transform's scale transpose): one
// warp per (128-row block, K step of 128); lane l gathers the step's four
// scale bytes of rows l, l + 32, l + 64 and l + 96 of the block and stores
// them as its 16 bytes of the block's 512-byte piece (the layout the grouped
// GEMM's scale warp would otherwise build in shared memory).
__global__ void __launch_bounds__(256) transform_sf_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                           long blocks, int K) {
  const int lane = threadIdx.x & 31;
  const long gw = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long nw = ((long)gridDim.x * blockDim.x) >> 5;
  const int steps = K / 128, ld = K / 32;
  for (long p = gw; p < blocks * steps; p += nw) {
    const long b = p / steps;
    const int ks = (int)(p - b * steps);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = __ldg(reinterpret_cast<const uint32_t*>(src + (b * 128 + 32 * i + lane) * ld + 4 * ks));
    *reinterpret_cast<uint4*>(dst + p * 512 + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
}  // namespace mm

extern "C" int mm_launch_transform_sf(const uint8_t* src, uint8_t* dst, long blocks, int K, void* stream) {
  const long warps = blocks * (K / 128);
  if (warps <= 0) return 0;
  long grid = (warps + 7) / 8;
  if (grid > 152 * 16) grid = 152 * 16;
  return (int)mm::launch_kernel(mm::transform_sf_kernel, dim3((unsigned)grid), dim3(256), 0, (cudaStream_t)stream,
                                false, src, dst, blocks, K);
}

extern "C" int mm_launch_gather(const mm::GatherArgs* a, void* stream) {
  if (a->T <= 0) return 0;
  // 4 KB chunks per warp from kGatherRowsMin tokens up, else 1 KB chunks
  const bool rows = a->T >= mm::kGatherRowsMin;
  const int per = 32 * (rows ? 8 : 2);
  const long items = (long)a->T * ((a->H / 16 + per - 1) / per);
  long blocks = (items + 7) / 8;  // eight warps per block
  if (blocks > 152 * 16) blocks = 152 * 16;
  return (int)(rows ? mm::launch_kernel(mm::gather_kernel<8>, dim3((unsigned)blocks), dim3(256), 0,
                                        (cudaStream_t)stream, true, *a)
                    : mm::launch_kernel(mm::gather_kernel<2>, dim3((unsigned)blocks), dim3(256), 0,
                                        (cudaStream_t)stream, true, *a));
}

extern "C" int mm_launch_combine(const mm::CombineArgs* a, void* stream, bool pdl) {
  if (a->T <= 0) return 0;
  const long threads = (long)a->T * (a->H / 8);
  long blocks = (threads + 127) / 128;
  if (blocks > 152 * 32) blocks = 152 * 32;
  return (int)(a->Kp <= 8 ? mm::launch_kernel(mm::combine_kernel<8>, dim3((unsigned)blocks), dim3(128), 0,
                                              (cudaStream_t)stream, pdl, *a)
                          : mm::launch_kernel(mm::combine_kernel<mm::kMaxSlots>, dim3((unsigned)blocks), dim3(128), 0,
                                              (cudaStream_t)stream, pdl, *a));
}

extern "C" int mm_launch_div_check(unsigned long long pairs, unsigned long long seed, unsigned long long* counts,
                                   void* stream) {
  mm::div_check_kernel<<<152 * 4, 256, 0, (cudaStream_t)stream>>>(pairs, seed, counts);
  return (int)cudaGetLastError();
}

extern "C" int mm_launch_timeout_probe(uint32_t* status, unsigned long long timeout_ns, void* stream) {
  mm::timeout_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, timeout_ns);
  return (int)cudaGetLastError();
}
