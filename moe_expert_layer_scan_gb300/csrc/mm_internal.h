// Internal host/device definitions shared by the MegaMoE CUDA translation units:
// workspace layout, kernel argument blocks and tile-shape constants.
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>

#include "../../include/megamoe.h"

namespace mm {

constexpr int kMaxExperts = 1024;  // E + S
constexpr int kMaxSlots = 16;      // topk + S
constexpr int kRowMargin = 256;    // pool rows beyond the last valid row that tiles may touch
constexpr int kRouteChunk = 8192;  // slots per CTA when routing runs on several CTAs
constexpr int kRouteSingleMax = 16384;  // up to this many slots, one CTA routes everything
constexpr int kRouteSmallMax = 512;     // up to this many slots, the lean one-CTA routing kernel
// Scheduling words of a forward, zeroed by the routing kernel: the tile
// counters of the persistent GEMM launches (0: the L1 or fused launch, 1: the
// L2 launch of the split schedule) and the number of heavy experts (those
// with more than one token tile; the tile order puts them first).
constexpr int kSchedCounters = 8;
constexpr int kSchedHeavyExperts = 4;
// Per-expert tile widths (two concurrent launches, one per expert class): the
// heavy experts' tiles run 224 tokens wide on kSchedHeavyCtas of the SMs, the
// others 112 wide on the rest; counters 0/1 are the light class's L1/L2
// launches, 2/3 the heavy class's. The routing kernel splits the SMs in
// proportion to each class's tiles weighted by their measured relative cost
// (a heavy 224-token tile computes up to twice the rows of a light tile).
constexpr int kSchedHeavyCtas = 5;
constexpr int kCostHeavyTile = 3, kCostLightTile = 2;

// Token-tile widths (the largest MMA N) of the GEMM variants. "small" serves
// decode-like calls (few rows per expert), "large" and "wide" everything else;
// an expert's rows are split into equal tiles (rounded up to 16 rows) and the
// MMA N of a tile is its rows rounded up to 16, so ragged tails never pay for
// a full tile.
constexpr int kBnSmall = 16;
constexpr int kBnLarge = 112;
// 224-token tiles: one MMA of N up to 224 per K step and weight block keeps
// the tensor pipe busy (two 112-wide MMAs cost two instruction issues for the
// same work); their two 224-column accumulators fill TMEM, so there is one
// accumulator buffer. For the compute-bound calls with many rows per expert.
constexpr int kBnWide = 224;
// 64-token tiles: the MMA shape and epilogue of the 112-token tiles with a
// smaller token box, which leaves room for a fifth pipeline stage (more weight
// bytes in flight) when the call has at most kDeepMaxExperts experts. For the
// weight-bandwidth bound calls with a few dozen rows per expert.
constexpr int kBnMid = 64;
// 16-token tiles run six pipeline stages (instead of five), and 64-token tiles
// exist at all (five stages), when the call has at most this many experts
// (E + S): the smaller tile tables and fewer scale groups make room.
constexpr int kDeepMaxExperts = 300;
// 16-token tiles with four 128-row weight blocks per tile (two gate/up pairs in
// L1, four W2 blocks in L2) and four MMA-issuing warps: twice the MMA issue
// capacity per weight byte, which is what limits the two-block tiles when they
// stream E4M3 weights. Three 66 KB stages; the tile tables fit for at most
// this many experts (E + S), and I must be a multiple of 256.
constexpr int kQuadMaxExperts = 264;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Byte offsets of every workspace region for one (shape, T).
struct Layout {
  size_t status, sched, counts, offsets, tiles_l1, tiles_l2, eorder, rank_offsets, perm, pos, row_w, chunk_cnt,
      chunk_base, chunk_bad, ready;
  size_t pool_x, pool_sf, l2a, l2a_sf, z, total;
  int rows_cap;
};

inline Layout make_layout(int E, int S, int H, int I, int k, int T) {
  Layout L{};
  const int Ep = E + S, Kp = k + S;
  const size_t R = (size_t)T * Kp;
  L.rows_cap = (int)R + kRowMargin;
  size_t o = 0;
  auto take = [&](size_t bytes, size_t align) { o = align_up(o, align); size_t at = o; o += bytes; return at; };
  L.status = take(256, 256);
  L.sched = take(sizeof(int32_t) * kSchedCounters, 256);
  L.counts = take(sizeof(int32_t) * Ep, 256);
  L.offsets = take(sizeof(int32_t) * (Ep + 1), 256);
  L.tiles_l1 = take(sizeof(int32_t) * (Ep + 2), 256);
  L.tiles_l2 = take(sizeof(int32_t) * (Ep + 2), 256);
  L.eorder = take(sizeof(int32_t) * Ep, 256);
  L.rank_offsets = take(sizeof(int32_t) * (E + 1), 256);
  L.perm = take(sizeof(int32_t) * (R + 1), 256);
  L.pos = take(sizeof(int32_t) * (R + 1), 256);
  L.row_w = take(sizeof(float) * (R + 1), 256);
  const size_t G = (R + kRouteChunk - 1) / kRouteChunk + 1;
  L.chunk_cnt = take(sizeof(int32_t) * G * Ep, 256);
  L.chunk_base = take(sizeof(int32_t) * G * Ep, 256);
  L.chunk_bad = take(sizeof(int32_t) * G, 256);
  L.ready = take(sizeof(int32_t) * (R + 1), 256);
  L.pool_x = take((size_t)L.rows_cap * H, 1024);
  L.pool_sf = take((size_t)L.rows_cap * (H / 32), 1024);
  L.l2a = take((size_t)L.rows_cap * I, 1024);
  L.l2a_sf = take((size_t)L.rows_cap * (I / 32), 1024);
  L.z = take((size_t)L.rows_cap * H * 2, 1024);
  L.total = align_up(o, 1024);
  return L;
}

struct RouteArgs {
  const int32_t* topk_idx;
  const float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  // Tile tables in tile order: the experts with more than one token tile
  // ("heavy") first, then the others, each in expert order; eorder[j] is the
  // expert at position j, tiles_*[j] the first tile of position j,
  // tiles_*[Ep] the tile count and tiles_*[Ep + 1] the heavy experts' tiles.
  int32_t* tiles_l1;
  int32_t* tiles_l2;
  int32_t* eorder;
  int32_t* perm;
  int32_t* pos;
  float* row_w;
  uint32_t* status;
  int32_t* chunk_cnt;   // [G][E+S] per-chunk expert counts (multi-CTA routing)
  int32_t* chunk_base;  // [G][E+S] first pool row of each chunk's slots per expert
  int32_t* chunk_bad;   // [G] out-of-range ids seen in the chunk
  int32_t* ready;       // [R + 1] arrival counters of the fused GEMM, zeroed here
  int32_t* sched;       // [kSchedCounters] tile counters of the GEMM launches, zeroed here
  int T, E, k, S;
  int bn_l1, bn_l2;  // token-tile widths of the two GEMMs (per-expert widths: of the light experts)
  int bn_heavy;      // token-tile width of the heavy experts (bn_l1 unless the widths are per expert)
  int dual_sms;      // per-expert widths: the SMs to split between the two classes (0: one class)
  int fb_l1, fb_l2;  // weight tiles per expert: I/128 (gate/up pairs) and ceil(H/256)
  // expert-parallel-ready outputs: the routed experts split over ep_ranks
  // destination ranks in contiguous blocks; rank_offsets[g] = first sorted row
  // bound for rank g ([ep_ranks + 1]); stats (optional, caller-owned [E + S])
  // accumulates every call's rows per expert
  int32_t* rank_offsets;
  int32_t* stats;
  int ep_ranks;
};

struct GatherArgs {
  const uint8_t* x;
  const uint8_t* x_sf;
  const int32_t* pos;  // [T * Kp] pool row of each slot, -1 if disabled
  uint8_t* pool_x;
  uint8_t* pool_sf;
  int T, H, Kp;
};

struct GemmArgs {
  const uint8_t* w_sf;        // [Ep * rows_w][K/32] UE8M0
  const uint8_t* act_sf;      // [rows_cap][K/32]     UE8M0
  const int32_t* offsets;     // [Ep + 1]
  const int32_t* tile_start;  // [Ep + 2] in tile order (see RouteArgs)
  const int32_t* eorder;      // [Ep] expert at each tile-order position
  const float* row_w;         // L1: top-k weight per pool row
  uint8_t* out_q;             // L1: [rows_cap][I] E4M3
  uint8_t* out_sf;            // L1: [rows_cap][I/32] UE8M0
  uint16_t* out_z;            // L2: [rows_cap][H] BF16
  uint32_t* status;
  int Ep, K, rows_w, I, H;
  int fb_total;  // weight tiles per expert (L1: I/128 gate/up pairs, L2: ceil(H/256) block pairs)
  float clamp;
  int fast_math;
  int w_sf_vec, act_sf_vec;  // scale rows allow 16-byte loads (16-byte aligned base and row stride)
  unsigned long long timeout_ns;
  // Fused L1 -> L2 launch: ready[row0] counts the L1 epilogue warps that have
  // stored their part of the token tile starting at pool row row0; the L2
  // tiles of that token tile wait for ready_target arrivals.
  int32_t* ready;
  int ready_target;
  int w_fp8;  // weights are E4M3 (one byte per element) instead of packed E2M1
  int32_t* tile_ctr;  // this launch's tile counter (zero at launch): CTAs claim tiles in index order
  // 0: every tile of the phase; 1: the light experts' tiles only, on the CTAs
  // below (grid - sched[kSchedHeavyCtas]); 2: the heavy experts' tiles only,
  // on the CTAs below sched[kSchedHeavyCtas] (per-expert tile widths)
  int tile_class;
  const int32_t* sched;  // the forward's scheduling words (kSched*)
  int sf_tma;  // scale rows are loaded by TMA (every K a multiple of 512, 16-byte aligned scale tensors)
  // with sf_tma: the transformed weight scales (mm_transform_weight_scales),
  // 512 bytes per 128-row block and K step in the tcgen05.cp layout, or null
  const uint8_t* w_sf_t;
};

// Tensor maps of one GEMM launch (L1 and L2; a single-linear launch repeats its
// own): weights, activations, weight scales, activation scales.
struct GemmMaps {
  CUtensorMap w1, a1, w2, a2;
  CUtensorMap wsf1, asf1, wsf2, asf2;
  // 224-token tiles: token boxes of 112 and 32 rows for the narrower tiles
  // (the CTA-pair launches load each CTA's half of a token tile with the
  // 112-row boxes)
  CUtensorMap a1n, a2n, a1s, a2s;
  // CTA-pair L1 launches: W1 rows and W1 scale rows in boxes of 64 rows (each
  // CTA's A block is 64 gate rows and the matching 64 up rows)
  CUtensorMap w1h, wsf1h;
};

struct CombineArgs {
  const uint16_t* z;
  const int32_t* pos;
  uint16_t* out;
  int T, H, Kp;
};

}  // namespace mm

// Kernel launchers (one translation unit each); return cudaError_t as int.
extern "C" {
int mm_launch_route(const mm::RouteArgs* a, void* stream);
int mm_route_launches(int slots);  // kernels mm_launch_route enqueues for this many slots
int mm_launch_gather(const mm::GatherArgs* a, void* stream);
// Weight-scale transform: for `blocks` 128-row blocks of a UE8M0 scale tensor
// with K/32 bytes per row, the 512-byte tcgen05.cp piece of every (block, K
// step of 128) into dst, block-major.
int mm_launch_transform_sf(const uint8_t* src, uint8_t* dst, long blocks, int K, void* stream);
int mm_launch_combine(const mm::CombineArgs* a, void* stream, bool pdl);
// variant: 0 = small tiles, 1 = large tiles, 2 = small tiles with six stages
// (E + S <= kDeepMaxExperts), 3 = 224-token tiles, 4 = small tiles with four
// weight blocks (E + S <= kQuadMaxExperts, I % 256 == 0), 5 = 64-token tiles
// (E + S <= kDeepMaxExperts). maps: the launch's tensor maps (a
// single-linear launch reads w1/a1/wsf1/asf1 for L1 and w2/a2/wsf2/asf2 for L2).
int mm_launch_gemm(int l1, int variant, const mm::GemmMaps* maps, const mm::GemmArgs* a, int num_ctas, void* stream);
// A single-linear launch of the 112- or 224-token tiles (variant 1 or 3) in
// ordinary stream order (no programmatic serialisation): the per-expert-width
// launches, which must not hold SMs early.
int mm_launch_gemm_class(int l1, int variant, const mm::GemmMaps* maps, const mm::GemmArgs* a, void* stream);
// One persistent launch of both GEMMs: every L1 tile, then every L2 tile; an L2
// tile starts once the L1 epilogues of its token tile have arrived on `ready`.
int mm_launch_gemm_fused(int variant, const mm::GemmMaps* maps, const mm::GemmArgs* g1, const mm::GemmArgs* g2,
                         void* stream);
// 224-token tiles of the split schedule on CTA pairs (clusters of two CTAs,
// M = 256 MMAs): each tile covers 256 weight rows (L1: 128 features' gate and
// up rows; L2: two 128-row W2 blocks) and every CTA double-buffers its
// 224-column accumulator, so the epilogue of one tile runs under the MMAs of
// the next. Needs the scale rows by TMA (sf_tma) and an even grid.
int mm_launch_gemm_pair(int l1, const mm::GemmMaps* maps, const mm::GemmArgs* a, void* stream);
int mm_pair_prepare(void);  // shared-memory limits and the launch size (CTAs of the clusters resident at once)
int mm_pair_ctas(void);     // CTAs per CTA-pair launch (0: unavailable)
int mm_gemm_prepare(void);  // sets the dynamic shared-memory limits and the persistent grid sizes
int mm_gemm_blocks(int variant);   // 128-row weight blocks per tile (2 or 4)
int mm_gemm_epilogue_warps(int variant);  // epilogue warps per CTA (arrivals per L1 tile in the fused schedule)
int mm_gemm_token_scale_box_rows(int variant);  // token rows per TMA box of the token scale rows
int mm_launch_timeout_probe(uint32_t* status, unsigned long long timeout_ns, void* stream);
int mm_launch_div_check(unsigned long long pairs, unsigned long long seed, unsigned long long* counts, void* stream);
}
