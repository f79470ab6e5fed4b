// Persistent grouped GEMM over experts for the two linears of the MegaMoE
// expert path, on 5th-generation tensor cores (tcgen05, kind::mxf8f6f4 with
// UE8M0 block scales, FP32 accumulators in TMEM).
//
//   L1 ("MegaMoE research report" sec. 4.1, Linear1 phase):
//     acc[n, r] = sum_k W1[e, n, k] * x[r, k] for the gate rows n and the
//     matching up rows I + n of the tile's 128-row feature blocks, then the
//     fused epilogue y = silu(clamp(gate)) * clamp(up) * w_r, per (row, 32
//     columns) amax -> UE8M0 scale (smallest power of two >= amax/448) -> E4M3
//     ("MEGAMOE_SM90_DESIGN" sec. 10.1, steps 2-5; UE8M0 per the SM100 kernel).
//   L2 (Linear2 phase; sec. 11.1): acc[h, r] = sum_i W2[e, h, i] * q[r, i]
//     for the tile's consecutive 128-row blocks of W2, written as BF16 into
//     the per-slot row r.
//
// Orientation: the weights are the MMA's M=128 operand (E2M1, read by TMA as
// 16 x 4-bit groups padded to 16 bytes in SMEM; or E4M3 weights, one byte per
// element, the same 128-byte SMEM rows) and the expert's token rows are
// the N operand (E4M3), N = the tile's rows rounded up to 16. One CTA per SM
// walks a flat list of (expert, weight blocks, token tile) tiles; an expert's
// rows are split into equal token tiles of at most BN (16, 64, 112 or 224) rows.
//
// Warp roles: warp 0 = TMA producer; one MMA-issuing warp per weight block of
// a tile (NA = 2: warps 1 and 2; NA = 4 adds warps 4 + EPI and 5 + EPI), one
// thread each, since one warp issues only about one block-scaled MMA per 125
// cycles (warp 2 also allocates TMEM); warp 3 = scale rows into the
// tcgen05.cp layout and their copies into TMEM; warps 4 .. 4 + EPI - 1 =
// epilogue (warp w reads TMEM lanes 32*(w%4)..+31, i.e. 32 consecutive weight
// rows; with eight or twelve of them the warps of a quadrant take turns over
// the column chunks of the token tile).
// Pipelines: STAGES shared-memory stages (full/empty mbarriers) and two TMEM
// accumulator buffers (tmem_full/tmem_empty) so the epilogue of one tile
// overlaps the main loop of the next; the 224-token tiles fill TMEM with one
// buffer. Every wait is bounded.
//
// Modes: one launch per linear (L1, L2), or both in one persistent launch
// (fused, the arrival-mask scheme of the research report's Linear1 -> Linear2
// hand-off): the tile list is every L1 tile followed by every L2 tile; each L1
// epilogue warp publishes its stores and counts itself on its token tile's
// arrival counter, and the loads of an L2 tile start once that counter is
// complete. Every CTA finishes its own L1 tiles before its first L2 tile and
// the persistent grid is co-resident, so the waits always end.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "mm_common.cuh"
#include "mm_internal.h"
#include "mm_ptx.cuh"

namespace mm {

// Epilogue warps: one per TMEM lane quadrant for the 16-column decode tiles,
// two for the 64- and 112-token tiles (their L1 epilogue is as long as the
// main loop), three for the 224-token tiles, whose epilogue runs between tiles
// (measured against two: prefill L2 GEMM 1.69 -> 1.61 ms; four were slower,
// at 96 registers a thread).
// One MMA-issuing warp per weight block of a tile (NA of them): warp 0 is the
// producer, warps 1 and 2 issue for blocks 0 and 1 (warp 2 also allocates
// TMEM), warp 3 handles the scales, warps 4 .. 4 + EPI - 1 are the epilogue
// and warps 4 + EPI .. issue for blocks 2 .. NA - 1.
template <int BN, int NA>
struct Warps {
  static constexpr int EPI = BN > 112 ? 12 : BN > 16 ? 8 : 4;
  static constexpr int THREADS = 32 * (2 + NA + EPI);
};

enum : int { kModeL2 = 0, kModeL1 = 1, kModeFused = 2 };

// PROMO: the float-scale FP8 recipe (E4M3 weights with a float32 scale per
// 128 x 128 block, activations with a float32 scale per (row, 128)). The
// block-scaled MMA reads only power-of-two scales, so each 128-long K block
// is an unscaled kind::f8f6f4 partial sum in TMEM (one buffer per stage); the
// epilogue warps multiply it by (activation scale x weight scale) and add it
// to their FP32 registers ("MEGAMOE_SM90_DESIGN" sec. 5.3, scale factors
// applied in software after the MMA), then store the sum into the tile's
// accumulator columns for the usual epilogue.
template <int BN, int STAGES, int NA_ = 2, bool PROMO = false>
struct GemmCfg {
  static constexpr int BM = 128;                         // weight rows per MMA
  static constexpr int BK = 128;                         // K per stage
  // NA 128-row weight blocks per stage (2 or 4): L1 the gate rows of NA / 2
  // feature blocks and the matching up rows; L2 NA consecutive 128-row blocks
  // of W2 (the last ones may be absent at the end of H).
  static constexpr int NA = NA_;
  static constexpr int NI = NA;                          // MMA-issuing threads, one per weight tile
  static constexpr int A_BYTES = BM * BK;                // 16 KB in SMEM (4-bit codes padded to bytes)
  static constexpr int A_TX = BM * BK / 2;               // transaction bytes of one weight box (packed 4-bit size)
  static constexpr int B_BYTES = BN * BK;
  static constexpr int SFB_ROWS = BN <= 128 ? 128 : 256;
  static constexpr int SF_STAGE_BYTES = PROMO ? 0 : NA * 512 + SFB_ROWS * 4;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * NA * A_BYTES;
  static constexpr int SF_OFF = B_OFF + STAGES * B_BYTES;
  static constexpr int BAR_OFF = SF_OFF + STAGES * SF_STAGE_BYTES;
  static constexpr int RAW_G_MAX = 3;  // scale-row groups in flight (RAW_G below) at most
  // The deep configurations (16-token tiles with six stages, 64-token tiles
  // with five) keep room for them by supporting at most kDeepMaxExperts
  // experts and two scale groups in flight.
  static constexpr bool DEEP = (BN == kBnSmall && STAGES > 5) || (BN == kBnMid && STAGES > 4);
  // tiles handed from the producer to the other warps: a ring of RING tile
  // indices with a full/empty mbarrier pair per slot; every role except the
  // producer consumes each tile once (the scale warp, the MMA issuers and the
  // epilogue warps)
  static constexpr int RING = 4;
  // accumulator barrier pairs (tfull / tempty): the two accumulator buffers,
  // or PROMO's partial-sum buffers, one per stage (the K block in stage s
  // accumulates into buffer s, so the stage's empty barrier also tells the
  // epilogue that the partial sum is complete)
  static constexpr int NTB = PROMO ? STAGES : 2;
  static constexpr int CONSUMERS = 1 + NI + Warps<BN, NA_>::EPI;
  // barriers (full, empty, sfready per stage; two accumulator pairs; the raw
  // scale groups' pair; the ring's pair per slot), the TMEM address, the abort
  // flag and the tile ring, rounded up to 16 bytes
  // (PROMO: eight more, the L1 epilogue's exchange of per-quadrant amax values)
  static constexpr int XBARS = PROMO ? 8 : 0;
  static constexpr int BAR_BYTES =
      ((3 * STAGES + 2 * NTB + 2 * RAW_G_MAX + 2 * RING + XBARS) * 8 + 8 + 4 * RING + 15) / 16 * 16;
  // TMA-loaded scale rows: RAW_G groups of four K steps; per group 16 bytes of
  // each of 128 rows for each weight block and of RAW_B_ROWS token rows
  static constexpr int RAW_G = PROMO ? 1 : DEEP || NA > 2 ? 2 : 3;  // (PROMO: unused, kept well-formed)
  static_assert(RAW_G <= RAW_G_MAX, "barrier region sized for RAW_G_MAX groups");
  static constexpr int RAW_ROWS_BYTES = 128 * 16;
  static constexpr int RAW_B_ROWS = BN <= 32 ? 32 : (BN <= 128 ? 128 : 256);
  static constexpr int RAW_B_BYTES = RAW_B_ROWS * 16;
  static constexpr int RAW_GROUP_BYTES = NA * RAW_ROWS_BYTES + RAW_B_BYTES;
  // PROMO: per-quadrant column maxima exchanged by the L1 epilogue warps,
  // [2 buffers][2 warp halves][4 quadrants][32 columns] floats, then each
  // epilogue warp's scale products of one K block ([blocks][columns] floats,
  // at most 2 x 32 for a warp)
  static constexpr int XA_EXCH_BYTES = 2 * 2 * 4 * 32 * 4;
  static constexpr int XA_BYTES = PROMO ? XA_EXCH_BYTES + 16 + 8 * 64 * 4 : 0;  // (+16: alignment of the products)
  // copies of the two tile tables and the row offsets ([experts + 1] each),
  // and, where shared memory has room, of the tile-order expert list
  static constexpr int TAB_OFF = BAR_OFF + BAR_BYTES;
  static constexpr int TAB_INTS = (NA > 2 ? kQuadMaxExperts : DEEP ? kDeepMaxExperts : kMaxExperts) + 1;
  static constexpr int smem_with(int tables) {
    return ((TAB_OFF + tables * TAB_INTS * 4 + 16 + XA_BYTES + 127) / 128 * 128) + RAW_G * RAW_GROUP_BYTES + 1024;
  }
  static constexpr bool EO_SMEM = smem_with(4) <= 232448;
  // L2 tiles whose L1 rows the producer has seen stored (fused schedule)
  static constexpr int L2RDY_OFF = TAB_OFF + (EO_SMEM ? 4 : 3) * TAB_INTS * 4;
  static constexpr int XA_OFF = L2RDY_OFF + 16;
  static constexpr int PS_OFF = (XA_OFF + XA_EXCH_BYTES + 15) / 16 * 16;  // PROMO: the scale products (16-byte aligned)
  static constexpr int RAW_OFF = (XA_OFF + XA_BYTES + 127) / 128 * 128;
  static constexpr int SMEM_BYTES = RAW_OFF + RAW_G * RAW_GROUP_BYTES + 1024;  // + alignment slack
  // TMEM columns: the accumulator buffers, then one scale-factor slot per
  // stage (every scale-factor address stays a multiple of 4 columns)
  static constexpr int ACC_COLS = NA * BN;
  // per stage: 4 columns of scales per weight block, then the token tile's
  // (4 per 128 rows), shared by both MMA streams
  static constexpr int SF_STAGE_COLS = 4 * NA + SFB_ROWS / 32;
  // Two accumulator buffers (the epilogue of one tile overlaps the main loop
  // of the next) where TMEM holds them; the 224-token tiles fill TMEM with one
  // and the epilogue drains it between tiles.
  // PROMO: one accumulator region (each epilogue warp writes and then reads
  // only its own columns) and a partial-sum buffer per stage after it, no
  // scale slots.
  static constexpr int ACC_BUFS = PROMO ? 1 : 2 * ACC_COLS + STAGES * SF_STAGE_COLS <= 512 ? 2 : 1;
  static constexpr int SF_BASE = ACC_BUFS * ACC_COLS;
  static constexpr int PART_BASE = ACC_COLS;
  // HALF: with one accumulator buffer (224-token tiles), a tile of at most
  // HALF_N rows needs only half of it (its two blocks at HALF_N columns
  // apart), so such narrow tiles alternate between the two halves and the
  // epilogue of one overlaps the main loop of the next; a wider tile takes
  // both halves.
  static constexpr bool HALF = !PROMO && ACC_BUFS == 1;
  static constexpr int HALF_N = BN / 2;
  static constexpr int TMEM_USED = PROMO ? (1 + NTB) * ACC_COLS : SF_BASE + STAGES * SF_STAGE_COLS;
  static_assert(!PROMO || NTB == STAGES, "PROMO: a partial-sum buffer per stage");
  static_assert(!PROMO || (NA == 2 && (BN == 16 || BN == 64)), "promotion: 16- and 64-token two-block tiles");
  static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256 : 512;
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(!PROMO || Warps<BN, NA_>::EPI * NA * (BN / 16 / (Warps<BN, NA_>::EPI / 4)) * 16 * 4 <= 8 * 64 * 4,
                "PROMO: the scale products fit their region");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(BN <= RAW_B_ROWS, "every token row of a tile has its scale row in the raw group");
  static_assert(B_BYTES % 1024 == 0, "B tiles must keep 1024-byte alignment");
  static_assert(BN % 8 == 0, "token tiles are whole 8-row swizzle atoms");
};

// The per-phase arguments a role needs for one tile, selected field by field
// from the L1 or L2 argument block (each a constant-bank read).
struct Phase {
  const uint8_t* w_sf;
  const uint8_t* w_sf_t;  // transformed weight scales (512 bytes per 128-row block and K step), or null
  const uint8_t* act_sf;
  int K, rows_w, second, w_sf_vec, act_sf_vec;
  bool l1;
};
__device__ __forceinline__ Phase phase_of(bool l1, const GemmArgs& g1, const GemmArgs& g2) {
  Phase p;
  p.l1 = l1;
  p.w_sf = l1 ? g1.w_sf : g2.w_sf;
  p.w_sf_t = l1 ? g1.w_sf_t : g2.w_sf_t;
  p.act_sf = l1 ? g1.act_sf : g2.act_sf;
  p.K = l1 ? g1.K : g2.K;
  p.rows_w = l1 ? g1.rows_w : g2.rows_w;
  p.second = g1.I;  // L1: row offset of the up rows from the gate rows
  p.w_sf_vec = l1 ? g1.w_sf_vec : g2.w_sf_vec;
  p.act_sf_vec = l1 ? g1.act_sf_vec : g2.act_sf_vec;
  return p;
}

// First weight row of weight block u of a tile with na blocks, and whether it
// exists. L1: block 2j holds the gate rows of the tile's j-th 128-row feature
// block, block 2j + 1 the matching up rows (I rows further); L2: na
// consecutive 128-row blocks of W2, the last ones absent at the end of H.
__device__ __forceinline__ int block_wrow(const Phase& p, const Tile& t, int u, int na) {
  return p.l1 ? t.e * p.rows_w + (t.fb * (na / 2) + (u >> 1)) * 128 + (u & 1) * p.second
              : t.e * p.rows_w + (t.fb * na + u) * 128;
}
__device__ __forceinline__ bool block_active(const Phase& p, const Tile& t, int u, int na) {
  return t.active && (p.l1 || (t.fb * na + u) * 128 < p.rows_w);
}

// Four K steps of one row's UE8M0 scales (16 bytes); `avail` steps exist.
// fresh: the bytes were written by other CTAs during this launch, so the load
// bypasses L1 (ld.global.cg) instead of using the read-only path.
__device__ __forceinline__ uint4 load_sf4(const uint8_t* p, bool vec16, int avail, bool fresh) {
  if (vec16) return fresh ? __ldcg(reinterpret_cast<const uint4*>(p)) : __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t* q = reinterpret_cast<const uint32_t*>(p);
  auto ld = [fresh](const uint32_t* x) { return fresh ? __ldcg(x) : __ldg(x); };
  uint4 r = make_uint4(ld(q), 0u, 0u, 0u);
  if (avail > 1) r.y = ld(q + 1);
  if (avail > 2) r.z = ld(q + 2);
  if (avail > 3) r.w = ld(q + 3);
  return r;
}

template <int MODE, int BN, int STAGES, int NA, bool PROMO>
__global__ void __launch_bounds__(Warps<BN, NA>::THREADS, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs g1,
                const __grid_constant__ GemmArgs g2) {
  using C = GemmCfg<BN, STAGES, NA, PROMO>;
  using W = Warps<BN, NA>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + C::NTB;
  uint64_t* sfready = tempty + C::NTB;      // [STAGES] a stage's scales are in TMEM (tcgen05.commit of the copies)
  uint64_t* rfull = sfready + STAGES;  // [RAW_G] TMA scale rows landed
  uint64_t* rempty = rfull + C::RAW_G;  // [RAW_G] scale warp done with a group
  uint64_t* tr_full = rempty + C::RAW_G;  // [RING] a tile index is in the ring slot
  uint64_t* tr_empty = tr_full + C::RING;  // [RING] every consumer has read the slot
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tr_empty + C::RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* tring = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [RING] tile indices
  // PROMO: amax exchange barriers [buffer * 2 + half]: written by the four
  // quadrant warps of a half, and read by them
  uint64_t* xwrit = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF + C::BAR_BYTES - 8 * C::XBARS);
  uint64_t* xread = xwrit + C::XBARS / 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);     // TMA expect_tx arrival
      mbar_init(&sfready[s], 1);  // the scale warp's tcgen05.commit
      mbar_init(&empty[s], C::NI);  // one tcgen05.commit per issuing thread
    }
    for (int b = 0; b < C::NTB; ++b) {
      mbar_init(&tfull[b], C::NI);  // tcgen05.commit after the last K step, per issuing thread
      mbar_init(&tempty[b], W::EPI);  // one arrival per epilogue warp
    }
    for (int b = 0; b < C::RAW_G; ++b) {
      mbar_init(&rfull[b], 1);   // producer's expect_tx arrival
      mbar_init(&rempty[b], 1);  // scale warp, lane 0
    }
    for (int b = 0; b < C::RING; ++b) {
      mbar_init(&tr_full[b], 1);              // the producer's arrival after writing the index
      mbar_init(&tr_empty[b], C::CONSUMERS);  // one arrival per consuming warp
    }
    for (int b = 0; b < C::XBARS; ++b) mbar_init(&xwrit[b], 4);  // (xread follows xwrit) four quadrant warps
    *abort_flag = 0;
    *reinterpret_cast<int*>(smem + C::L2RDY_OFF) = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (MODE != kModeL2) {
      prefetch_tmap(&maps.w1);
      prefetch_tmap(&maps.a1);
    }
    if (MODE != kModeL1) {
      prefetch_tmap(&maps.w2);
      prefetch_tmap(&maps.a2);
    }
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the prologue above overlaps the previous kernel; its outputs are read below
  pdl_trigger();
  pdl_wait();
  int* s_t1 = reinterpret_cast<int*>(smem + C::TAB_OFF);  // L1 tile table
  int* s_t2 = s_t1 + C::TAB_INTS;                         // L2 tile table
  int* s_off = s_t2 + C::TAB_INTS;                        // row offsets per expert
  int* s_eo = s_off + C::TAB_INTS;                        // tile-order expert list (EO_SMEM)
  {
    const GemmArgs& ga = MODE == kModeL2 ? g2 : g1;
    for (int i = threadIdx.x; i <= ga.Ep; i += blockDim.x) {
      if (MODE != kModeL2) s_t1[i] = g1.tile_start[i];
      if (MODE != kModeL1) s_t2[i] = g2.tile_start[i];
      s_off[i] = ga.offsets[i];
      if (C::EO_SMEM && i < ga.Ep) s_eo[i] = ga.eorder[i];
    }
  }
  __syncthreads();
  // the tile order is the expert order when every expert is heavy or none is
  const int nheavy = g1.sched[kSchedHeavyExperts];
  const int32_t* eord = nheavy == 0 || nheavy == g1.Ep ? nullptr : C::EO_SMEM ? s_eo : g1.eorder;
  const uint32_t tmem = *tmem_slot;
  // tiles [0, n1) are L1 tiles, [n1, num_tiles) L2 tiles
  const int n1 = MODE == kModeL2 ? 0 : s_t1[g1.Ep];
  const int num_tiles = MODE == kModeL1 ? n1 : n1 + s_t2[g2.Ep];
  auto is_l1 = [&](int tile) { return MODE == kModeL1 || (MODE == kModeFused && tile < n1); };
  // flat tile index -> tile of its phase
  auto tile_of = [&](int tile, bool l1) {
    return decode_tile(l1 ? tile : tile - n1, l1 ? s_t1 : s_t2, eord, s_off, g1.Ep,
                       l1 ? g1.fb_total : g2.fb_total, BN);
  };
  // Per-expert tile widths (split schedule): this launch serves one class of
  // experts, the heavy ones (tiles [0, h) of the phase, on the first
  // sched[kSchedHeavyCtas] CTAs) or the others (tiles [h, end), on the CTAs
  // below grid - sched[kSchedHeavyCtas]); the other CTAs leave at once, so the
  // two classes' launches share the SMs.
  int t_lo = 0, t_hi = num_tiles;
  bool cta_serves = true;
  if (g1.tile_class != 0) {
    const int h = g1.tile_start[g1.Ep + 1];  // (single-linear launch: g1 is its own phase)
    const int heavy_ctas = g1.sched[kSchedHeavyCtas];
    if (g1.tile_class == 2) {
      t_hi = h;
      cta_serves = (int)blockIdx.x < heavy_ctas;
    } else {
      t_lo = h;
      cta_serves = (int)blockIdx.x < (int)gridDim.x - heavy_ctas;
    }
  }
  // wait site of the tile ring (status bit 8 + 15)
  constexpr uint32_t kSiteRing = 15u;
  // Dynamic tile schedule: the producer claims tiles from the launch's
  // counter (zeroed by the routing kernel), in increasing index order across
  // all CTAs, and hands each to the other roles through the tile ring. Tiles
  // claimed at about the same time are adjacent (concurrent CTAs share weight
  // blocks through L2), CTAs that finish early take more, and in the fused
  // schedule every L1 tile is claimed, by a running CTA, before any L2 tile:
  // an L2 tile only waits for L1 tiles that running CTAs hold and finish
  // without waiting on anything, so the waits end whether or not the whole
  // grid is resident at once.
  // Consumer side: the next tile of this CTA, num_tiles or more when there are
  // no more, -1 when the wait gave up. whole_warp: all 32 lanes call it (else
  // one thread). Each consumer takes its next tile early, during the current
  // one (the producer publishes it during the current tile's second stage),
  // so that the hand-off stays off the path between two tiles.
  auto take_tile = [&](uint32_t& n, bool whole_warp) -> int {
    const int slot = (int)(n % C::RING);
    const uint32_t ph = (n / C::RING) & 1u;
    if (!mbar_wait(&tr_full[slot], ph, abort_flag, g1.status, g1.timeout_ns, kSiteRing, 0)) return -1;
    const int t = tring[slot];
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) mbar_arrive(&tr_empty[slot]);
    ++n;
    return t;
  };
  // wait sites reported in the status word on expiry: L1 tiles s, L2 tiles 8 + s
  constexpr uint32_t kSiteReady = 8u + 6u;  // an L2 tile waiting for its L1 rows (fused)
  int* l2rdy = reinterpret_cast<int*>(smem + C::L2RDY_OFF);
  // scale rows by TMA (else the scale warp loads them from global memory)
  const bool sf_tma = g1.sf_tma != 0;
  // The scale warp's lane 0 copies a stage's scales from the SMEM layout into
  // the stage's TMEM slot (the weight blocks' and the token tile's, the latter
  // shared by both MMA streams) and commits the copies to sfready[s]; the MMA
  // threads then issue only MMAs. The slot is free once empty[s] completed.
  // (the weight blocks' 512-byte pieces at wsrc + u * wstride: the stage's
  // scale slot, or a raw group holding transformed weight scales)
  auto copy_scales = [&](int s, uint32_t amask, const uint8_t* sF, const uint8_t* wsrc, int wstride) {
    tc_fence_after();
    const uint32_t slot = tmem + (uint32_t)(C::SF_BASE + s * C::SF_STAGE_COLS);
#pragma unroll
    for (int u = 0; u < C::NA; ++u)
      if ((amask >> u) & 1u) tc_cp_32x128b_warpx4(slot + 4u * u, sdesc_sf_32x16(smem_u32(wsrc + wstride * u)));
#pragma unroll
    for (int gq = 0; gq < C::SFB_ROWS / 128; ++gq)
      tc_cp_32x128b_warpx4(slot + 4u * C::NA + 4u * gq, sdesc_sf_32x16(smem_u32(sF + C::NA * 512 + gq * 512)));
    tc_commit(&sfready[s]);
  };

  // the tile's existing weight blocks (bit u) and their first rows
  auto block_mask = [&](const Phase& ph, const Tile& t) {
    uint32_t m = 0;
#pragma unroll
    for (int u = 0; u < C::NA; ++u)
      if (block_active(ph, t, u, C::NA)) m |= 1u << u;
    return m;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Fused: an L2 tile's loads start once its arrival counter is complete.
    // The counter of the next L2 tile is peeked early (after the first stage of
    // the current tile) so that the wait is usually over before the tile
    // starts; every observation is handed on to the scale-factor warp
    // (l2rdy counts this CTA's L2 tiles observed ready, in tile order).
    uint32_t it = 0, gi = 0, pub = 0;  // stages, scale groups and ring slots issued
    bool ok = true;
    bool cur_ready = false;  // the current tile's counter was seen complete by a peek
    // transaction bytes of one 128x128 weight box: packed E2M1 or E4M3
    const uint32_t a_tx = g1.w_fp8 ? (uint32_t)(C::BM * C::BK) : (uint32_t)C::A_TX;
    // claim: lane 0's atomic on the launch's tile counter; two claims are in
    // flight (the next tile's and the one after), each read a whole tile after
    // it was issued, so the atomic's round trip never stalls the loads.
    // publish: the index into the next ring slot once every consumer has read
    // its old one. (A claimed tile is always processed by this running CTA
    // after its current one, and claims rise monotonically, so an L2 tile is
    // never claimed ahead of an L1 tile a running CTA still has to claim.)
    int claim_a = 0, claim_b = 0;
    bool next_in_a = true;  // which of the two holds the next tile's claim
    auto claim = [&](int& c) {
      if (lane == 0) c = cta_serves ? t_lo + atomicAdd(g1.tile_ctr, 1) : t_hi;
    };
    auto publish = [&](int c) -> int {
      int t = __shfl_sync(0xffffffffu, c, 0);
      if (t >= t_hi) t = num_tiles;  // no more tiles of this launch
      const int slot = (int)(pub % C::RING);
      const uint32_t ph = (pub / C::RING) & 1u;
      if (!mbar_wait(&tr_empty[slot], ph ^ 1u, abort_flag, g1.status, g1.timeout_ns, kSiteRing)) return -1;
      if (lane == 0) {
        tring[slot] = t;
        mbar_arrive(&tr_full[slot]);
      }
      __syncwarp();
      ++pub;
      return t;
    };
    claim(claim_a);
    int tile = publish(claim_a);
    claim(claim_a);  // the second tile, in flight during the first
    ok = tile >= 0;
    // the next tile's index: published during the current tile's second stage
    auto publish_next = [&]() -> int {
      const int t = next_in_a ? publish(claim_a) : publish(claim_b);
      next_in_a = !next_in_a;
      return t;
    };
    while (ok && tile < num_tiles) {
      const bool l1 = is_l1(tile);
      const Phase g = phase_of(l1, g1, g2);
      const uint32_t site0 = l1 ? 0u : 8u;
      const Tile t = tile_of(tile, l1);
      const uint32_t amask = block_mask(g, t);
      const int nact = __popc(amask);
      const int kblocks = g.K / C::BK;
      const CUtensorMap* tw = l1 ? &maps.w1 : &maps.w2;
      // the token box: the smallest of the launch's boxes that holds the tile
      const int brows = !C::HALF ? BN : t.nrows <= 32 ? 32 : t.nrows <= C::HALF_N ? C::HALF_N : BN;
      const CUtensorMap* ta = !C::HALF || brows == BN ? (l1 ? &maps.a1 : &maps.a2)
                              : brows == 32 ? (l1 ? &maps.a1s : &maps.a2s)
                                            : (l1 ? &maps.a1n : &maps.a2n);
      const CUtensorMap* twsf = l1 ? &maps.wsf1 : &maps.wsf2;
      const CUtensorMap* tasf = l1 ? &maps.asf1 : &maps.asf2;
      if (MODE == kModeFused && !l1 && !cur_ready &&
          counter_ready_relay(g1.ready + t.row0, g1.ready_target, true, l2rdy, abort_flag, g1.status,
                              g1.timeout_ns, kSiteReady) != 1) {
        ok = false;
        break;
      }
      bool next_ready = false;
      int ntile = -1;  // the next tile, claimed during this one's first stage and published at its second
      for (int kb = 0; kb < kblocks; ++kb, ++it) {
        if (!PROMO && sf_tma && (kb & 3) == 0) {
          // this group's scale rows (16 bytes = four K steps per row) into a raw slot
          const int gslot = (int)(gi % C::RAW_G);
          const uint32_t gph = (gi / C::RAW_G) & 1u;
          if (!mbar_wait(&rempty[gslot], gph ^ 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 0)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            uint8_t* raw = smem + C::RAW_OFF + gslot * C::RAW_GROUP_BYTES;
            mbar_arrive_expect_tx(&rfull[gslot], nact * C::RAW_ROWS_BYTES + C::RAW_B_BYTES);
#pragma unroll
            for (int u = 0; u < C::NA; ++u)
              if ((amask >> u) & 1u) {
                if (g.w_sf_t)  // transformed: the group's four 512-byte pieces are contiguous
                  bulk_load(raw + u * C::RAW_ROWS_BYTES,
                            g.w_sf_t + ((size_t)(block_wrow(g, t, u, C::NA) / 128) * kblocks + kb) * 512,
                            (uint32_t)C::RAW_ROWS_BYTES, &rfull[gslot]);
                else
                  tma_load_2d(raw + u * C::RAW_ROWS_BYTES, twsf, &rfull[gslot], kb * 4, block_wrow(g, t, u, C::NA));
              }
            tma_load_2d(raw + C::NA * C::RAW_ROWS_BYTES, tasf, &rfull[gslot], kb * 4, t.row0);
          }
          ++gi;
        }
        if (kb == 1) {
          ntile = publish_next();
          if (ntile < 0) { ok = false; break; }
          // fused: peek at the next L2 tile's counter (usually complete by the time it starts)
          if (MODE == kModeFused && ntile < num_tiles && !is_l1(ntile)) {
            const Tile tn = tile_of(ntile, false);
            next_ready = counter_ready_relay(g1.ready + tn.row0, g1.ready_target, false, l2rdy, abort_flag,
                                             g1.status, g1.timeout_ns, kSiteReady) == 1;
          }
        }
        const int s = (int)(it % STAGES);
        const uint32_t ph = (it / STAGES) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 0)) { ok = false; break; }
        uint8_t* sA = smem + C::A_OFF + s * C::NA * C::A_BYTES;
        uint8_t* sB = smem + C::B_OFF + s * C::B_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], (uint32_t)nact * a_tx + (uint32_t)(brows * C::BK));
#pragma unroll
          for (int u = 0; u < C::NA; ++u)
            if ((amask >> u) & 1u) tma_load_2d(sA + u * C::A_BYTES, tw, &full[s], kb * C::BK, block_wrow(g, t, u, C::NA));
          tma_load_2d(sB, ta, &full[s], kb * C::BK, t.row0);
        }
        if (kb == 0) {  // the tile after next
          if (next_in_a) claim(claim_b);
          else claim(claim_a);
        }
      }
      if (!ok) break;
      if (kblocks == 1) {
        ntile = publish_next();
        if (ntile < 0) { ok = false; break; }
      }
      cur_ready = next_ready;
      tile = ntile;
    }
    const GemmArgs& gl = MODE == kModeL1 ? g1 : g2;  // status word and limit (shared by both)
    constexpr uint32_t kSiteTail = (MODE == kModeL1 ? 0u : 8u) + 4u;
    if (!ok) {
      // Let the copies already issued land before the CTA can exit (the
      // stage's barrier may never complete if another role gave up, so the
      // limit here is short).
      const uint32_t issued = it;
      for (uint32_t j = (issued > (uint32_t)STAGES ? issued - STAGES : 0u); j < issued; ++j) {
        int dummy = 0;
        mbar_wait(&full[j % STAGES], (j / STAGES) & 1u, reinterpret_cast<volatile int*>(&dummy), gl.status,
                  gl.timeout_ns < 10000000ull ? gl.timeout_ns : 10000000ull, kSiteTail);
      }
    }
  } else if (warp == 3 && !PROMO && sf_tma) {
    // ------------------------------------------------------------ scale-factor transposer
    // The producer TMA-loads each group's scale rows (16 bytes = four K steps
    // per row) into a raw slot; per K step this warp writes the layout
    // tcgen05.cp.32x128b.warpx4 reads: 16 bytes per lane l holding the step's
    // four scale bytes of rows l, l+32, l+64, l+96 of each 128-row group.
    constexpr int NB = C::SFB_ROWS / 32;
    uint32_t it = 0, gi = 0, tn = 0;
    bool ok = true;
    int tile = take_tile(tn, true);
    while (tile >= 0 && tile < num_tiles) {
      int next = -2;  // the next tile, taken after this tile's first scale group
      const bool l1 = is_l1(tile);
      const Phase g = phase_of(l1, g1, g2);
      const uint32_t site0 = l1 ? 0u : 8u;
      const Tile t = tile_of(tile, l1);
      const uint32_t amask = block_mask(g, t);
      const int nb = (t.nrows + 31) / 32;
      const int kblocks = g.K / C::BK;
      const bool tw = g.w_sf_t != nullptr;  // weight scales arrive already laid out (read in place by the copies)
      for (int kg = 0; kg < kblocks && ok; kg += 4, ++gi) {
        const int gslot = (int)(gi % C::RAW_G);
        const uint32_t gph = (gi / C::RAW_G) & 1u;
        if (!mbar_wait(&rfull[gslot], gph, abort_flag, g1.status, g1.timeout_ns, site0 + 5)) { ok = false; break; }
        const uint8_t* raw = smem + C::RAW_OFF + gslot * C::RAW_GROUP_BYTES;
        uint4 wa[C::NA][4], wb[NB];
#pragma unroll
        for (int op = 0; op < C::NA; ++op)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            wa[op][i] = ((amask >> op) & 1u) && !tw
                            ? *reinterpret_cast<const uint4*>(raw + op * C::RAW_ROWS_BYTES + (32 * i + lane) * 16)
                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < NB; ++j)
          wb[j] = (j < nb && 32 * j < C::RAW_B_ROWS)
                      ? *reinterpret_cast<const uint4*>(raw + C::NA * C::RAW_ROWS_BYTES + (32 * j + lane) * 16)
                      : make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
        // the raw slot may be refilled (transformed weight scales: once the
        // group's copies, which read them in place, have completed)
        if (lane == 0 && !tw) mbar_arrive(&rempty[gslot]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int s = (int)(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 5)) { ok = false; break; }
          uint8_t* sF = smem + C::SF_OFF + s * C::SF_STAGE_BYTES;
          if (!tw) {
#pragma unroll
            for (int op = 0; op < C::NA; ++op)
              st_shared_v4(sF + op * 512 + lane * 16, word(wa[op][0], c), word(wa[op][1], c), word(wa[op][2], c),
                           word(wa[op][3], c));
          }
#pragma unroll
          for (int q = 0; q < NB / 4; ++q)
            st_shared_v4(sF + C::NA * 512 + q * 512 + lane * 16, word(wb[4 * q], c), word(wb[4 * q + 1], c),
                         word(wb[4 * q + 2], c), word(wb[4 * q + 3], c));
          fence_proxy_async_smem();  // generic-proxy writes, read next by tcgen05.cp
          __syncwarp();
          if (lane == 0) {
            if (tw)
              copy_scales(s, amask, sF, raw + c * 512, C::RAW_ROWS_BYTES);
            else
              copy_scales(s, amask, sF, sF, 512);
          }
          ++it;
        }
        if (lane == 0 && tw) tc_commit(&rempty[gslot]);  // after the group's copies complete
        if (ok && kg == 0) next = take_tile(tn, true);
      }
      if (!ok) break;
      tile = next == -2 ? take_tile(tn, true) : next;
    }
  } else if (warp == 3 && !PROMO && C::NA == 2) {
    // ------------------------------------------------------------ scale-factor producer
    // (tiles of two weight blocks only: the host runs four-block tiles only
    // with TMA-loaded scale rows)
    // Loads each row's UE8M0 bytes for a group of four K steps at once (one
    // 16-byte request per row) and, per K step, writes the layout
    // tcgen05.cp.32x128b.warpx4 reads: 16 bytes per lane l holding the step's
    // four scale bytes of rows l, l+32, l+64, l+96 of each 128-row group.
    // The warp walks the flattened (tile, group) sequence and issues the loads
    // of the next group before it stores the current one, so their latency
    // overlaps four pipeline stages instead of stalling the ring.
    constexpr int NB = C::SFB_ROWS / 32;  // 32-row blocks of the token operand
    uint4 ca[C::NA][4], cb[NB];           // current group
    uint4 xa[C::NA][4], xb[NB];           // next group
    auto load_group = [&](int tile, int kg, uint4(&wa)[C::NA][4], uint4(&wb)[NB]) {
      const bool l1 = is_l1(tile);
      const Phase g = phase_of(l1, g1, g2);
      const Tile t = tile_of(tile, l1);
      const uint32_t amask = block_mask(g, t);
      const int nb = (t.nrows + 31) / 32;
      const int sf_ld = g.K / 32;
      const int avail = g.K / C::BK - kg;
      const bool fresh = MODE == kModeFused && !l1;  // token scales written by this launch's L1 tiles
      const bool wvec = g.w_sf_vec && avail >= 4, bvec = g.act_sf_vec && avail >= 4;
#pragma unroll
      for (int op = 0; op < C::NA; ++op)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          wa[op][i] = ((amask >> op) & 1u)
                          ? load_sf4(g.w_sf + (size_t)(block_wrow(g, t, op, C::NA) + 32 * i + lane) * sf_ld + 4 * kg,
                                     wvec, avail, false)
                          : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < NB; ++j)
        wb[j] = j < nb ? load_sf4(g.act_sf + (size_t)(t.row0 + 32 * j + lane) * sf_ld + 4 * kg, bvec, avail, fresh)
                       : make_uint4(0u, 0u, 0u, 0u);
    };
    // fused: an L2 tile's token scales are read only once the producer has
    // seen its L1 rows stored (the producer counts its L2 tiles in l2rdy;
    // both warps walk the same tiles, so this warp's n-th L2 tile waits for n)
    int l2seen = 0;
    auto ready_wait = [&](int tile) {
      if (MODE != kModeFused || is_l1(tile)) return true;
      return wait_shared_counter(l2rdy, ++l2seen, abort_flag, g1.status, g1.timeout_ns, kSiteReady);
    };
    uint32_t it = 0, tn = 0;
    int tile = take_tile(tn, true), kg = 0;
    bool ok = tile >= 0;
    if (ok && tile < num_tiles) {
      ok = ready_wait(tile);
      if (ok) load_group(tile, kg, ca, cb);
    }
    while (ok && tile < num_tiles) {
      const bool l1 = is_l1(tile);
      const Phase g = phase_of(l1, g1, g2);
      const uint32_t site0 = l1 ? 0u : 8u;
      const int kblocks = g.K / C::BK;
      const int avail = kblocks - kg;
      const Tile tc = tile_of(tile, l1);
      const uint32_t cur_mask = block_mask(g, tc);
      int ntile = tile, nkg = kg + 4;
      if (nkg >= kblocks) {
        ntile = take_tile(tn, true);  // published by the producer during this tile's first stages
        nkg = 0;
        if (ntile < 0) break;
      }
      const bool has_next = ntile < num_tiles;
      // a next group whose L1 rows are not all stored yet is loaded after this
      // group is stored (its rows may come from this CTA's own tile in flight)
      bool next_waits = false;
      if (MODE == kModeFused && has_next && nkg == 0 && !is_l1(ntile)) {
        int done = 0;
        if (lane == 0) done = ld_acquire_cta_shared(l2rdy) > l2seen;
        next_waits = !__shfl_sync(0xffffffffu, done, 0);
        __syncwarp();
        if (!next_waits) ++l2seen;
      }
      if (has_next && !next_waits) load_group(ntile, nkg, xa, xb);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c >= avail) break;
        const int s = (int)(it % STAGES);
        const uint32_t ph = (it / STAGES) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 5)) { ok = false; break; }
        uint8_t* sF = smem + C::SF_OFF + s * C::SF_STAGE_BYTES;
#pragma unroll
        for (int op = 0; op < C::NA; ++op)
          st_shared_v4(sF + op * 512 + lane * 16, word(ca[op][0], c), word(ca[op][1], c), word(ca[op][2], c),
                       word(ca[op][3], c));
#pragma unroll
        for (int q = 0; q < NB / 4; ++q)
          st_shared_v4(sF + C::NA * 512 + q * 512 + lane * 16, word(cb[4 * q], c), word(cb[4 * q + 1], c),
                       word(cb[4 * q + 2], c), word(cb[4 * q + 3], c));
        fence_proxy_async_smem();  // generic-proxy writes, read next by tcgen05.cp
        __syncwarp();
        if (lane == 0) copy_scales(s, cur_mask, sF, sF, 512);
        ++it;
      }
      if (!ok || !has_next) break;
      if (next_waits) {
        if (!ready_wait(ntile)) break;
        load_group(ntile, nkg, xa, xb);
      }
#pragma unroll
      for (int op = 0; op < C::NA; ++op)
#pragma unroll
        for (int i = 0; i < 4; ++i) ca[op][i] = xa[op][i];
#pragma unroll
      for (int j = 0; j < NB; ++j) cb[j] = xb[j];
      tile = ntile;
      kg = nkg;
    }
  } else if (warp == 3) {
    // (float-scale tiles have no UE8M0 scales to stage; four-block tiles
    // always take their scale rows by TMA. This warp still consumes the ring
    // so that every slot is released.)
    uint32_t tn = 0;
    for (;;) {
      const int tile = take_tile(tn, true);
      if (tile < 0 || tile >= num_tiles) break;
    }
  } else if (warp == 1 || warp == 2 || warp >= 4 + W::EPI) {
    // ------------------------------------------------------------ MMA issuers
    // One thread per weight block (warps 1, 2, then 4 + EPI ...): one warp
    // issues about one block-scaled MMA per 125 cycles, so the instruction
    // stream of a K step is split between them. Each commits its own work (a
    // missing last L2 block still commits, so the barrier counts hold).
    if (lane == 0) {
      const int u = warp <= 2 ? warp - 1 : warp - (4 + W::EPI) + 2;
      // A (weights): E2M1 (format 5) or E4M3 (format 0); B (tokens): E4M3
      const uint32_t a_fmt = g1.w_fp8 ? 0u : 5u;
      uint32_t it = 0, tcount = 0, tn = 0, pk = 0;  // pk: K blocks issued (PROMO partial buffers)
      uint32_t hc0 = 0, hc1 = 0, nt = 0;  // HALF: uses of each half, the next narrow tile's half
      bool ok = true;
      int tile = take_tile(tn, false);
      for (;; ++tcount) {
        if (tile < 0 || tile >= num_tiles) break;
        int next = -2;  // the next tile, taken after this tile's first K step
        const bool l1 = is_l1(tile);
        const Phase g = phase_of(l1, g1, g2);
        const uint32_t site0 = l1 ? 0u : 8u;
        const Tile t = tile_of(tile, l1);
        const int kblocks = g.K / C::BK;
        if constexpr (PROMO) {
          // one unscaled partial sum per K block into partial buffer pk % NTB (= its stage)
          const uint32_t n_mma = (uint32_t)((t.nrows + 15) & ~15);
          const bool active = block_active(g, t, u, C::NA);
          const uint32_t id = idesc_f8f6f4_e4m3(n_mma);
          for (int kb = 0; kb < kblocks; ++kb, ++it, ++pk) {
            const int s = (int)(it % STAGES);
            const uint32_t ph = (it / STAGES) & 1u;
            const int pb = (int)(pk % (uint32_t)C::NTB);
            if (!mbar_wait(&full[s], ph, abort_flag, g1.status, g1.timeout_ns, site0 + 2)) { ok = false; break; }
            if (!mbar_wait(&tempty[pb], ((pk / (uint32_t)C::NTB) & 1u) ^ 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (active) {
              const uint32_t d = tmem + (uint32_t)(C::PART_BASE + pb * C::ACC_COLS + u * BN);
              const uint64_t da = sdesc_kmajor_sw128(smem_u32(smem + C::A_OFF + (s * C::NA + u) * C::A_BYTES));
              const uint64_t db = sdesc_kmajor_sw128(smem_u32(smem + C::B_OFF + s * C::B_BYTES));
#pragma unroll
              for (int k = 0; k < 4; ++k) tc_mma_f8f6f4(d, da + 2u * k, db + 2u * k, id, k > 0 ? 1u : 0u);
            }
            // one commit: the stage is free and partial sum pb (= s) is complete
            tc_commit(&empty[s]);
            if (kb == 0) next = take_tile(tn, false);
          }
          if (!ok) break;
          tile = next == -2 ? take_tile(tn, false) : next;
          continue;
        }
        int buf = C::ACC_BUFS == 2 ? (int)(tcount & 1u) : 0;
        uint32_t d;
        const bool narrow = C::HALF && t.nrows <= C::HALF_N;
        if (C::HALF && narrow) {
          buf = (int)nt;
          nt ^= 1u;
          if (!mbar_wait(&tempty[buf], ((buf ? hc1 : hc0) & 1u) ^ 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 1))
            break;
          d = tmem + (uint32_t)(buf * (C::ACC_COLS / 2) + u * C::HALF_N);
        } else if (C::HALF) {
          nt = 0;
          if (!mbar_wait(&tempty[0], (hc0 & 1u) ^ 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 1) ||
              !mbar_wait(&tempty[1], (hc1 & 1u) ^ 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 1))
            break;
          d = tmem + (uint32_t)(u * BN);
        } else {
          const uint32_t bph = (C::ACC_BUFS == 2 ? tcount >> 1 : tcount) & 1u;
          if (!mbar_wait(&tempty[buf], bph ^ 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 1)) break;
          d = tmem + (uint32_t)(buf * C::ACC_COLS + u * BN);
        }
        tc_fence_after();
        const uint32_t n_mma = (uint32_t)((t.nrows + 15) & ~15);
        const bool active = block_active(g, t, u, C::NA);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, abort_flag, g1.status, g1.timeout_ns, site0 + 2)) { ok = false; break; }
          if (!mbar_wait(&sfready[s], ph, abort_flag, g1.status, g1.timeout_ns, site0 + 2)) { ok = false; break; }
          tc_fence_after();
          const uint8_t* sA = smem + C::A_OFF + (s * C::NA + u) * C::A_BYTES;
          const uint8_t* sB = smem + C::B_OFF + s * C::B_BYTES;
          if (active) {
            const uint32_t slot = tmem + (uint32_t)(C::SF_BASE + s * C::SF_STAGE_COLS);
            const uint32_t sfa = slot + 4u * (uint32_t)u;
            const uint32_t sfb = slot + 4u * C::NA;
            const uint64_t da = sdesc_kmajor_sw128(smem_u32(sA));
            const uint64_t db = sdesc_kmajor_sw128(smem_u32(sB));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t id = idesc_mxf8f6f4(a_fmt, 0u, n_mma, (uint32_t)k);
              // +32 bytes of K per step inside the 128-byte swizzle atom (2 in 16-byte units)
              tc_mma_mxf8f6f4(d, da + 2u * k, db + 2u * k, id, sfa, sfb, (kb > 0 || k > 0) ? 1u : 0u);
            }
          }
          tc_commit(&empty[s]);  // the stage is free once these MMAs have read it
          if (kb == 0) next = take_tile(tn, false);
        }
        if (!ok) break;
        if (C::HALF && !narrow) {
          // a wide tile fills both halves: both complete with it
          tc_commit(&tfull[0]);
          tc_commit(&tfull[1]);
          ++hc0;
          ++hc1;
        } else {
          tc_commit(&tfull[buf]);
          if (C::HALF) (buf ? hc1 : hc0) += 1u;
        }
        tile = next == -2 ? take_tile(tn, false) : next;
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + W::EPI) {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM lanes 32*(w%4)..+31 (hardware rule); the two warps of
    // a quadrant take alternate 16-column chunks of the token tile.
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;  // 0 when there is one warp per quadrant
    uint32_t tcount = 0, tn = 0, pk = 0, xc = 0;  // pk, xc: PROMO partial sums and amax exchanges
    uint32_t hc0 = 0, hc1 = 0, nt = 0;             // HALF: as the MMA warps count them
    int tile = take_tile(tn, true);
    for (;; ++tcount) {
      if (tile < 0 || tile >= num_tiles) break;
      const bool l1 = is_l1(tile);
      const Phase g = phase_of(l1, g1, g2);
      const uint32_t site0 = l1 ? 0u : 8u;
      const Tile t = tile_of(tile, l1);
      int buf = C::ACC_BUFS == 2 ? (int)(tcount & 1u) : 0;
      const uint32_t bph = (C::ACC_BUFS == 2 ? tcount >> 1 : tcount) & 1u;
      const uint32_t lanes = (uint32_t)(32 * q) << 16;
      // HALF: a narrow tile's accumulators sit in half `buf` (blocks HALF_N
      // columns apart), a wide tile's in both (blocks BN apart)
      const bool narrow = C::HALF && t.nrows <= C::HALF_N;
      uint32_t acc_base = (uint32_t)(buf * C::ACC_COLS), bstride = BN;
      if (C::HALF && narrow) {
        buf = (int)nt;
        nt ^= 1u;
        acc_base = (uint32_t)(buf * (C::ACC_COLS / 2));
        bstride = C::HALF_N;
      } else if (C::HALF) {
        nt = 0;
      }
      if constexpr (PROMO) {
        // The warp's 16-column chunks are the ones the epilogue below reads:
        // L1 in chunks of 32 (64-token tiles) or 16, L2 in chunks of 16, the
        // warps of a quadrant alternating. Per K block: wait for the partial
        // sum, load it, hand the buffer back, scale and accumulate.
        constexpr int CH = BN / 16 / (W::EPI / 4);
        constexpr int NCL1 = BN > 16 ? 32 : 16;
        auto chunk_col = [&](int i) {
          return l1 ? NCL1 * half + (i / (NCL1 / 16)) * NCL1 * (W::EPI / 4) + 16 * (i % (NCL1 / 16))
                    : 16 * half + i * 16 * (W::EPI / 4);
        };
        const int KB = g.K / C::BK;
        const float* wsf = reinterpret_cast<const float*>(g.w_sf);
        const float* asf = reinterpret_cast<const float*>(g.act_sf);
        // fused L2 tiles: their activation scales are stored during this launch
        // by the L1 epilogues of the token tile, so wait (acquire, bounded) for
        // the tile's arrival counter before reading any of them; this warp may
        // take the tile from the ring before the producer has seen it complete
        const bool fresh = MODE == kModeFused && !l1;
        if (fresh) {
          int rdy = 1;
          if (lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(g1.ready + t.row0) < g1.ready_target) {
              __nanosleep(64);
              if (*abort_flag) { rdy = 0; break; }
              if (globaltimer_ns() - t0 > g1.timeout_ns) {
                *abort_flag = 1;
                atomicOr(g1.status, MM_DEV_TIMEOUT | (1u << (8u + kSiteReady)));
                rdy = 0;
                break;
              }
            }
          }
          rdy = __shfl_sync(0xffffffffu, rdy, 0);
          __syncwarp();  // orders lane 0's acquire before the other lanes' loads
          if (!rdy) break;
        }
        float acc[C::NA][CH][16];
#pragma unroll
        for (int u = 0; u < C::NA; ++u)
#pragma unroll
          for (int i = 0; i < CH; ++i)
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[u][i][j] = 0.0f;
        // Per K block, lane l < 16 * CH owns column chunk_col(l / 16) + l % 16
        // of the warp's columns: it multiplies that column's activation scale
        // by each weight block's scale once and stores the products into the
        // warp's slice of shared memory, from which every lane reads them back
        // 16 at a time (broadcast loads); each partial sum then takes one FMA.
        // The scales are loaded AH K blocks ahead: a ring of AH registers,
        // the K loop unrolled by AH so that each slot is a fixed register.
        constexpr int AH = 4;
        float* ps = reinterpret_cast<float*>(smem + C::PS_OFF) + (warp - 4) * (C::NA * CH * 16);
        const int my_i = lane >> 4;
        const int my_col = my_i < CH ? chunk_col(my_i) + (lane & 15) : 0;
        const bool my_ok = my_i < CH && my_col < t.nrows;
        const float* my_ap = asf + (size_t)(t.row0 + my_col) * KB;
        bool bact[C::NA];
        const float* wsp[C::NA];
#pragma unroll
        for (int u = 0; u < C::NA; ++u) {
          bact[u] = block_active(g, t, u, C::NA);
          wsp[u] = wsf + (size_t)(bact[u] ? block_wrow(g, t, u, C::NA) / 128 : 0) * KB;
        }
        auto ld_sa = [&](int kb) -> float {
          return my_ok && kb < KB ? (fresh ? __ldcg(my_ap + kb) : __ldg(my_ap + kb)) : 0.0f;
        };
        float sa_q[AH];
#pragma unroll
        for (int a = 0; a < AH; ++a) sa_q[a] = ld_sa(a);
        // weight-block scales 32 K blocks at a time: lane l holds K block
        // 32 * group + l (the next group's loaded one group ahead)
        auto ld_sw = [&](int u, int kb) -> float { return bact[u] && kb < KB ? __ldg(wsp[u] + kb) : 0.0f; };
        float sw_c[C::NA], sw_n[C::NA];
#pragma unroll
        for (int u = 0; u < C::NA; ++u) {
          sw_c[u] = ld_sw(u, lane);
          sw_n[u] = ld_sw(u, 32 + lane);
        }
        bool ok = true;
        for (int kb0 = 0; kb0 < KB && ok; kb0 += AH) {
#pragma unroll
         for (int a = 0; a < AH; ++a) {
          const int kb = kb0 + a;
          if (kb >= KB) break;
          // slot a of the ring: this K block's scales out, block kb + AH's in
          const float sa = sa_q[a];
          sa_q[a] = ld_sa(kb + AH);
          if (kb > 0 && (kb & 31) == 0) {
#pragma unroll
            for (int u = 0; u < C::NA; ++u) {
              sw_c[u] = sw_n[u];
              sw_n[u] = ld_sw(u, kb + 32 + lane);
            }
          }
          float sw[C::NA];
#pragma unroll
          for (int u = 0; u < C::NA; ++u) sw[u] = __shfl_sync(0xffffffffu, sw_c[u], kb & 31);
          __syncwarp();  // the previous K block's reads of the slice are done
          if (my_i < CH) {
#pragma unroll
            for (int u = 0; u < C::NA; ++u) ps[(u * CH + my_i) * 16 + (lane & 15)] = __fmul_rn(sa, sw[u]);
          }
          __syncwarp();
          // the partial sum of this K block is complete when its stage's MMAs are
          // (K block pk ran in stage pk % STAGES, into buffer pk % NTB: the same)
          const int pb = (int)(pk % (uint32_t)C::NTB);
          if (!mbar_wait(&empty[pb], (pk / (uint32_t)C::NTB) & 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int u = 0; u < C::NA; ++u) {
            uint32_t r[CH][16];
#pragma unroll
            for (int i = 0; i < CH; ++i)
              if (bact[u] && chunk_col(i) < t.nrows)
                tmem_ld_x16(tmem + lanes + (uint32_t)(C::PART_BASE + pb * C::ACC_COLS + u * BN + chunk_col(i)), r[i]);
            tmem_ld_wait();
            if (u + 1 == C::NA) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty[pb]);  // this partial buffer may be overwritten
            }
#pragma unroll
            for (int i = 0; i < CH; ++i) {
              if (!bact[u] || chunk_col(i) >= t.nrows) continue;  // (warp-uniform)
              const float4* pv = reinterpret_cast<const float4*>(ps + (u * CH + i) * 16);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const float4 sc = pv[v];
                acc[u][i][4 * v + 0] = fmaf(__uint_as_float(r[i][4 * v + 0]), sc.x, acc[u][i][4 * v + 0]);
                acc[u][i][4 * v + 1] = fmaf(__uint_as_float(r[i][4 * v + 1]), sc.y, acc[u][i][4 * v + 1]);
                acc[u][i][4 * v + 2] = fmaf(__uint_as_float(r[i][4 * v + 2]), sc.z, acc[u][i][4 * v + 2]);
                acc[u][i][4 * v + 3] = fmaf(__uint_as_float(r[i][4 * v + 3]), sc.w, acc[u][i][4 * v + 3]);
              }
            }
          }
          ++pk;
         }
        }
        if (!ok) break;
        // columns past the tile's rows (their partial sums are stale TMEM
        // contents times a zero scale) are cleared before the epilogue sees them
#pragma unroll
        for (int u = 0; u < C::NA; ++u)
#pragma unroll
          for (int i = 0; i < CH; ++i)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (chunk_col(i) + j >= t.nrows) acc[u][i][j] = 0.0f;
        // the sums into the accumulator columns the epilogue below reads
#pragma unroll
        for (int u = 0; u < C::NA; ++u)
#pragma unroll
          for (int i = 0; i < CH; ++i)
            if (chunk_col(i) < t.nrows) tmem_st_x16(tmem + lanes + (uint32_t)(u * BN + chunk_col(i)), acc[u][i]);
        tmem_st_wait();
      } else if (C::HALF && !narrow) {
        if (!mbar_wait(&tfull[0], hc0 & 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 3, 256) ||
            !mbar_wait(&tfull[1], hc1 & 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 3, 256))
          break;
      } else {
        const uint32_t ph = C::HALF ? ((buf ? hc1 : hc0) & 1u) : bph;
        if (!mbar_wait(&tfull[buf], ph, abort_flag, g1.status, g1.timeout_ns, site0 + 3, 256)) break;
      }
      // the next tile (published long before this one's accumulator completed)
      const int next = take_tile(tn, true);
      tc_fence_after();
      const uint32_t tbase = tmem + lanes + acc_base;
      if (MODE != kModeL2 && l1) {
        // The per-column amax over the warp's 32 features (one UE8M0 group) is
        // a transpose-reduction: after the exchange steps lane c (32 columns)
        // or lanes 2c, 2c+1 (16 columns) hold the maximum of column c, compute
        // that column's scale once, and the inverse scales are broadcast back.
        // NC = 32 columns per step; 16 for the 16-row decode tiles, and for
        // the 224-row tiles, whose 14 chunks of 16 split evenly between the
        // two warps of a quadrant (7 chunks of 32 would not).
        constexpr int NC = (BN > 16 && BN != 224) ? 32 : 16;
        constexpr int LOG2NC = NC == 32 ? 5 : 4;
        // feature block j of the tile: gate accumulator 2j, up accumulator 2j + 1
        for (int jb = 0; jb < C::NA / 2; ++jb) {
        const uint32_t tg = tbase + 2u * (uint32_t)jb * bstride, tu = tg + bstride;
        const int fblk = t.fb * (C::NA / 2) + jb;  // 128-feature block of the intermediate
        const int feat = fblk * 128 + 32 * q + lane;
        for (int c0 = NC * half; t.active && c0 < t.nrows; c0 += NC * (W::EPI / 4)) {
          const int ncol = min(NC, t.nrows - c0);
          uint32_t gt0[16], gt1[16], u0[16], u1[16];
          tmem_ld_x16(tg + (uint32_t)c0, gt0);
          tmem_ld_x16(tu + (uint32_t)c0, u0);
          if (NC == 32 && ncol > 16) {
            tmem_ld_x16(tg + (uint32_t)(c0 + 16), gt1);
            tmem_ld_x16(tu + (uint32_t)(c0 + 16), u1);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) gt1[j] = u1[j] = 0u;
          }
          tmem_ld_wait();
          const float wl = lane < ncol ? g1.row_w[t.row0 + c0 + lane] : 0.0f;
          float y[NC], v[NC];
#pragma unroll
          for (int j = 0; j < NC; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wl, j);
            float gv = __uint_as_float(j < 16 ? gt0[j] : gt1[j - 16]);
            float uv = __uint_as_float(j < 16 ? u0[j] : u1[j - 16]);
            if (g1.clamp > 0.0f) {
              gv = fminf(fmaxf(gv, -g1.clamp), g1.clamp);
              uv = fminf(fmaxf(uv, -g1.clamp), g1.clamp);
            }
            // silu(g) = g / (1 + exp(-g)); the fast path: __expf and the
            // approximate reciprocal
            const float silu = g1.fast_math ? __fmul_rn(gv, rcp_approx(__fadd_rn(1.0f, __expf(-gv))))
                                            : div_ge1(gv, __fadd_rn(1.0f, expf(-gv)));
            y[j] = j < ncol ? __fmul_rn(__fmul_rn(silu, uv), wj) : 0.0f;
            v[j] = fabsf(y[j]);
          }
          // halve the columns each lane holds at every exchange; with 16
          // columns a last butterfly step pairs lanes 2c and 2c+1
#pragma unroll
          for (int o = 16, n = NC; n > 1; o >>= 1, n >>= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
              const float recv = __shfl_xor_sync(0xffffffffu, upper ? v[i] : v[i + n / 2], o);
              v[i] = fmaxf(upper ? v[i + n / 2] : v[i], recv);
            }
          }
          if (NC == 16) v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
          const int mycol = lane >> (5 - LOG2NC);
          const bool col_lead = (lane & ((1 << (5 - LOG2NC)) - 1)) == 0;
          if constexpr (PROMO) {
            // float scale per (row, 128 features): the maximum over the four
            // quadrant warps of this half (exchanged through shared memory,
            // double-buffered, with bounded barrier waits), amax / 448 by IEEE
            // division (1 when amax is 0), elements E4M3 of y / scale
            const int xb = (int)(xc & 1u), xi = xb * 2 + half;
            float* xa = reinterpret_cast<float*>(smem + C::XA_OFF) + xi * 128;
            if (xc >= 2 &&
                !mbar_wait(&xread[xi], ((xc - 2) >> 1) & 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 3)) break;
            if (col_lead) xa[q * 32 + mycol] = v[0];
            __syncwarp();
            if (lane == 0) mbar_arrive(&xwrit[xi]);
            if (!mbar_wait(&xwrit[xi], (xc >> 1) & 1u, abort_flag, g1.status, g1.timeout_ns, site0 + 3)) break;
            const float am = fmaxf(fmaxf(xa[mycol], xa[32 + mycol]), fmaxf(xa[64 + mycol], xa[96 + mycol]));
            __syncwarp();
            if (lane == 0) mbar_arrive(&xread[xi]);
            ++xc;
            float sc = __fdiv_rn(am, 448.0f);
            if (!(sc > 0.0f)) sc = 1.0f;
            if (q == 0 && col_lead && mycol < ncol)
              reinterpret_cast<float*>(g1.out_sf)[(size_t)(t.row0 + c0 + mycol) * (g1.I / 128) + fblk] = sc;
#pragma unroll
            for (int j = 0; j < NC; ++j) {
              const float sj = __shfl_sync(0xffffffffu, sc, j << (5 - LOG2NC));
              const uint8_t qb = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(y[j], sj), __NV_SATFINITE, __NV_E4M3);
              if (j < ncol) g1.out_q[(size_t)(t.row0 + c0 + j) * g1.I + feat] = qb;
            }
          } else {
          const uint32_t code = requant_code(v[0]);  // column c0 + mycol
          const float inv = inv_scale(code);
          if (col_lead && mycol < ncol)
            g1.out_sf[(size_t)(t.row0 + c0 + mycol) * (g1.I / 32) + fblk * 4 + q] = (uint8_t)code;
          uint32_t qw[NC / 4];
#pragma unroll
          for (int j = 0; j < NC; ++j) {
            const float ij = __shfl_sync(0xffffffffu, inv, j << (5 - LOG2NC));
            const uint32_t qb = (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(y[j], ij), __NV_SATFINITE, __NV_E4M3) & 0xFFu;
            qw[j >> 2] = (j & 3) == 0 ? qb : qw[j >> 2] | (qb << (8 * (j & 3)));
          }
          store_u8_rows_4x4(g1.out_q, (size_t)g1.I, t.row0, c0, ncol, feat - lane, qw);
          }
        }
        }
        // fused: this warp's share of the token tile's L2 operand is stored
        if (MODE == kModeFused && t.active) warp_signal(g1.ready + t.row0);
      } else if (MODE != kModeL1) {
        // W2 blocks 2j and 2j + 1 of the tile: hidden columns feat and feat + 128
        const Phase g2p = phase_of(false, g1, g2);
        for (int jb = 0; jb < C::NA / 2; ++jb) {
        if (!block_active(g2p, t, 2 * jb, C::NA)) break;
        const bool two = block_active(g2p, t, 2 * jb + 1, C::NA);
        const int feat = (t.fb * C::NA + 2 * jb) * 128 + 32 * q + lane;
        const uint32_t tg = tbase + 2u * (uint32_t)jb * bstride, th = tg + bstride;
        for (int c0 = 16 * half; c0 < t.nrows; c0 += 16 * (W::EPI / 4)) {
          uint32_t gv[16], hv[16];
          tmem_ld_x16(tg + (uint32_t)c0, gv);
          tmem_ld_x16(th + (uint32_t)c0, hv);
          tmem_ld_wait();
          // (measured: 8-byte stores after a 4 x 4 lane transpose, or
          // evict-first stores, were no faster than these 64-byte rows)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (col < t.nrows) {
              uint16_t* zr = g2.out_z + (size_t)(t.row0 + col) * g2.H;
              zr[feat] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(gv[j])));
              if (two) zr[feat + 128] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(hv[j])));
            }
          }
        }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (C::HALF && !narrow) {
        if (lane == 0) {
          mbar_arrive(&tempty[0]);
          mbar_arrive(&tempty[1]);
        }
        ++hc0;
        ++hc1;
      } else {
        if (!PROMO && lane == 0) mbar_arrive(&tempty[buf]);
        if (C::HALF) (buf ? hc1 : hc0) += 1u;
      }
      tile = next;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int MODE, int BN, int STAGES, int NA = 2, bool PROMO = false>
static int set_smem_attr(int* max_ctas) {
  using C = GemmCfg<BN, STAGES, NA, PROMO>;
  auto k = gemm_kernel<MODE, BN, STAGES, NA, PROMO>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return (int)e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  *max_ctas = sms;
  return 0;
}

template <int MODE, int BN, int STAGES, int NA = 2, bool PROMO = false>
static int launch(const GemmMaps* maps, const GemmArgs* g1, const GemmArgs* g2, int num_ctas, cudaStream_t st,
                  bool pdl = true) {
  using C = GemmCfg<BN, STAGES, NA, PROMO>;
  return (int)launch_kernel(gemm_kernel<MODE, BN, STAGES, NA, PROMO>, dim3((unsigned)num_ctas),
                            dim3(Warps<BN, NA>::THREADS), C::SMEM_BYTES, st, pdl, *maps, *g1, *g2);
}

// Pipeline depths: as many stages as the 227 KB of shared memory allows (small:
// five, measured as fast as six).
constexpr int kStagesSmall = 5, kStagesSmallDeep = 6, kStagesLarge = 4, kStagesWide = 3, kStagesQuad = 3,
              kStagesMid = 5, kStagesPromoSmall = 5, kStagesPromoMid = 3;
// CTAs per launch of each instantiation: [mode][variant] (variant 2: 16-token
// tiles with six stages, for at most kDeepMaxExperts experts; variant 3:
// 224-token tiles; variant 4: 16-token tiles with four weight blocks, for at
// most kQuadMaxExperts experts; variant 5: 64-token tiles, for at most
// kDeepMaxExperts experts; variants 6 and 7: 16- and 64-token tiles of the
// float-scale recipe)
static int g_ctas[3][8];

}  // namespace mm

extern "C" int mm_gemm_prepare(void) {
  using namespace mm;
  int e = 0;
  if ((e = set_smem_attr<kModeL1, kBnSmall, kStagesSmall>(&g_ctas[kModeL1][0]))) return e;
  if ((e = set_smem_attr<kModeL2, kBnSmall, kStagesSmall>(&g_ctas[kModeL2][0]))) return e;
  if ((e = set_smem_attr<kModeFused, kBnSmall, kStagesSmall>(&g_ctas[kModeFused][0]))) return e;
  if ((e = set_smem_attr<kModeL1, kBnLarge, kStagesLarge>(&g_ctas[kModeL1][1]))) return e;
  if ((e = set_smem_attr<kModeL2, kBnLarge, kStagesLarge>(&g_ctas[kModeL2][1]))) return e;
  if ((e = set_smem_attr<kModeFused, kBnLarge, kStagesLarge>(&g_ctas[kModeFused][1]))) return e;
  if ((e = set_smem_attr<kModeL1, kBnSmall, kStagesSmallDeep>(&g_ctas[kModeL1][2]))) return e;
  if ((e = set_smem_attr<kModeL2, kBnSmall, kStagesSmallDeep>(&g_ctas[kModeL2][2]))) return e;
  if ((e = set_smem_attr<kModeFused, kBnSmall, kStagesSmallDeep>(&g_ctas[kModeFused][2]))) return e;
  if ((e = set_smem_attr<kModeL1, kBnWide, kStagesWide>(&g_ctas[kModeL1][3]))) return e;
  if ((e = set_smem_attr<kModeL2, kBnWide, kStagesWide>(&g_ctas[kModeL2][3]))) return e;
  if ((e = set_smem_attr<kModeFused, kBnWide, kStagesWide>(&g_ctas[kModeFused][3]))) return e;
  if ((e = set_smem_attr<kModeL1, kBnSmall, kStagesQuad, 4>(&g_ctas[kModeL1][4]))) return e;
  if ((e = set_smem_attr<kModeL2, kBnSmall, kStagesQuad, 4>(&g_ctas[kModeL2][4]))) return e;
  if ((e = set_smem_attr<kModeFused, kBnSmall, kStagesQuad, 4>(&g_ctas[kModeFused][4]))) return e;
  if ((e = set_smem_attr<kModeL1, kBnMid, kStagesMid>(&g_ctas[kModeL1][5]))) return e;
  if ((e = set_smem_attr<kModeL2, kBnMid, kStagesMid>(&g_ctas[kModeL2][5]))) return e;
  if ((e = set_smem_attr<kModeFused, kBnMid, kStagesMid>(&g_ctas[kModeFused][5]))) return e;
  if ((e = set_smem_attr<kModeL1, kBnSmall, kStagesPromoSmall, 2, true>(&g_ctas[kModeL1][6]))) return e;
  if ((e = set_smem_attr<kModeL2, kBnSmall, kStagesPromoSmall, 2, true>(&g_ctas[kModeL2][6]))) return e;
  if ((e = set_smem_attr<kModeFused, kBnSmall, kStagesPromoSmall, 2, true>(&g_ctas[kModeFused][6]))) return e;
  if ((e = set_smem_attr<kModeL1, kBnMid, kStagesPromoMid, 2, true>(&g_ctas[kModeL1][7]))) return e;
  if ((e = set_smem_attr<kModeL2, kBnMid, kStagesPromoMid, 2, true>(&g_ctas[kModeL2][7]))) return e;
  if ((e = set_smem_attr<kModeFused, kBnMid, kStagesPromoMid, 2, true>(&g_ctas[kModeFused][7]))) return e;
  if ((e = mm_pair_prepare())) return e;
  return 0;
}

extern "C" int mm_gemm_blocks(int variant) { return variant == 4 ? 4 : 2; }

extern "C" int mm_gemm_epilogue_warps(int variant) {
  return variant == 1   ? mm::Warps<mm::kBnLarge, 2>::EPI
         : variant == 3 ? mm::Warps<mm::kBnWide, 2>::EPI
         : variant == 4 ? mm::Warps<mm::kBnSmall, 4>::EPI
         : variant == 5 || variant == 7 ? mm::Warps<mm::kBnMid, 2>::EPI
                        : mm::Warps<mm::kBnSmall, 2>::EPI;
}

extern "C" int mm_gemm_token_scale_box_rows(int variant) {
  return variant == 1   ? mm::GemmCfg<mm::kBnLarge, mm::kStagesLarge>::RAW_B_ROWS
         : variant == 3 ? mm::GemmCfg<mm::kBnWide, mm::kStagesWide>::RAW_B_ROWS
         : variant == 4 ? mm::GemmCfg<mm::kBnSmall, mm::kStagesQuad, 4>::RAW_B_ROWS
         : variant == 5 ? mm::GemmCfg<mm::kBnMid, mm::kStagesMid>::RAW_B_ROWS
                        : mm::GemmCfg<mm::kBnSmall, mm::kStagesSmall>::RAW_B_ROWS;
}

extern "C" int mm_launch_gemm(int l1, int variant, const mm::GemmMaps* maps, const mm::GemmArgs* a, int num_ctas,
                              void* stream) {
  using namespace mm;
  (void)num_ctas;
  cudaStream_t st = (cudaStream_t)stream;
  const int mode = l1 ? kModeL1 : kModeL2;
  const int n = g_ctas[mode][variant];
  if (l1) {
    return variant == 0   ? launch<kModeL1, kBnSmall, kStagesSmall>(maps, a, a, n, st)
           : variant == 6 ? launch<kModeL1, kBnSmall, kStagesPromoSmall, 2, true>(maps, a, a, n, st)
           : variant == 7 ? launch<kModeL1, kBnMid, kStagesPromoMid, 2, true>(maps, a, a, n, st)
           : variant == 2 ? launch<kModeL1, kBnSmall, kStagesSmallDeep>(maps, a, a, n, st)
           : variant == 3 ? launch<kModeL1, kBnWide, kStagesWide>(maps, a, a, n, st)
           : variant == 4 ? launch<kModeL1, kBnSmall, kStagesQuad, 4>(maps, a, a, n, st)
           : variant == 5 ? launch<kModeL1, kBnMid, kStagesMid>(maps, a, a, n, st)
                          : launch<kModeL1, kBnLarge, kStagesLarge>(maps, a, a, n, st);
  }
  return variant == 0   ? launch<kModeL2, kBnSmall, kStagesSmall>(maps, a, a, n, st)
         : variant == 6 ? launch<kModeL2, kBnSmall, kStagesPromoSmall, 2, true>(maps, a, a, n, st)
         : variant == 7 ? launch<kModeL2, kBnMid, kStagesPromoMid, 2, true>(maps, a, a, n, st)
         : variant == 2 ? launch<kModeL2, kBnSmall, kStagesSmallDeep>(maps, a, a, n, st)
         : variant == 3 ? launch<kModeL2, kBnWide, kStagesWide>(maps, a, a, n, st)
         : variant == 4 ? launch<kModeL2, kBnSmall, kStagesQuad, 4>(maps, a, a, n, st)
         : variant == 5 ? launch<kModeL2, kBnMid, kStagesMid>(maps, a, a, n, st)
                        : launch<kModeL2, kBnLarge, kStagesLarge>(maps, a, a, n, st);
}

extern "C" int mm_launch_gemm_class(int l1, int variant, const mm::GemmMaps* maps, const mm::GemmArgs* a,
                                    void* stream) {
  using namespace mm;
  cudaStream_t st = (cudaStream_t)stream;
  // the heavy class runs 224-token tiles, the light class 112-token tiles
  if (variant == 3)
    return l1 ? launch<kModeL1, kBnWide, kStagesWide>(maps, a, a, g_ctas[kModeL1][3], st, false)
              : launch<kModeL2, kBnWide, kStagesWide>(maps, a, a, g_ctas[kModeL2][3], st, false);
  if (variant == 1)
    return l1 ? launch<kModeL1, kBnLarge, kStagesLarge>(maps, a, a, g_ctas[kModeL1][1], st, false)
              : launch<kModeL2, kBnLarge, kStagesLarge>(maps, a, a, g_ctas[kModeL2][1], st, false);
  return (int)cudaErrorInvalidValue;
}

extern "C" int mm_launch_gemm_fused(int variant, const mm::GemmMaps* maps, const mm::GemmArgs* g1,
                                    const mm::GemmArgs* g2, void* stream) {
  using namespace mm;
  cudaStream_t st = (cudaStream_t)stream;
  const int n = g_ctas[kModeFused][variant];
  return variant == 0   ? launch<kModeFused, kBnSmall, kStagesSmall>(maps, g1, g2, n, st)
         : variant == 6 ? launch<kModeFused, kBnSmall, kStagesPromoSmall, 2, true>(maps, g1, g2, n, st)
         : variant == 7 ? launch<kModeFused, kBnMid, kStagesPromoMid, 2, true>(maps, g1, g2, n, st)
         : variant == 2 ? launch<kModeFused, kBnSmall, kStagesSmallDeep>(maps, g1, g2, n, st)
         : variant == 3 ? launch<kModeFused, kBnWide, kStagesWide>(maps, g1, g2, n, st)
         : variant == 4 ? launch<kModeFused, kBnSmall, kStagesQuad, 4>(maps, g1, g2, n, st)
         : variant == 5 ? launch<kModeFused, kBnMid, kStagesMid>(maps, g1, g2, n, st)
                        : launch<kModeFused, kBnLarge, kStagesLarge>(maps, g1, g2, n, st);
}
