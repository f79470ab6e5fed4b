// Grouped GEMMs of the split schedule on CTA pairs: the 224-token tiles as M =
// 256 block-scaled MMAs over two SMs (tcgen05 cta_group::2).
//
// Each cluster of two CTAs takes one tile at a time: 256 weight rows x up to
// 224 tokens. CTA r holds 128 of the weight rows (L1: the gate rows of 64
// features and the matching up rows, so that its SwiGLU needs no other CTA;
// L2: one 128-row block of W2) and half of the token rows, and accumulates
// its 128 weight rows x all tokens in its own TMEM. A CTA's accumulator is
// 224 columns, so two buffers fit: the epilogue of one tile runs while the
// MMAs of the next fill the other buffer (the one-CTA 224-token tiles hold
// 448 columns per tile and drain them between tiles). Each stage of a CTA is
// 30 KB (its 128 weight rows and half of the token tile), five stages deep.
//
// Roles per CTA (13 warps): warp 0 loads (TMA) this CTA's operands; warp 1
// of the leader (rank 0) issues the MMAs for both CTAs; warp 2 allocates TMEM
// (collectively with the other CTA) and then loads (TMA) this CTA's weight
// scale rows and the token tile's, up to RAW_G groups of four K steps ahead
// and across tiles; warp 3 lays them out for tcgen05.cp in this CTA's shared
// memory, one ready signal per group (the other CTA's warp 1 relays it to
// the leader); the leader's warp 12 copies each K step's scales of both CTAs
// into their TMEM once the stage's scale columns are free (a copy issued by
// the MMA thread would wait for that thread's earlier MMAs); warps 4 .. 11
// are the epilogue.
//
// Synchronisation: both CTAs' operand loads of a stage complete on the
// leader's stage barrier (the other CTA's by the cta_group::2 form of the
// tensor copy), so the leader's MMAs start once every byte has landed; one
// commit per CTA frees the stage in both. The only other signal that crosses
// SMs is the per-group relay (a remote mbarrier arrival blocks its thread for
// about a thousand cycles, so a thread of its own makes it). A tile's last commit per CTA hands the accumulator to
// both epilogues, whose warps (of both CTAs) arrive on the leader's
// buffer-empty barrier. Every wait is bounded (status word, abort).
//
// "MEGAMOE_SM90_DESIGN" sec. 4.1 (pr-304 SM100 fused MegaMoE: a 2-CTA cluster,
// the leader CTA issuing the UMMA and the scale-factor copies into TMEM,
// double-buffered TMEM accumulators between the MMA and the epilogue warps).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "mm_common.cuh"
#include "mm_internal.h"
#include "mm_ptx.cuh"

namespace mm {
namespace {

enum : int { kPairL2 = 0, kPairL1 = 1 };

constexpr int kPairEpi = 4;  // epilogue warps per CTA (one per TMEM lane quadrant)
constexpr int kPairEpiStride = 16 * (kPairEpi / 4);  // columns between a warp's 16-column chunks
constexpr int kPairCopyWarp = 4 + kPairEpi;  // the leader's scale-copy warp
constexpr int kPairThreads = 32 * (5 + kPairEpi);

struct PairCfg {
  static constexpr int BK = 128;                       // K per stage
  static constexpr int BN = kBnWide;                   // token rows of a tile at most (the MMA N)
  static constexpr int B_ROWS = BN / 2;                // each CTA's token rows
  static constexpr int A_BYTES = 128 * BK;             // 16 KB (4-bit codes padded to bytes)
  static constexpr int B_BYTES = B_ROWS * BK;          // 14 KB
  static constexpr int STAGES = 5;
  static constexpr int SF_SLOTS = 8;  // shared-memory scale slots: two groups of four K steps
  // a stage's scales in the layout tcgen05.cp.32x128b.warpx4 reads: this CTA's
  // 128 weight rows, then all token rows of the tile (every CTA's TMEM holds
  // the token scales of the whole MMA N)
  static constexpr int SFB_ROWS = 256;
  static constexpr int SF_STAGE_BYTES = 512 + SFB_ROWS * 4;
  // TMA-loaded scale rows, four K steps (16 bytes) per row and group: this
  // CTA's 128 weight rows, then the tile's token rows
  static constexpr int RAW_G = 4;
  static constexpr int RAW_A_BYTES = 128 * 16;
  static constexpr int RAW_B_BYTES = SFB_ROWS * 16;
  static constexpr int RAW_GROUP_BYTES = RAW_A_BYTES + RAW_B_BYTES;
  // L1 epilogue: a gate warp and its up warp exchange half of a 16-column
  // chunk; [4 warp pairs][2 buffers][gate, up][8 columns][32 lanes] floats
  static constexpr int XCH_BYTES = 4 * 2 * 2 * 8 * 32 * 4;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
  static constexpr int SF_OFF = B_OFF + STAGES * B_BYTES;
  static constexpr int RAW_OFF = SF_OFF + SF_SLOTS * SF_STAGE_BYTES;
  static constexpr int XCH_OFF = RAW_OFF + RAW_G * RAW_GROUP_BYTES;
  static constexpr int TAB_INTS = kMaxExperts + 1;     // tile table and row offsets, [experts + 1] each
  static constexpr int TAB_OFF = XCH_OFF + XCH_BYTES;
  static constexpr int BAR_OFF = TAB_OFF + 2 * TAB_INTS * 4;
  // full, empty, sfready per stage; ready, peer-ready, free per scale-slot
  // group; tfull, tempty per buffer; rfull, rempty per raw group; the L1
  // exchange's per warp pair and buffer
  static constexpr int NBARS = 3 * STAGES + 6 + 4 + 2 * RAW_G + 8;
  static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;  // + the TMEM address, abort flag, alignment
  // TMEM: two accumulator buffers of BN columns, then a scale slot per stage
  // (4 columns of weight scales, 4 per 128 token rows)
  static constexpr int ACC_COLS = BN;
  static constexpr int SF_BASE = 2 * ACC_COLS;
  static constexpr int SF_STAGE_COLS = 4 + SFB_ROWS / 32;
  static constexpr int TMEM_COLS = 512;
  static_assert(SF_BASE + STAGES * SF_STAGE_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "operand tiles keep 1024-byte alignment");
  static_assert(RAW_OFF % 128 == 0 && BAR_OFF % 8 == 0, "alignment");
};

// wait sites in the status word (bit 8 + site)
constexpr uint32_t kPSiteLoad = 0, kPSiteMma = 1, kPSiteScale = 2, kPSiteEpi = 3, kPSiteTail = 4;

template <int MODE>
__global__ void __launch_bounds__(kPairThreads, 1)
    pair_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs g) {
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);  // [STAGES] (leader) both CTAs' bytes landed
  uint64_t* empty = full + C::STAGES;      // [STAGES] the MMAs that read the stage completed
  uint64_t* sfready = empty + C::STAGES;   // [STAGES] (leader) the K step's scales are in both CTAs' TMEM
  uint64_t* sgready = sfready + C::STAGES; // [2] this CTA's group of four scale slots is laid out
  uint64_t* sgpeer = sgready + 2;          // [2] (leader) the other CTA's group is laid out
  uint64_t* sgfree = sgpeer + 2;           // [2] the copies that read a group of scale slots completed
  uint64_t* tfull = sgfree + 2;            // [2] the accumulator buffer is complete
  uint64_t* tempty = tfull + 2;            // [2] (leader) both CTAs' epilogues have read the buffer
  uint64_t* rfull = tempty + 2;            // [RAW_G] scale rows landed
  uint64_t* rempty = rfull + C::RAW_G;     // [RAW_G] the scale warp has read them
  uint64_t* xbar = rempty + C::RAW_G;      // [4 warp pairs][2 buffers] (L1) both warps wrote their half
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);     // the leader's expect_tx arrival (both CTAs' bytes)
      mbar_init(&empty[s], 1);    // the leader's commit
      mbar_init(&sfready[s], 1);  // the scale warp's commit of its copies
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sgready[b], 1);  // this CTA's scale warp
      mbar_init(&sgpeer[b], 1);   // the other CTA's relay
      mbar_init(&sgfree[b], 1);   // the copy warp's commit after a group's copies
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);              // the leader's commit after a tile's last K step
      mbar_init(&tempty[b], 2 * kPairEpi);  // every epilogue warp of both CTAs
    }
    for (int b = 0; b < C::RAW_G; ++b) {
      mbar_init(&rfull[b], 1);
      mbar_init(&rempty[b], 1);
    }
    for (int b = 0; b < 8; ++b) mbar_init(&xbar[b], 2);  // the gate warp and the up warp of a pair
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (MODE == kPairL1) {
      prefetch_tmap(&maps.w1h);
      prefetch_tmap(&maps.a1n);
    } else {
      prefetch_tmap(&maps.w2);
      prefetch_tmap(&maps.a2n);
    }
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised, TMEM allocated in both
  tc_fence_after();
  // the prologue above overlaps the previous kernel; its outputs are read below
  pdl_trigger();
  pdl_wait();
  int* s_t = reinterpret_cast<int*>(smem + C::TAB_OFF);
  int* s_off = s_t + C::TAB_INTS;
  for (int i = threadIdx.x; i <= g.Ep; i += blockDim.x) {
    s_t[i] = g.tile_start[i];
    s_off[i] = g.offsets[i];
  }
  __syncthreads();
  const uint32_t tmem = *tmem_slot;
  const int num_tiles = s_t[g.Ep];
  const int P = (int)(gridDim.x >> 1), first = (int)(blockIdx.x >> 1);  // clusters, this cluster
  const int KB = g.K / C::BK;
  auto tile_of = [&](int tile) { return decode_tile(tile, s_t, nullptr, s_off, g.Ep, g.fb_total, C::BN); };
  // this CTA's 128-row weight block: L1 gate rows of features fb*128 + 64 rank
  // + [0, 64) (the up rows I further), L2 W2 block 2 fb + rank
  auto a_active_r = [&](const Tile& t, int r) {
    return t.active && (MODE == kPairL1 || (2 * t.fb + r) * 128 < g.rows_w);
  };
  auto a_row_r = [&](const Tile& t, int r) {
    return MODE == kPairL1 ? t.e * g.rows_w + t.fb * 128 + 64 * r : t.e * g.rows_w + (2 * t.fb + r) * 128;
  };
  auto a_active = [&](const Tile& t) { return a_active_r(t, (int)rank); };
  auto a_row = [&](const Tile& t) { return a_row_r(t, (int)rank); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;
    bool ok = true;
    const uint32_t a_tx = g.w_fp8 ? (uint32_t)C::A_BYTES : (uint32_t)(C::A_BYTES / 2);
    const CUtensorMap* tb = MODE == kPairL1 ? &maps.a1n : &maps.a2n;
    const uint32_t full0 = mapa_shared(smem_u32(full), 0u);  // the leader's stage barriers
    for (int tile = first; ok && tile < num_tiles; tile += P) {
      const Tile t = tile_of(tile);
      const int half = ((t.nrows + 15) & ~15) / 2;
      const bool act = a_active(t);
      // the leader expects both CTAs' bytes (the other CTA's block may be absent)
      const bool peer_act = a_active_r(t, 1);
      const int wrow = a_row(t);
      const int brow = t.row0 + (int)rank * half;  // this CTA's half of the token tile
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int s = (int)(it % C::STAGES);
        const uint32_t ph = (it / C::STAGES) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, g.status, g.timeout_ns, kPSiteLoad)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* sA = smem + C::A_OFF + s * C::A_BYTES;
          uint8_t* sB = smem + C::B_OFF + s * C::B_BYTES;
          const CUtensorMap* tw = MODE == kPairL1 ? &maps.w1h : &maps.w2;
          if (leader) {
            mbar_arrive_expect_tx(&full[s], (act ? a_tx : 0u) + (peer_act ? a_tx : 0u) + 2u * (uint32_t)C::B_BYTES);
            if (act) {
              tma_load_2d(sA, tw, &full[s], kb * C::BK, wrow);
              if (MODE == kPairL1) tma_load_2d(sA + C::A_BYTES / 2, tw, &full[s], kb * C::BK, wrow + g.I);
            }
            tma_load_2d(sB, tb, &full[s], kb * C::BK, brow);
          } else {
            const uint32_t fb = full0 + 8u * (uint32_t)s;
            if (act) {
              tma_load_2d_pair(sA, tw, fb, kb * C::BK, wrow);
              if (MODE == kPairL1) tma_load_2d_pair(sA + C::A_BYTES / 2, tw, fb, kb * C::BK, wrow + g.I);
            }
            tma_load_2d_pair(sB, tb, fb, kb * C::BK, brow);
          }
        }
      }
    }
    if (!ok && leader) {
      // let the copies already issued (by both CTAs, counted on the leader's
      // barriers) land before the CTAs can exit
      for (uint32_t j = (it > (uint32_t)C::STAGES ? it - C::STAGES : 0u); j < it; ++j) {
        int dummy = 0;
        mbar_wait(&full[j % C::STAGES], (j / C::STAGES) & 1u, reinterpret_cast<volatile int*>(&dummy), g.status,
                  g.timeout_ns < 10000000ull ? g.timeout_ns : 10000000ull, kPSiteTail);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ scale-row loader
    if (lane == 0) {
      const CUtensorMap* tbs = MODE == kPairL1 ? &maps.asf1 : &maps.asf2;
      uint32_t gi = 0;
      bool ok = true;
      for (int tile = first; ok && tile < num_tiles; tile += P) {
        const Tile t = tile_of(tile);
        const bool act = a_active(t);
        const int wrow = a_row(t);
        for (int kb = 0; kb < KB; kb += 4, ++gi) {
          const int gs = (int)(gi % C::RAW_G);
          if (!mbar_wait(&rempty[gs], ((gi / C::RAW_G) & 1u) ^ 1u, abort_flag, g.status, g.timeout_ns, kPSiteLoad)) {
            ok = false;
            break;
          }
          uint8_t* raw = smem + C::RAW_OFF + gs * C::RAW_GROUP_BYTES;
          mbar_arrive_expect_tx(&rfull[gs], (act ? (uint32_t)C::RAW_A_BYTES : 0u) + (uint32_t)C::RAW_B_BYTES);
          if (act) {
            if (MODE == kPairL1) {
              tma_load_2d(raw, &maps.wsf1h, &rfull[gs], kb * 4, wrow);
              tma_load_2d(raw + C::RAW_A_BYTES / 2, &maps.wsf1h, &rfull[gs], kb * 4, wrow + g.I);
            } else {
              tma_load_2d(raw, &maps.wsf2, &rfull[gs], kb * 4, wrow);
            }
          }
          tma_load_2d(raw + C::RAW_A_BYTES, tbs, &rfull[gs], kb * 4, t.row0);
        }
      }
      if (!ok) {
        // let the scale rows already requested land before the CTA can exit
        for (uint32_t j = (gi > (uint32_t)C::RAW_G ? gi - C::RAW_G : 0u); j < gi; ++j) {
          int dummy = 0;
          mbar_wait(&rfull[j % C::RAW_G], (j / C::RAW_G) & 1u, reinterpret_cast<volatile int*>(&dummy), g.status,
                    g.timeout_ns < 10000000ull ? g.timeout_ns : 10000000ull, kPSiteTail);
        }
      }
    }
  } else if (warp == 1 && !leader) {
    // ------------------------------------------------------------ relay (other CTA)
    if (lane == 0) {
      const uint32_t gp = mapa_shared(smem_u32(sgpeer), 0u);
      const uint32_t groups = first < num_tiles ? (uint32_t)((num_tiles - first + P - 1) / P) * (uint32_t)(KB / 4) : 0u;
      for (uint32_t gi = 0; gi < groups; ++gi) {
        if (!mbar_wait(&sgready[gi & 1u], (gi >> 1) & 1u, abort_flag, g.status, g.timeout_ns, kPSiteScale)) break;
        mbar_arrive_cluster(gp + 8u * (gi & 1u));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0) {
      const uint32_t a_fmt = g.w_fp8 ? 0u : 5u;  // A (weights): E4M3 or E2M1; B (tokens): E4M3
      const uint32_t e0 = mapa_shared(smem_u32(empty), 0u), e1 = mapa_shared(smem_u32(empty), 1u);
      const uint32_t f0 = mapa_shared(smem_u32(tfull), 0u), f1 = mapa_shared(smem_u32(tfull), 1u);
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int tile = first; ok && tile < num_tiles; tile += P, ++tc) {
        const Tile t = tile_of(tile);
        const uint32_t n_mma = (uint32_t)((t.nrows + 15) & ~15);
        const int b = (int)(tc & 1u);
        if (!mbar_wait_cluster(&tempty[b], ((tc >> 1) & 1u) ^ 1u, abort_flag, g.status, g.timeout_ns, kPSiteMma)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * C::ACC_COLS);
        // Two K steps per round: wait for both stages, issue their eight MMAs,
        // then commit both (the first commit of a batch stalls the issuing
        // thread for about a hundred cycles, the following ones do not; a
        // single issuing thread cannot hide that behind another's MMAs).
        for (int kb = 0; kb < KB; kb += 2, it += 2) {
          const int s0 = (int)(it % C::STAGES), s1 = (int)((it + 1u) % C::STAGES);
          const uint32_t ph0 = (it / C::STAGES) & 1u, ph1 = ((it + 1u) / C::STAGES) & 1u;
          if (!mbar_wait_cluster(&full[s0], ph0, abort_flag, g.status, g.timeout_ns, kPSiteMma) ||
              !mbar_wait(&sfready[s0], ph0, abort_flag, g.status, g.timeout_ns, kPSiteMma) ||
              !mbar_wait_cluster(&full[s1], ph1, abort_flag, g.status, g.timeout_ns, kPSiteMma) ||
              !mbar_wait(&sfready[s1], ph1, abort_flag, g.status, g.timeout_ns, kPSiteMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int s = h ? s1 : s0;
            const uint64_t da = sdesc_kmajor_sw128(smem_u32(smem + C::A_OFF + s * C::A_BYTES));
            const uint64_t db = sdesc_kmajor_sw128(smem_u32(smem + C::B_OFF + s * C::B_BYTES));
            const uint32_t sfa = tmem + (uint32_t)(C::SF_BASE + s * C::SF_STAGE_COLS), sfb = sfa + 4u;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_pair_mxf8f6f4(d, da + 2u * k, db + 2u * k, idesc_pair_mxf8f6f4(a_fmt, 0u, n_mma, (uint32_t)k),
                                   sfa, sfb, (kb > 0 || h > 0 || k > 0) ? 1u : 0u);
          }
          // both stages are free in both CTAs once these MMAs have read them
          tc_commit_pair(e0 + 8u * (uint32_t)s0);
          tc_commit_pair(e1 + 8u * (uint32_t)s0);
          tc_commit_pair(e0 + 8u * (uint32_t)s1);
          tc_commit_pair(e1 + 8u * (uint32_t)s1);
        }
        if (!ok) break;
        tc_commit_pair(f0 + 8u * (uint32_t)b);  // the accumulators are complete in both CTAs
        tc_commit_pair(f1 + 8u * (uint32_t)b);
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ scale layout
    // Per K step lane l writes 16 bytes per 128-row group: the step's scale
    // byte of rows l, l + 32, l + 64, l + 96 (this CTA's weight rows, then the
    // tile's token rows), into the step's slot in a ring of two groups of
    // four; one fence and one ready signal per group.
    uint32_t gi = 0;
    bool ok = true;
    for (int tile = first; ok && tile < num_tiles; tile += P) {
      const Tile t = tile_of(tile);
      const bool act = a_active(t);
      const int nb = (t.nrows + 31) / 32;
      for (int kg = 0; kg < KB; kg += 4, ++gi) {
        const int gs = (int)(gi % C::RAW_G);
        if (!mbar_wait(&rfull[gs], (gi / C::RAW_G) & 1u, abort_flag, g.status, g.timeout_ns, kPSiteScale)) {
          ok = false;
          break;
        }
        const uint8_t* raw = smem + C::RAW_OFF + gs * C::RAW_GROUP_BYTES;
        uint4 wa[4], wb[8];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          wa[i] = act ? *reinterpret_cast<const uint4*>(raw + (32 * i + lane) * 16) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          wb[j] = j < nb ? *reinterpret_cast<const uint4*>(raw + C::RAW_A_BYTES + (32 * j + lane) * 16)
                         : make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[gs]);
        const uint32_t gb = gi & 1u;  // slot group
        if (!mbar_wait(&sgfree[gb], ((gi >> 1) & 1u) ^ 1u, abort_flag, g.status, g.timeout_ns, kPSiteScale)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint8_t* sF = smem + C::SF_OFF + (int)(gb * 4u + (uint32_t)c) * C::SF_STAGE_BYTES;
          st_shared_v4(sF + lane * 16, word(wa[0], c), word(wa[1], c), word(wa[2], c), word(wa[3], c));
#pragma unroll
          for (int q = 0; q < 2; ++q)
            st_shared_v4(sF + 512 + q * 512 + lane * 16, word(wb[4 * q], c), word(wb[4 * q + 1], c),
                         word(wb[4 * q + 2], c), word(wb[4 * q + 3], c));
        }
        fence_proxy_async_smem();  // read next by tcgen05.cp
        __syncwarp();
        if (lane == 0) mbar_arrive(&sgready[gb]);
      }
    }
  } else if (warp == kPairCopyWarp && leader) {
    // ------------------------------------------------------------ scale copies (leader)
    // Per K step, once both CTAs' slot group is laid out and the MMAs that
    // read the stage's TMEM scale columns before have completed: one
    // cta_group::2 copy per 128-row group moves both CTAs' slots into their
    // TMEM, committed to the stage's sfready; a group's last copies are also
    // committed to both CTAs' slot-free barriers.
    if (lane == 0) {
      const uint32_t sfr0 = mapa_shared(smem_u32(sfready), 0u);
      const uint32_t sgf0 = mapa_shared(smem_u32(sgfree), 0u), sgf1 = mapa_shared(smem_u32(sgfree), 1u);
      const uint32_t groups = first < num_tiles ? (uint32_t)((num_tiles - first + P - 1) / P) * (uint32_t)(KB / 4) : 0u;
      uint32_t it = 0;
      for (uint32_t gi = 0; gi < groups; ++gi) {
        const uint32_t gb = gi & 1u, gph = (gi >> 1) & 1u;
        if (!mbar_wait(&sgready[gb], gph, abort_flag, g.status, g.timeout_ns, kPSiteScale) ||
            !mbar_wait_cluster(&sgpeer[gb], gph, abort_flag, g.status, g.timeout_ns, kPSiteScale))
          break;
        bool ok = true;
        for (int c = 0; c < 4; ++c, ++it) {
          const int s = (int)(it % C::STAGES);
          if (!mbar_wait(&empty[s], ((it / C::STAGES) & 1u) ^ 1u, abort_flag, g.status, g.timeout_ns, kPSiteScale)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* sF = smem + C::SF_OFF + (int)(gb * 4u + (uint32_t)c) * C::SF_STAGE_BYTES;
          const uint32_t slot = tmem + (uint32_t)(C::SF_BASE + s * C::SF_STAGE_COLS);
          tc_cp_pair_32x128b_warpx4(slot, sdesc_sf_32x16(smem_u32(sF)));
          tc_cp_pair_32x128b_warpx4(slot + 4u, sdesc_sf_32x16(smem_u32(sF + 512)));
          tc_cp_pair_32x128b_warpx4(slot + 8u, sdesc_sf_32x16(smem_u32(sF + 1024)));
          tc_commit_pair(sfr0 + 8u * (uint32_t)s);
        }
        if (!ok) break;
        tc_commit_pair(sgf0 + 8u * gb);
        tc_commit_pair(sgf1 + 8u * gb);
      }
    }
  } else if (warp >= 4 && warp < 4 + kPairEpi) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;          // TMEM lane quadrant of this warp
    const int hcol = (warp - 4) >> 2;  // which 16-column chunks: 16 hcol + 32 i
    const uint32_t te0 = mapa_shared(smem_u32(tempty), 0u);
    const uint32_t lanes = (uint32_t)(32 * q) << 16;
    uint32_t tc = 0, xc = 0;  // tiles, and L1 exchange chunks (both warps of a pair count alike)
    for (int tile = first; tile < num_tiles; tile += P, ++tc) {
      const Tile t = tile_of(tile);
      const int b = (int)(tc & 1u);
      if (!mbar_wait(&tfull[b], (tc >> 1) & 1u, abort_flag, g.status, g.timeout_ns, kPSiteEpi, 256)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + lanes + (uint32_t)(b * C::ACC_COLS);
      if (MODE == kPairL2) {
        // lane = W2 row = hidden feature; columns = token rows: BF16 per slot row
        const int blk = 2 * t.fb + (int)rank;
        const bool act = a_active(t);
        for (int c0 = 16 * hcol; act && c0 < t.nrows; c0 += kPairEpiStride) {
          uint32_t v[16];
          tmem_ld_x16(tbase + (uint32_t)c0, v);
          tmem_ld_wait();
          const int feat = blk * 128 + 32 * q + lane;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < t.nrows)
              g.out_z[(size_t)(t.row0 + c0 + j) * g.H + feat] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
        }
      } else {
        // Lanes 0-63 of the accumulator are the gate rows, 64-127 the up rows
        // of the same 64 features: quadrant q < 2 (gate) pairs with q + 2 (up).
        // Per 16-column chunk each warp of a pair takes 8 columns and receives
        // the other's half of them through shared memory; then per column the
        // 32 lanes (32 consecutive features: one UE8M0 group) hold
        // y = SwiGLU x top-k weight, and the group's amax is a transpose
        // reduction (after three exchange steps lanes 4c .. 4c + 3 share
        // column c, two more make it their common maximum).
        const bool gate = q < 2;
        const int fq = q & 1, pair = fq + 2 * hcol;
        float* xbuf = reinterpret_cast<float*>(smem + C::XCH_OFF) + pair * (2 * 2 * 256);
        const int feat = t.fb * 128 + 64 * (int)rank + 32 * fq + lane;
        const int fgroup = t.fb * 4 + 2 * (int)rank + fq;
        bool failed = false;
        for (int c0 = 16 * hcol; c0 < t.nrows; c0 += kPairEpiStride, ++xc) {
          uint32_t v[16];
          tmem_ld_x16(tbase + (uint32_t)c0, v);
          tmem_ld_wait();
          // double-buffered by chunk parity (a warp writes a buffer again only
          // after the exchange of the chunk in between, which its partner
          // joins once it has read this one)
          float* xb = xbuf + (xc & 1u) * 512;  // [0]: gate of columns 8..15, [1]: up of columns 0..7
#pragma unroll
          for (int j = 0; j < 8; ++j) xb[(gate ? 0 : 256) + j * 32 + lane] = __uint_as_float(v[gate ? 8 + j : j]);
          __syncwarp();
          uint64_t* xw = &xbar[pair * 2 + (int)(xc & 1u)];
          if (lane == 0) mbar_arrive(xw);
          if (!mbar_wait(xw, (xc >> 1) & 1u, abort_flag, g.status, g.timeout_ns, kPSiteEpi)) {
            failed = true;
            break;
          }
          float gv[8], uv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            gv[j] = gate ? __uint_as_float(v[j]) : xb[j * 32 + lane];
            uv[j] = gate ? xb[256 + j * 32 + lane] : __uint_as_float(v[8 + j]);
          }
          const int cb = c0 + (gate ? 0 : 8);  // this warp's first column
          const int ncol = min(8, t.nrows - cb);
          const float wl = lane < ncol ? g.row_w[t.row0 + cb + lane] : 0.0f;
          float y[8], a[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wl, j);
            float gj = gv[j], uj = uv[j];
            if (g.clamp > 0.0f) {
              gj = fminf(fmaxf(gj, -g.clamp), g.clamp);
              uj = fminf(fmaxf(uj, -g.clamp), g.clamp);
            }
            // silu(g) = g / (1 + exp(-g)); the fast path: __expf and the
            // approximate reciprocal
            const float silu = g.fast_math ? __fmul_rn(gj, rcp_approx(__fadd_rn(1.0f, __expf(-gj))))
                                           : div_ge1(gj, __fadd_rn(1.0f, expf(-gj)));
            y[j] = j < ncol ? __fmul_rn(__fmul_rn(silu, uj), wj) : 0.0f;
            a[j] = fabsf(y[j]);
          }
#pragma unroll
          for (int o = 16, n = 8; n > 1; o >>= 1, n >>= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
              const float recv = __shfl_xor_sync(0xffffffffu, upper ? a[i] : a[i + n / 2], o);
              a[i] = fmaxf(upper ? a[i + n / 2] : a[i], recv);
            }
          }
          a[0] = fmaxf(a[0], __shfl_xor_sync(0xffffffffu, a[0], 2));
          a[0] = fmaxf(a[0], __shfl_xor_sync(0xffffffffu, a[0], 1));
          const int mycol = lane >> 2;
          const uint32_t code = requant_code(a[0]);
          const float inv = inv_scale(code);
          if ((lane & 3) == 0 && mycol < ncol)
            g.out_sf[(size_t)(t.row0 + cb + mycol) * (g.I / 32) + fgroup] = (uint8_t)code;
          uint32_t qw[2];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float ij = __shfl_sync(0xffffffffu, inv, j << 2);
            const uint32_t qb = (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(y[j], ij), __NV_SATFINITE, __NV_E4M3) & 0xFFu;
            qw[j >> 2] = (j & 3) == 0 ? qb : qw[j >> 2] | (qb << (8 * (j & 3)));
          }
          store_u8_rows_4x4(g.out_q, (size_t)g.I, t.row0, cb, ncol, feat - lane, qw);
        }
        if (failed) break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(te0 + 8u * (uint32_t)b);  // this warp has read the buffer
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no arrival or copy of either CTA still targets the other
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

int g_pair_ctas = 0;  // CTAs per launch: twice the clusters that can be resident at once

template <int MODE>
cudaError_t launch_pair(const GemmMaps* maps, const GemmArgs* a, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)g_pair_ctas);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = PairCfg::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<MODE>, *maps, *a);
}

}  // namespace
}  // namespace mm

extern "C" int mm_pair_prepare(void) {
  using namespace mm;
  cudaError_t e = cudaFuncSetAttribute(pair_gemm_kernel<kPairL1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PairCfg::SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pair_gemm_kernel<kPairL2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairCfg::SMEM_BYTES);
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = PairCfg::SMEM_BYTES;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, pair_gemm_kernel<kPairL1>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();  // no CTA pairs on this device: the one-CTA 224-token tiles serve instead
    clusters = 0;
  }
  g_pair_ctas = 2 * clusters;
  return 0;
}

extern "C" int mm_pair_ctas(void) { return mm::g_pair_ctas; }

extern "C" int mm_launch_gemm_pair(int l1, const mm::GemmMaps* maps, const mm::GemmArgs* a, void* stream) {
  using namespace mm;
  if (g_pair_ctas < 2) return (int)cudaErrorInvalidConfiguration;
  cudaStream_t st = (cudaStream_t)stream;
  return (int)(l1 ? launch_pair<kPairL1>(maps, a, st) : launch_pair<kPairL2>(maps, a, st));
}
