// Host side of the C ABI declared in include/megamoe.h: argument checks,
// workspace carving, TMA tensor-map encoding and the launches of one forward
// (route -> gather -> L1 GEMM -> L2 GEMM -> combine, the two GEMMs in one
// persistent launch by default).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "mm_internal.h"

using namespace mm;

// Scratch for mm_run_noalloc: a fixed-size device array owned by this library,
// for callers that cannot allocate device memory where they run the layer.
// Host code must not use the symbol as an address: mm_create looks up its
// device address (cudaGetSymbolAddress, on the device current at creation)
// and keeps it in the handle.
namespace {
constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;
static __device__ __align__(256) uint8_t mm_static_ws[kStaticWorkspaceBytes];
}  // namespace

struct mm_handle {
  int E, H, I, k, S;
  float clamp;
  int fast_math;
  int device;
  int num_sms;
  unsigned long long timeout_ns;
  void* static_ws;  // device address of mm_static_ws on this handle's device
  // cached weight tensor maps (keyed by base pointer)
  const void* w1_key;
  const void* w2_key;
  const void* w1sf_key;
  const void* w2sf_key;
  CUtensorMap tm_w1;
  CUtensorMap tm_w2;
  CUtensorMap tm_w1sf;  // scale rows, 16-byte x 128-row boxes
  CUtensorMap tm_w2sf;
  // CTA-pair L1 launches: W1 and its scale rows in 64-row boxes (keyed by w1 / w1_sf)
  const void* w1h_key;
  const void* w1sfh_key;
  CUtensorMap tm_w1h;
  CUtensorMap tm_w1sfh;
  // transformed weight scales (mm_transform_weight_scales): the caller's copy
  // and the two scale tensors it was made from (null: none registered)
  const void* tsf_w1;
  const void* tsf_w2;
  uint8_t* tsf_dst;
  // GEMM schedule: MM_SCHEDULE_AUTO / _SPLIT / _FUSED
  int schedule;
  // expert-parallel-ready routing: destination ranks and the caller's
  // cumulative per-expert row counts (device, may be null)
  int ep_ranks;
  int32_t* expert_stats;
  // weight format: MM_WEIGHTS_MXFP4 / MM_WEIGHTS_MXFP8
  int w_fmt;
  // token-tile width: MM_TILES_AUTO / _16 / _64 / _112 / _224
  int tiles;
  // per-expert tile widths: the heavy class's launches run on this stream,
  // forked from and joined back into the caller's stream by the two events
  cudaStream_t side;
  cudaEvent_t fork, join;
  // optional per-launch events (route, gather, L1, L2, combine, end) and the
  // stage name of each recorded interval
  bool profile;
  int n_recorded;
  cudaEvent_t ev[6];
  const char* ev_name[6];
};

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2D map over a row-major [rows][k_elems] tensor, box = 128 elements of K x box_rows rows, 128-byte swizzle.
bool encode_2d(CUtensorMap* m, const void* base, bool fp4, uint64_t k_elems, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {k_elems, rows};
  cuuint64_t strides[1] = {fp4 ? k_elems / 2 : k_elems};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Scale rows [rows][cols] bytes, boxes of 16 bytes (four K steps) x 128 rows,
// no swizzle (the scale warp reads them with plain 16-byte loads).
bool encode_sf(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {16, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Whether a call of T tokens runs both GEMMs in one launch.
bool use_fused(const mm_handle* h, int T) {
  if (h->schedule != MM_SCHEDULE_AUTO) return h->schedule == MM_SCHEDULE_FUSED;
  const long long rows = (long long)T * (h->k + h->S);
  return rows <= (long long)MM_FUSED_MAX_ROWS_PER_EXPERT * (h->E + h->S);
}

// Kernel variant of a call: 0 = 16-token tiles, 2 = 16-token tiles with six
// stages (at most kDeepMaxExperts experts), 4 = 16-token tiles with four weight
// blocks (E4M3 weights, at most kQuadMaxExperts experts, I a multiple of 256:
// measured 97% -> 100% of the copy bandwidth at decode; with E2M1 weights it
// was 2% slower than variant 2), 5 = 64-token tiles with five stages (at most
// kDeepMaxExperts experts; 112-token tiles otherwise), 1 = 112-token tiles,
// 3 = 224-token tiles.
int variant_for(const mm_handle* h, int T) {
  const long long rows = (long long)T * (h->k + h->S), ep = h->E + h->S;
  int width = h->tiles;
  // float-scale weights: 16- or 64-token tiles (the epilogue keeps the
  // promoted sums in registers, which wider tiles would not fit)
  if (h->w_fmt == MM_WEIGHTS_FP8_F128)
    return width == MM_TILES_16 || (width == MM_TILES_AUTO && rows <= MM_TILES16_MAX_ROWS_PER_EXPERT * ep) ? 6 : 7;
  // (per-expert widths where a call does not run them: as AUTO)
  if (width == MM_TILES_AUTO || width == MM_TILES_PER_EXPERT)
    width = rows <= MM_TILES16_MAX_ROWS_PER_EXPERT * ep   ? MM_TILES_16
            : rows > MM_TILES224_MIN_ROWS_PER_EXPERT * ep ? MM_TILES_224
            : rows <= MM_TILES64_MAX_ROWS_PER_EXPERT * ep && h->S == 0 ? MM_TILES_64
                                                                       : MM_TILES_112;
  if (width == MM_TILES_112) return 1;
  if (width == MM_TILES_224 || width == MM_TILES_224_PAIRS) return 3;
  if (width == MM_TILES_64) return h->E + h->S <= kDeepMaxExperts ? 5 : 1;
  if (h->w_fmt == MM_WEIGHTS_MXFP8 && h->E + h->S <= kQuadMaxExperts && h->I % 256 == 0)
    return 4;
  return (h->E + h->S <= kDeepMaxExperts) ? 2 : 0;
}

// Whether a call runs per-expert tile widths: two concurrent launches per
// linear, the experts with more than 112 routed rows on 224-token tiles and
// the others on 112-token tiles (split schedule, MXFP4/MXFP8 weights). AUTO
// takes them for split calls above MM_TILES224_MIN_ROWS_PER_EXPERT rows per
// expert: with uniform routing every expert is then heavy and the call runs
// the 224-token tiles alone; with a skewed load the light experts' tiles
// stay 112 wide.
bool use_dual(const mm_handle* h, int T) {
  if (h->w_fmt == MM_WEIGHTS_FP8_F128 || use_fused(h, T) || T == 0) return false;
  if (h->tiles == MM_TILES_PER_EXPERT) return true;
  const long long rows = (long long)T * (h->k + h->S), ep = h->E + h->S;
  return h->tiles == MM_TILES_AUTO && rows > MM_TILES224_MIN_ROWS_PER_EXPERT * ep;
}

int tile_width(int variant) {
  return variant == 1 ? kBnLarge : variant == 3 ? kBnWide : variant == 5 || variant == 7 ? kBnMid : kBnSmall;
}

}  // namespace

extern "C" {

const char* mm_status_string(mm_status_t s) {
  switch (s) {
    case MM_OK: return "ok";
    case MM_ERR_INVALID_ARG: return "invalid argument";
    case MM_ERR_UNSUPPORTED: return "unsupported shape";
    case MM_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MM_ERR_CUDA: return "CUDA error";
    case MM_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MM_ERR_BAD_ROUTING: return "top-k index out of range";
    case MM_ERR_ALIGNMENT: return "pointer misaligned";
  }
  return "unknown status";
}

mm_status_t mm_create(mm_handle_t* out, int E, int H, int I, int topk, int num_shared) {
  if (!out) return MM_ERR_INVALID_ARG;
  *out = nullptr;
  if (E < 1 || topk < 1 || num_shared < 0) return MM_ERR_INVALID_ARG;
  if (E + num_shared > kMaxExperts || topk + num_shared > kMaxSlots || num_shared > 4) return MM_ERR_UNSUPPORTED;
  if (H < 128 || I < 128 || H % 128 || I % 128 || H > 16384 || I > 16384) return MM_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MM_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MM_ERR_CUDA;
  if (major != 10 || minor != 3) return MM_ERR_CUDA;  // built for sm_103a only
  if (!encode_fn()) return MM_ERR_CUDA;
  if (mm_gemm_prepare() != 0) return MM_ERR_CUDA;
  void* static_ws = nullptr;
  if (cudaGetSymbolAddress(&static_ws, mm_static_ws) != cudaSuccess || !static_ws) return MM_ERR_CUDA;
  mm_handle* h = new (std::nothrow) mm_handle();
  if (!h) return MM_ERR_INVALID_ARG;
  h->E = E; h->H = H; h->I = I; h->k = topk; h->S = num_shared;
  h->clamp = 0.0f; h->fast_math = 0; h->device = dev; h->num_sms = sms;
  h->static_ws = static_ws;
  h->timeout_ns = 4000000000ull;
  if (const char* t = getenv("MM_DEVICE_TIMEOUT_MS")) {
    long ms = atol(t);
    if (ms > 0) h->timeout_ns = (unsigned long long)ms * 1000000ull;
  }
  h->w1_key = h->w2_key = h->w1sf_key = h->w2sf_key = nullptr;
  h->w1h_key = h->w1sfh_key = nullptr;
  h->tsf_w1 = h->tsf_w2 = nullptr;
  h->tsf_dst = nullptr;
  h->schedule = MM_SCHEDULE_AUTO;
  h->ep_ranks = 1;
  h->expert_stats = nullptr;
  h->w_fmt = MM_WEIGHTS_MXFP4;
  h->tiles = MM_TILES_AUTO;
  h->profile = false;
  h->n_recorded = 0;
  if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess) {
    delete h;
    return MM_ERR_CUDA;
  }
  if (cudaEventCreateWithFlags(&h->fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->join, cudaEventDisableTiming) != cudaSuccess) {
    cudaStreamDestroy(h->side);
    delete h;
    return MM_ERR_CUDA;
  }
  *out = h;
  return MM_OK;
}

mm_status_t mm_set_options(mm_handle_t h, float swiglu_clamp, int fast_math) {
  if (!h || swiglu_clamp != swiglu_clamp) return MM_ERR_INVALID_ARG;
  h->clamp = swiglu_clamp > 0.0f ? swiglu_clamp : 0.0f;
  h->fast_math = fast_math ? 1 : 0;
  return MM_OK;
}

mm_status_t mm_set_schedule(mm_handle_t h, int schedule) {
  if (!h || schedule < MM_SCHEDULE_AUTO || schedule > MM_SCHEDULE_FUSED) return MM_ERR_INVALID_ARG;
  h->schedule = schedule;
  return MM_OK;
}

mm_status_t mm_set_tile_policy(mm_handle_t h, int policy) {
  if (!h || (policy != MM_TILES_AUTO && policy != MM_TILES_16 && policy != MM_TILES_64 && policy != MM_TILES_112 &&
             policy != MM_TILES_224 && policy != MM_TILES_PER_EXPERT && policy != MM_TILES_224_PAIRS))
    return MM_ERR_INVALID_ARG;
  h->tiles = policy;
  return MM_OK;
}

mm_status_t mm_set_weight_format(mm_handle_t h, int format) {
  if (!h || (format != MM_WEIGHTS_MXFP4 && format != MM_WEIGHTS_MXFP8 && format != MM_WEIGHTS_FP8_F128))
    return MM_ERR_INVALID_ARG;
  if (format != h->w_fmt) h->w1_key = h->w2_key = h->w1h_key = nullptr;  // cached weight maps describe the old layout
  h->w_fmt = format;
  return MM_OK;
}

mm_status_t mm_transformed_scale_bytes(mm_handle_t h, size_t* bytes) {
  if (!h || !bytes) return MM_ERR_INVALID_ARG;
  const size_t ep = (size_t)(h->E + h->S);
  *bytes = ep * 2 * h->I * (h->H / 32) + ep * h->H * (h->I / 32);
  return MM_OK;
}

mm_status_t mm_transform_weight_scales(mm_handle_t h, const void* w1_sf, const void* w2_sf, void* dst,
                                       size_t dst_bytes, mm_stream_t stream) {
  if (!h) return MM_ERR_INVALID_ARG;
  if (!dst) {
    h->tsf_w1 = h->tsf_w2 = nullptr;
    h->tsf_dst = nullptr;
    return MM_OK;
  }
  size_t need = 0;
  mm_transformed_scale_bytes(h, &need);
  if (!w1_sf || !w2_sf || !aligned(dst, 16) || dst_bytes < need) return MM_ERR_INVALID_ARG;
  if (h->w_fmt == MM_WEIGHTS_FP8_F128 || h->H % 512 || h->I % 512 || !aligned(w1_sf, 16) || !aligned(w2_sf, 16))
    return MM_ERR_UNSUPPORTED;
  if (cudaSetDevice(h->device) != cudaSuccess) return MM_ERR_CUDA;
  const long ep = h->E + h->S;
  uint8_t* d1 = static_cast<uint8_t*>(dst);
  uint8_t* d2 = d1 + (size_t)ep * 2 * h->I * (h->H / 32);
  if (mm_launch_transform_sf(static_cast<const uint8_t*>(w1_sf), d1, ep * 2 * h->I / 128, h->H, stream) != 0 ||
      mm_launch_transform_sf(static_cast<const uint8_t*>(w2_sf), d2, ep * h->H / 128, h->I, stream) != 0)
    return MM_ERR_CUDA;
  h->tsf_w1 = w1_sf;
  h->tsf_w2 = w2_sf;
  h->tsf_dst = d1;
  return MM_OK;
}

mm_status_t mm_set_ep_ranks(mm_handle_t h, int num_ranks) {
  if (!h || num_ranks < 1 || num_ranks > h->E) return MM_ERR_INVALID_ARG;
  if (h->E % num_ranks != 0) return MM_ERR_UNSUPPORTED;
  h->ep_ranks = num_ranks;
  return MM_OK;
}

mm_status_t mm_set_expert_stats(mm_handle_t h, int32_t* cumulative_counts) {
  if (!h) return MM_ERR_INVALID_ARG;
  if (cumulative_counts && !aligned(cumulative_counts, 4)) return MM_ERR_ALIGNMENT;
  h->expert_stats = cumulative_counts;
  return MM_OK;
}

mm_status_t mm_workspace_bytes(mm_handle_t h, int T, size_t* bytes) {
  if (!h || !bytes || T < 0) return MM_ERR_INVALID_ARG;
  *bytes = make_layout(h->E, h->S, h->H, h->I, h->k, T).total;
  return MM_OK;
}

mm_status_t mm_token_tile_width(mm_handle_t h, int T, int* width) {
  if (!h || !width || T < 0) return MM_ERR_INVALID_ARG;
  *width = use_dual(h, T) ? kBnWide : tile_width(variant_for(h, T));  // (per expert: the heavy experts' width)
  return MM_OK;
}

mm_status_t mm_launches_per_run(mm_handle_t h, int T, int* launches) {
  if (!h || !launches || T < 0) return MM_ERR_INVALID_ARG;
  const int route = mm_route_launches(T * (h->k + h->S));
  *launches = T == 0 ? route : route + (use_fused(h, T) ? 3 : use_dual(h, T) ? 6 : 4);
  return MM_OK;
}

mm_status_t mm_run(mm_handle_t h, int T, const void* x_fp8, const void* x_sf, const int32_t* topk_idx,
                   const float* topk_w, const void* w1, const void* w1_sf, const void* w2, const void* w2_sf,
                   void* out_bf16, void* ws, size_t ws_bytes, mm_stream_t stream) {
  if (!h || T < 0 || !ws) return MM_ERR_INVALID_ARG;
  const Layout L = make_layout(h->E, h->S, h->H, h->I, h->k, T);
  if (ws_bytes < L.total) return MM_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(ws, 256)) return MM_ERR_ALIGNMENT;
  if (T > 0) {
    if (!x_fp8 || !x_sf || !topk_idx || !topk_w || !w1 || !w1_sf || !w2 || !w2_sf || !out_bf16)
      return MM_ERR_INVALID_ARG;
    if (!aligned(x_fp8, 16) || !aligned(x_sf, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
        !aligned(w1, 32) || !aligned(w2, 32) || !aligned(w1_sf, 4) || !aligned(w2_sf, 4) || !aligned(out_bf16, 16))
      return MM_ERR_ALIGNMENT;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return MM_ERR_CUDA;

  uint8_t* base = static_cast<uint8_t*>(ws);
  const int Ep = h->E + h->S, Kp = h->k + h->S;
  // Scale rows by TMA when every scale row is a whole number of 16-byte groups
  // (K a multiple of 512) and the weight scale tensors are 16-byte aligned;
  // otherwise the scale warp loads them itself (two-block tiles only).
  const bool sf_tma = h->w_fmt != MM_WEIGHTS_FP8_F128 && h->H % 512 == 0 && h->I % 512 == 0 && aligned(w1_sf, 16) &&
                      aligned(w2_sf, 16);
  const bool fused = use_fused(h, T), dual = use_dual(h, T);
  int variant = dual ? 1 : variant_for(h, T);  // (per expert: the light class's tiles)
  if (variant == 4 && !sf_tma) variant = (h->E + h->S <= kDeepMaxExperts) ? 2 : 0;
  const int bn1 = tile_width(variant);
  const int bn2 = bn1;
  // CTA pairs: the split schedule's 224-token tiles when asked for (scale rows by TMA)
  const bool pair = h->tiles == MM_TILES_224_PAIRS && !fused && sf_tma && mm_pair_ctas() >= 2;

  RouteArgs ra;
  ra.topk_idx = topk_idx;
  ra.topk_w = topk_w;
  ra.counts = reinterpret_cast<int32_t*>(base + L.counts);
  ra.offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  ra.tiles_l1 = reinterpret_cast<int32_t*>(base + L.tiles_l1);
  ra.tiles_l2 = reinterpret_cast<int32_t*>(base + L.tiles_l2);
  ra.eorder = reinterpret_cast<int32_t*>(base + L.eorder);
  ra.perm = reinterpret_cast<int32_t*>(base + L.perm);
  ra.pos = reinterpret_cast<int32_t*>(base + L.pos);
  ra.row_w = reinterpret_cast<float*>(base + L.row_w);
  ra.chunk_cnt = reinterpret_cast<int32_t*>(base + L.chunk_cnt);
  ra.chunk_base = reinterpret_cast<int32_t*>(base + L.chunk_base);
  ra.chunk_bad = reinterpret_cast<int32_t*>(base + L.chunk_bad);
  ra.ready = reinterpret_cast<int32_t*>(base + L.ready);
  ra.sched = reinterpret_cast<int32_t*>(base + L.sched);
  ra.rank_offsets = reinterpret_cast<int32_t*>(base + L.rank_offsets);
  ra.stats = h->expert_stats;
  ra.ep_ranks = h->ep_ranks;
  ra.status = reinterpret_cast<uint32_t*>(base + L.status);
  ra.T = T; ra.E = h->E; ra.k = h->k; ra.S = h->S;
  ra.bn_l1 = bn1; ra.bn_l2 = bn2;
  ra.bn_heavy = dual ? kBnWide : bn1;
  ra.dual_sms = dual ? h->num_sms : 0;
  const int na = mm_gemm_blocks(variant);                 // 128-row weight blocks per tile
  const int f1 = h->I / (64 * na), f2 = (h->H + 128 * na - 1) / (128 * na);  // weight tiles per expert
  ra.fb_l1 = f1;
  ra.fb_l2 = f2;
  int ev_i = 0;
  // an event before each launch (named for it) and one after the last
  auto mark = [&](const char* next) {
    if (h->profile && ev_i < 6) {
      h->ev_name[ev_i] = next;
      cudaEventRecord(h->ev[ev_i++], (cudaStream_t)stream);
    }
  };
  h->n_recorded = 0;
  mark("route");
  if (mm_launch_route(&ra, stream) != 0) return MM_ERR_CUDA;
  if (T == 0) {
    mark(nullptr);
    h->n_recorded = ev_i;
    return MM_OK;
  }

  GatherArgs ga;
  ga.x = static_cast<const uint8_t*>(x_fp8);
  ga.x_sf = static_cast<const uint8_t*>(x_sf);
  ga.pos = ra.pos;
  ga.pool_x = base + L.pool_x;
  ga.pool_sf = base + L.pool_sf;
  ga.T = T; ga.H = h->H; ga.Kp = Kp;
  mark("gather");
  if (mm_launch_gather(&ga, stream) != 0) return MM_ERR_CUDA;

  // Tensor maps: weights are cached per base pointer, activations live in the workspace.
  const bool fp4 = h->w_fmt == MM_WEIGHTS_MXFP4;
  if (h->w1_key != w1) {
    if (!encode_2d(&h->tm_w1, w1, fp4, (uint64_t)h->H, (uint64_t)Ep * 2 * h->I, 128)) return MM_ERR_CUDA;
    h->w1_key = w1;
  }
  if (h->w2_key != w2) {
    if (!encode_2d(&h->tm_w2, w2, fp4, (uint64_t)h->I, (uint64_t)Ep * h->H, 128)) return MM_ERR_CUDA;
    h->w2_key = w2;
  }
  GemmMaps maps;
  memset(&maps, 0, sizeof(maps));
  maps.w1 = h->tm_w1;
  maps.w2 = h->tm_w2;
  // token boxes: the whole token tile
  if (!encode_2d(&maps.a1, base + L.pool_x, false, (uint64_t)h->H, (uint64_t)L.rows_cap, (uint32_t)bn1))
    return MM_ERR_CUDA;
  if (!encode_2d(&maps.a2, base + L.l2a, false, (uint64_t)h->I, (uint64_t)L.rows_cap, (uint32_t)bn2))
    return MM_ERR_CUDA;
  if (variant == 3) {
    // narrower token boxes for the tiles that hold at most 112 or 32 rows
    if (!encode_2d(&maps.a1n, base + L.pool_x, false, (uint64_t)h->H, (uint64_t)L.rows_cap, (uint32_t)(bn1 / 2)) ||
        !encode_2d(&maps.a2n, base + L.l2a, false, (uint64_t)h->I, (uint64_t)L.rows_cap, (uint32_t)(bn2 / 2)) ||
        !encode_2d(&maps.a1s, base + L.pool_x, false, (uint64_t)h->H, (uint64_t)L.rows_cap, 32u) ||
        !encode_2d(&maps.a2s, base + L.l2a, false, (uint64_t)h->I, (uint64_t)L.rows_cap, 32u))
      return MM_ERR_CUDA;
  }
  if (sf_tma) {
    if (h->w1sf_key != w1_sf) {
      if (!encode_sf(&h->tm_w1sf, w1_sf, (uint64_t)h->H / 32, (uint64_t)Ep * 2 * h->I)) return MM_ERR_CUDA;
      h->w1sf_key = w1_sf;
    }
    if (h->w2sf_key != w2_sf) {
      if (!encode_sf(&h->tm_w2sf, w2_sf, (uint64_t)h->I / 32, (uint64_t)Ep * h->H)) return MM_ERR_CUDA;
      h->w2sf_key = w2_sf;
    }
    maps.wsf1 = h->tm_w1sf;
    maps.wsf2 = h->tm_w2sf;
    if (pair) {
      if (h->w1h_key != w1) {
        if (!encode_2d(&h->tm_w1h, w1, fp4, (uint64_t)h->H, (uint64_t)Ep * 2 * h->I, 64)) return MM_ERR_CUDA;
        h->w1h_key = w1;
      }
      if (h->w1sfh_key != w1_sf) {
        if (!encode_sf(&h->tm_w1sfh, w1_sf, (uint64_t)h->H / 32, (uint64_t)Ep * 2 * h->I, 64)) return MM_ERR_CUDA;
        h->w1sfh_key = w1_sf;
      }
      maps.w1h = h->tm_w1h;
      maps.wsf1h = h->tm_w1sfh;
    }
    const uint32_t tb = (uint32_t)mm_gemm_token_scale_box_rows(variant);
    if (!encode_sf(&maps.asf1, base + L.pool_sf, (uint64_t)h->H / 32, (uint64_t)L.rows_cap, tb)) return MM_ERR_CUDA;
    if (!encode_sf(&maps.asf2, base + L.l2a_sf, (uint64_t)h->I / 32, (uint64_t)L.rows_cap, tb)) return MM_ERR_CUDA;
  }
  GemmMaps maps_w;  // per-expert widths: the heavy class's 224-token tiles (token and token-scale boxes)
  if (dual) {
    maps_w = maps;
    const uint32_t tbw = (uint32_t)mm_gemm_token_scale_box_rows(3);
    if (!encode_2d(&maps_w.a1, base + L.pool_x, false, (uint64_t)h->H, (uint64_t)L.rows_cap, (uint32_t)kBnWide) ||
        !encode_2d(&maps_w.a2, base + L.l2a, false, (uint64_t)h->I, (uint64_t)L.rows_cap, (uint32_t)kBnWide) ||
        !encode_2d(&maps_w.a1n, base + L.pool_x, false, (uint64_t)h->H, (uint64_t)L.rows_cap, (uint32_t)(kBnWide / 2)) ||
        !encode_2d(&maps_w.a2n, base + L.l2a, false, (uint64_t)h->I, (uint64_t)L.rows_cap, (uint32_t)(kBnWide / 2)) ||
        !encode_2d(&maps_w.a1s, base + L.pool_x, false, (uint64_t)h->H, (uint64_t)L.rows_cap, 32u) ||
        !encode_2d(&maps_w.a2s, base + L.l2a, false, (uint64_t)h->I, (uint64_t)L.rows_cap, 32u) ||
        (sf_tma && (!encode_sf(&maps_w.asf1, base + L.pool_sf, (uint64_t)h->H / 32, (uint64_t)L.rows_cap, tbw) ||
                    !encode_sf(&maps_w.asf2, base + L.l2a_sf, (uint64_t)h->I / 32, (uint64_t)L.rows_cap, tbw))))
      return MM_ERR_CUDA;
  }

  GemmArgs g1;
  memset(&g1, 0, sizeof(g1));
  g1.w_sf = static_cast<const uint8_t*>(w1_sf);
  g1.act_sf = base + L.pool_sf;
  g1.offsets = ra.offsets;
  g1.tile_start = ra.tiles_l1;
  g1.eorder = ra.eorder;
  g1.row_w = ra.row_w;
  g1.out_q = base + L.l2a;
  g1.out_sf = base + L.l2a_sf;
  g1.status = ra.status;
  g1.Ep = Ep; g1.K = h->H; g1.rows_w = 2 * h->I; g1.I = h->I; g1.H = h->H; g1.fb_total = f1;
  g1.clamp = h->clamp; g1.fast_math = h->fast_math; g1.timeout_ns = h->timeout_ns;
  g1.w_sf_vec = aligned(w1_sf, 16) && (h->H / 32) % 16 == 0;
  g1.act_sf_vec = (h->H / 32) % 16 == 0;
  g1.w_fp8 = fp4 ? 0 : 1;
  g1.sf_tma = sf_tma ? 1 : 0;
  // the registered transformed weight scales, when this call's scale tensors
  // are the ones they were made from
  const bool tsf = sf_tma && h->tsf_dst && h->tsf_w1 == w1_sf && h->tsf_w2 == w2_sf;
  g1.w_sf_t = tsf ? h->tsf_dst : nullptr;
  g1.ready = reinterpret_cast<int32_t*>(base + L.ready);
  g1.ready_target = f1 * mm_gemm_epilogue_warps(variant);
  g1.tile_ctr = ra.sched + 0;
  g1.sched = ra.sched;

  GemmArgs g2 = g1;
  g2.w_sf = static_cast<const uint8_t*>(w2_sf);
  g2.w_sf_t = tsf ? h->tsf_dst + (size_t)Ep * 2 * h->I * (h->H / 32) : nullptr;
  g2.act_sf = base + L.l2a_sf;
  g2.tile_start = ra.tiles_l2;
  g2.row_w = nullptr;
  g2.out_q = nullptr;
  g2.out_sf = nullptr;
  g2.out_z = reinterpret_cast<uint16_t*>(base + L.z);
  g2.K = h->I; g2.rows_w = h->H; g2.fb_total = f2;
  g2.w_sf_vec = aligned(w2_sf, 16) && (h->I / 32) % 16 == 0;
  g2.tile_ctr = ra.sched + 1;  // the L2 launch of the split schedule (the fused launch uses g1's)
  g2.act_sf_vec = (h->I / 32) % 16 == 0;
  if (dual) {
    // the light class on the caller's stream (112-token tiles), the heavy
    // class on the side stream (224-token tiles), on disjoint SMs: each
    // launch's CTAs beyond its class's share leave at once
    mark("gemms");
    GemmArgs l1n = g1, l2n = g2, l1w = g1, l2w = g2;
    l1n.tile_class = l2n.tile_class = 1;
    l1w.tile_class = l2w.tile_class = 2;
    l1w.tile_ctr = ra.sched + 2;
    l2w.tile_ctr = ra.sched + 3;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaEventRecord(h->fork, st) != cudaSuccess || cudaStreamWaitEvent(h->side, h->fork, 0) != cudaSuccess)
      return MM_ERR_CUDA;
    // (ordinary stream order throughout: a launch allowed to start early would
    // hold SMs in its wait that the other class's launch is meant to get)
    if (mm_launch_gemm_class(1, variant, &maps, &l1n, stream) != 0) return MM_ERR_CUDA;
    if (mm_launch_gemm_class(1, 3, &maps_w, &l1w, h->side) != 0) return MM_ERR_CUDA;
    if (mm_launch_gemm_class(0, variant, &maps, &l2n, stream) != 0) return MM_ERR_CUDA;
    if (mm_launch_gemm_class(0, 3, &maps_w, &l2w, h->side) != 0) return MM_ERR_CUDA;
    if (cudaEventRecord(h->join, h->side) != cudaSuccess || cudaStreamWaitEvent(st, h->join, 0) != cudaSuccess)
      return MM_ERR_CUDA;
  } else if (fused) {
    mark("gemm");
    if (mm_launch_gemm_fused(variant, &maps, &g1, &g2, stream) != 0)
      return MM_ERR_CUDA;
  } else {
    mark("l1_gemm");
    if ((pair ? mm_launch_gemm_pair(1, &maps, &g1, stream)
              : mm_launch_gemm(1, variant, &maps, &g1, h->num_sms, stream)) != 0)
      return MM_ERR_CUDA;
    mark("l2_gemm");
    if ((pair ? mm_launch_gemm_pair(0, &maps, &g2, stream)
              : mm_launch_gemm(0, variant, &maps, &g2, h->num_sms, stream)) != 0)
      return MM_ERR_CUDA;
  }

  CombineArgs ca;
  ca.z = g2.out_z;
  ca.pos = ra.pos;
  ca.out = static_cast<uint16_t*>(out_bf16);
  ca.T = T; ca.H = h->H; ca.Kp = Kp;
  mark("combine");
  // (after the join of two streams: ordinary stream order)
  if (mm_launch_combine(&ca, stream, !dual) != 0) return MM_ERR_CUDA;
  mark(nullptr);
  h->n_recorded = ev_i;
  return MM_OK;
}

mm_status_t mm_profile_enable(mm_handle_t h, int on) {
  if (!h) return MM_ERR_INVALID_ARG;
  if (on && !h->profile) {
    for (int i = 0; i < 6; ++i)
      if (cudaEventCreate(&h->ev[i]) != cudaSuccess) return MM_ERR_CUDA;
    h->profile = true;
  } else if (!on && h->profile) {
    for (int i = 0; i < 6; ++i) cudaEventDestroy(h->ev[i]);
    h->profile = false;
  }
  h->n_recorded = 0;
  return MM_OK;
}

mm_status_t mm_profile_last(mm_handle_t h, float* ms, int n, int* written) {
  if (!h || !written || (n > 0 && !ms)) return MM_ERR_INVALID_ARG;
  *written = 0;
  if (!h->profile || h->n_recorded < 2) return MM_OK;
  if (cudaEventSynchronize(h->ev[h->n_recorded - 1]) != cudaSuccess) return MM_ERR_CUDA;
  int k = 0;
  for (int i = 0; i + 1 < h->n_recorded && k < n; ++i, ++k)
    if (cudaEventElapsedTime(&ms[k], h->ev[i], h->ev[i + 1]) != cudaSuccess) return MM_ERR_CUDA;
  *written = k;
  return MM_OK;
}

const char* mm_profile_name(mm_handle_t h, int i) {
  if (!h || i < 0 || i + 1 >= h->n_recorded) return nullptr;
  return h->ev_name[i];
}

mm_status_t mm_get_status(mm_handle_t h, const void* ws, mm_stream_t stream, uint32_t* device_status) {
  if (!h || !ws || !device_status) return MM_ERR_INVALID_ARG;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
    return MM_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MM_ERR_CUDA;
  *device_status = v;
  return MM_OK;
}

mm_status_t mm_debug_views(mm_handle_t h, void* ws, int T, mm_debug_views_t* v) {
  if (!h || !ws || !v || T < 0) return MM_ERR_INVALID_ARG;
  const Layout L = make_layout(h->E, h->S, h->H, h->I, h->k, T);
  uint8_t* b = static_cast<uint8_t*>(ws);
  v->counts = reinterpret_cast<int32_t*>(b + L.counts);
  v->offsets = reinterpret_cast<int32_t*>(b + L.offsets);
  v->perm = reinterpret_cast<int32_t*>(b + L.perm);
  v->pos = reinterpret_cast<int32_t*>(b + L.pos);
  v->row_w = reinterpret_cast<float*>(b + L.row_w);
  v->pool_x = b + L.pool_x;
  v->pool_sf = b + L.pool_sf;
  v->l2a = b + L.l2a;
  v->l2a_sf = b + L.l2a_sf;
  v->z = reinterpret_cast<uint16_t*>(b + L.z);
  v->status = reinterpret_cast<uint32_t*>(b + L.status);
  v->rows_capacity = L.rows_cap;
  v->rank_offsets = reinterpret_cast<int32_t*>(b + L.rank_offsets);
  return MM_OK;
}

mm_status_t mm_debug_div_check(uint64_t pairs, uint64_t seed, unsigned long long* counts, mm_stream_t stream) {
  if (!counts || pairs > (1ull << 40) || !aligned(counts, 8)) return MM_ERR_INVALID_ARG;
  if (cudaMemsetAsync(counts, 0, 5 * sizeof(unsigned long long), (cudaStream_t)stream) != cudaSuccess)
    return MM_ERR_CUDA;
  if (mm_launch_div_check(pairs, seed, counts, stream) != 0) return MM_ERR_CUDA;
  return MM_OK;
}

mm_status_t mm_debug_timeout_probe(void* ws, uint64_t timeout_ns, mm_stream_t stream) {
  if (!ws || timeout_ns == 0 || timeout_ns > 10000000000ull) return MM_ERR_INVALID_ARG;
  if (cudaMemsetAsync(ws, 0, 4, (cudaStream_t)stream) != cudaSuccess) return MM_ERR_CUDA;
  if (mm_launch_timeout_probe(static_cast<uint32_t*>(ws), timeout_ns, stream) != 0) return MM_ERR_CUDA;
  return MM_OK;
}

}  // extern "C"

extern "C" {

mm_status_t mm_run_noalloc(mm_handle_t h, int T, const void* x_fp8, const void* x_sf, const int32_t* topk_idx,
                           const float* topk_w, const void* w1, const void* w1_sf, const void* w2, const void* w2_sf,
                           void* out_bf16, mm_stream_t stream) {
  if (!h || T < 0) return MM_ERR_INVALID_ARG;
  if (make_layout(h->E, h->S, h->H, h->I, h->k, T).total > kStaticWorkspaceBytes) return MM_ERR_WORKSPACE_TOO_SMALL;
  // the array's address on the handle's device, looked up by mm_create (mm_run
  // checks that this device is current)
  return mm_run(h, T, x_fp8, x_sf, topk_idx, topk_w, w1, w1_sf, w2, w2_sf, out_bf16, h->static_ws,
                kStaticWorkspaceBytes, stream);
}

void mm_destroy(mm_handle_t h) {
  if (!h) return;
  cudaEventDestroy(h->fork);
  cudaEventDestroy(h->join);
  cudaStreamDestroy(h->side);
  if (h->profile)
    for (int i = 0; i < 6; ++i) cudaEventDestroy(h->ev[i]);
  delete h;
}

}  // extern "C"
