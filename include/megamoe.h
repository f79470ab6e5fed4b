/*
 * megamoe.h — C ABI of the GB300 (sm_103a) MegaMoE expert path.
 *
 * One call computes, for T tokens on one GPU, the expert part of a
 * Mixture-of-Experts layer as the DeepGEMM MegaMoE pages describe it
 * ("MegaMoE on SM100/SM90 research report", sec. 4.1 "pr-304: SM100 Fused
 * MegaMoE", Linear1 / Linear2 phases and the combine; "MEGAMOE_SM90_DESIGN",
 * sec. 9 dispatch, 10 L1 epilogue, 11 L2 epilogue + combine):
 *
 *   route    per-expert counts, prefix offsets and an expert-sorted permutation
 *            of the T*(k+S) slots (stable in slot order)
 *   L1       acc1[r, n] = sum_k x[t_r, k] * W1[e_r, n, k],  n in [0, 2I)
 *   SwiGLU   y = silu(clamp(gate)) * clamp(up) * w_r       (gate = acc1[:, :I], up = acc1[:, I:])
 *   requant  per row and 32 columns of y: UE8M0 scale = smallest power of two
 *            >= amax/448, E4M3 = round_nearest_even(y / scale)
 *   L2       z[r, h] = bf16( sum_i q[r, i] * W2[e_r, h, i] )
 *   combine  out[t, h] = bf16( sum over the token's valid slots j, ascending, of z[row(t, j), h] )
 *
 * Activations are FP8 E4M3 with one UE8M0 scale per 32 along K; expert
 * weights are MXFP4: E2M1 codes packed two per byte (even K index in the low
 * nibble) with one UE8M0 scale per 32 along K, or, after
 * mm_set_weight_format(h, MM_WEIGHTS_MXFP8), E4M3 codes one per byte with the
 * same scales. Accumulation is FP32.
 *
 * Call order: mm_create, optionally mm_set_options / mm_set_schedule /
 * mm_set_tile_policy / mm_set_weight_format / mm_set_ep_ranks /
 * mm_set_expert_stats, mm_workspace_bytes, then any number of mm_run calls,
 * then mm_destroy. Options may change between calls.
 * Shared experts (num_shared = S) are stacked after the E routed experts in
 * W1/W2 (indices E..E+S-1) and applied to every token with weight 1.
 *
 * Threading: a handle may be used from one host thread at a time. All device
 * work is enqueued on the caller's stream; no call synchronises the device
 * except mm_get_status (which synchronises the given stream).
 */
#ifndef MEGAMOE_H
#define MEGAMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MM_API __attribute__((visibility("default")))
#else
#define MM_API
#endif

/* Same type as cudaStream_t / CUstream (NULL = the legacy default stream). */
struct CUstream_st;
typedef struct CUstream_st* mm_stream_t;

typedef struct mm_handle* mm_handle_t;

typedef enum {
  MM_OK = 0,
  MM_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad option value      */
  MM_ERR_UNSUPPORTED = 2,        /* shape outside the supported set (see mm_create)    */
  MM_ERR_WORKSPACE_TOO_SMALL = 3,/* ws_bytes < mm_workspace_bytes(T)                   */
  MM_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed                  */
  MM_ERR_DEVICE_TIMEOUT = 5,     /* (device status) a bounded device wait expired      */
  MM_ERR_BAD_ROUTING = 6,        /* (device status) a topk_idx entry was out of range  */
  MM_ERR_ALIGNMENT = 7           /* a pointer violates the alignment stated below      */
} mm_status_t;

/* Device status bits written into the workspace by the kernels and returned
 * by mm_get_status (0 = no error). */
#define MM_DEV_BAD_ROUTING 0x1u   /* an out-of-range expert id was skipped (slot disabled) */
#define MM_DEV_TIMEOUT 0x2u       /* a pipeline wait exceeded its time limit; outputs invalid */
/* With MM_DEV_TIMEOUT, bits 8..23 name the wait that expired (diagnostic):
 * bit 8 + s for the L1 GEMM and 16 + s for the L2 GEMM, s = 0 stage free,
 * 1 accumulator free, 2 stage loaded, 3 accumulator ready, 4 copy drain,
 * 5 stage free (scale-factor writer), 6 (L2 tiles of the fused schedule) token
 * rows stored by the L1 epilogues; bit 15 for mm_debug_timeout_probe; bit 23
 * for the hand-off of tile indices from the loading warp to the others. */

/* Human-readable name of a status code (static string). The pages have no
 * counterpart: their Python entry points raise exceptions instead. */
MM_API const char* mm_status_string(mm_status_t s);

/* Creates a handle for one layer shape ("MegaMoE research report" sec. 6.4,
 * the per-shape set-up calls get_block_m_for_mega_moe and
 * get_symm_buffer_size_for_mega_moe that precede fp8_fp4_mega_moe;
 * "MEGAMOE_SM90_DESIGN" sec. 16.1 API Design).
 *   E           routed experts, 1 <= E and E + S <= 1024
 *   H           hidden size; multiple of 128, 128 <= H <= 16384
 *   I           intermediate size; multiple of 128, 128 <= I <= 16384
 *   topk        routed slots per token, 1 <= topk <= 16
 *   num_shared  shared experts S, 0 <= S <= 4, topk + S <= 16
 * The handle owns only host memory. It serves the device current at creation;
 * creating it also looks up the device address of the library's fixed scratch
 * array (see mm_run_noalloc). Returns MM_ERR_UNSUPPORTED for shapes outside
 * these limits and MM_ERR_CUDA if the device is not sm_103 (GB300) or a CUDA
 * query fails. */
MM_API mm_status_t mm_create(mm_handle_t* out, int E, int H, int I, int topk, int num_shared);

/* SwiGLU options (the SM90 design's activation_clamp / fast_math arguments,
 * "MEGAMOE_SM90_DESIGN" sec. 10.1): swiglu_clamp > 0 clamps gate and up to
 * [-c, c] before the SiLU, <= 0 disables the clamp; fast_math != 0 uses the
 * fast approximate exponential (__expf) and the approximate reciprocal in the
 * SiLU (the pages' fast path). Defaults: no clamp, accurate exp and a correctly
 * rounded division (see mm_debug_div_check). */
MM_API mm_status_t mm_set_options(mm_handle_t h, float swiglu_clamp, int fast_math);

/* GEMM schedule ("MegaMoE research report" sec. 4.1, the Linear1 -> Linear2
 * hand-off through per-row arrival flags).
 *   MM_SCHEDULE_FUSED: both grouped GEMMs in one persistent launch: every L1
 *     tile, then every L2 tile, an L2 tile starting once the L1 epilogues of
 *     its token rows have stored them, so the weight stream of L2 follows that
 *     of L1 without a drain between them (weight-bandwidth-bound calls).
 *   MM_SCHEDULE_SPLIT: one launch per linear (compute-bound calls).
 *   MM_SCHEDULE_AUTO (the default): fused when the call routes at most
 *     MM_FUSED_MAX_ROWS_PER_EXPERT rows per expert on average (T*(topk+S)/(E+S)),
 *     split above; the threshold is where the two measured equal on GB300.
 * The results are identical (the same tiles compute the same sums); only the
 * timing differs. Other values: MM_ERR_INVALID_ARG. */
#define MM_SCHEDULE_AUTO (-1)
#define MM_SCHEDULE_SPLIT 0
#define MM_SCHEDULE_FUSED 1
#define MM_FUSED_MAX_ROWS_PER_EXPERT 128
MM_API mm_status_t mm_set_schedule(mm_handle_t h, int schedule);

/* Token-tile width of the grouped GEMMs: the tuned expert-load buckets of
 * "MEGAMOE_SM90_DESIGN" sec. 13.1 (BLOCK_M chosen from three buckets by the
 * load) and "MegaMoE research report" sec. 5.5 (kernel configuration routed by
 * token count).
 *   MM_TILES_16: 16-token tiles pairing two 128-row weight blocks, one MMA
 *     stream per block (weight-stream bound calls);
 *   MM_TILES_64: 64-token tiles, otherwise as MM_TILES_112 but with five
 *     pipeline stages instead of four (more weight bytes in flight); only for
 *     calls with E + S <= 300 experts, larger calls run MM_TILES_112;
 *   MM_TILES_112: 112-token tiles, eight epilogue warps, two TMEM
 *     accumulator buffers so that a tile's epilogue overlaps the next tile's
 *     MMAs;
 *   MM_TILES_224: 224-token tiles, otherwise as MM_TILES_112 but with one
 *     accumulator buffer (two 224-column accumulators fill TMEM), twelve
 *     epilogue warps and three pipeline stages: one MMA per K step and weight block does twice the
 *     work of a 112-token MMA for one instruction issue (compute-bound calls
 *     with many rows per expert);
 *   MM_TILES_AUTO (the default): MM_TILES_16 while the call routes at most
 *     MM_TILES16_MAX_ROWS_PER_EXPERT rows per expert on average
 *     (T*(topk+S) <= 12*(E+S)); above MM_TILES224_MIN_ROWS_PER_EXPERT rows
 *     per expert MM_TILES_224 when the call runs fused and MM_TILES_PER_EXPERT
 *     when it runs split (with uniform routing every expert is then above 112
 *     rows and takes 224-token tiles; a skewed load keeps its light experts
 *     on 112-token tiles); MM_TILES_64 above MM_TILES16_MAX_ROWS_PER_EXPERT
 *     and up to MM_TILES64_MAX_ROWS_PER_EXPERT rows per expert when the call
 *     has no shared expert (a shared expert receives every token, far above
 *     the average, and would take many 64-token tiles) and E <= 300,
 *     MM_TILES_112 otherwise: the crossovers measured on GB300 at H = 7168,
 *     I = 2048, 256 experts, top-8 (above 112 rows per expert an expert's
 *     rows take one 224-token tile instead of two 112-token ones: 128 rows
 *     per expert 1.73 against 2.17 ms per forward, 150 rows 1.86 against
 *     2.27, 192 rows 2.13 against 2.43) and at H = 4096, I = 1536, 128
 *     experts, top-8.
 * Every width computes the same tiles' sums; the results are identical.
 * Other values: MM_ERR_INVALID_ARG. */
#define MM_TILES_AUTO (-1)
/* MM_TILES_PER_EXPERT: the token-tile width by each expert's routed rows
 * ("MEGAMOE_SM90_DESIGN" sec. 12.1 and 13.1, BLOCK_M by expert load; the
 * concurrent launches on disjoint SM partitions of "MegaMoE research report"
 * sec. 12, PR357, without green contexts), for calls that run the split
 * schedule (others run as MM_TILES_AUTO): the experts
 * with more than 112 rows on 224-token tiles and the others on 112-token
 * tiles, as two persistent launches per linear that share the SMs (the heavy
 * experts' launches on a stream of the handle, forked from and joined back
 * into the caller's stream; the split of the SMs follows each class's tile
 * count). MM_TILES_AUTO takes it for every split call above 112 rows per
 * expert (Zipf-skewed routing with a shared expert, T = 4096: 2.11 against
 * 2.25 ms per forward with one width). mm_token_tile_width reports 224 for
 * such calls. Results are identical to the other widths. */
#define MM_TILES_PER_EXPERT 0
/* MM_TILES_224_PAIRS: the 224-token tiles of the split schedule on CTA pairs
 * ("MEGAMOE_SM90_DESIGN" sec. 4.1: pr-304's 2-CTA cluster, the leader CTA
 * issuing the UMMA and the scale-factor copies into TMEM, double-buffered
 * TMEM accumulators): clusters of two CTAs compute M = 256 block-scaled MMAs
 * (tcgen05 cta_group::2), each CTA holding 128 weight rows, half of the token
 * tile and its own 224-column accumulator, twice, so that each tile's
 * epilogue runs under the next tile's MMAs. Needs the scale rows by TMA (H
 * and I multiples of 512, 16-byte aligned scale tensors) and a split call;
 * other calls run as MM_TILES_224. Results are identical to the other
 * widths. Measured slower than MM_TILES_224 at prefill: one thread issues
 * every MMA of a pair, and its per-K-step waits and commits cannot overlap
 * another issuer's MMAs. */
#define MM_TILES_224_PAIRS (-2)
#define MM_TILES_16 16
#define MM_TILES_64 64
#define MM_TILES_112 112
#define MM_TILES_224 224
#define MM_TILES16_MAX_ROWS_PER_EXPERT 12
#define MM_TILES64_MAX_ROWS_PER_EXPERT 48
#define MM_TILES224_MIN_ROWS_PER_EXPERT 112
MM_API mm_status_t mm_set_tile_policy(mm_handle_t h, int policy);

/* The token-tile width (16, 64, 112 or 224) a call of T tokens runs with under the
 * handle's current policy (the counterpart of get_block_m_for_mega_moe,
 * "MegaMoE research report" sec. 6.4, which returns the block the kernel
 * aligns an expert's tokens to). Host only. */
MM_API mm_status_t mm_token_tile_width(mm_handle_t h, int T, int* width);

/* Weight element format (both linears; the weight recipes (1,1,32) MXFP4 and
 * FP8 of the "SM90 FP8 x MXFP4 MegaMoE" pull request #411 page, and
 * "MEGAMOE_SM90_DESIGN" sec. 15.2 Weight SF Layout). MM_WEIGHTS_MXFP4 (the default): E2M1
 * codes packed two per byte, the even K index in the low nibble (OCP MXFP4).
 * MM_WEIGHTS_MXFP8: E4M3 codes, one byte per element (OCP MXFP8; the FP8 x FP8
 * variant of the pages' SM90 recipe, with the UE8M0-per-32 block scales the
 * block-scaled tensor-core MMA reads instead of float scales per 128). Either
 * way one UE8M0 scale per 32 elements along K. MM_WEIGHTS_FP8_F128: below.
 * Other values: MM_ERR_INVALID_ARG. */
#define MM_WEIGHTS_MXFP4 0
#define MM_WEIGHTS_MXFP8 1
/* MM_WEIGHTS_FP8_F128: the float-scale FP8 recipe (1, 128, 128) of the SM90
 * design ("MEGAMOE_SM90_DESIGN" sec. 5.3 and 15.2). Weights E4M3, one byte per
 * element, with one float32 scale per 128 x 128 block; activations x with one
 * float32 scale per (token, 128 along H); the L2 activations the path makes
 * get one float32 scale per (row, 128 along I), amax / 448. Buffers of mm_run:
 *   x_sf  float32 [T][H/128]                 (4-byte aligned)
 *   w1    [E+S][2I][H] E4M3,  w1_sf float32 [E+S][2I/128][H/128]
 *   w2    [E+S][H][I] E4M3,   w2_sf float32 [E+S][H/128][I/128]
 * Each 128-long K block is an unscaled FP8 partial sum (kind::f8f6f4) that the
 * epilogue warps multiply by the two scales and accumulate in FP32. Token
 * tiles are 16 or 64 wide (a 112 or 224 policy runs 64). */
#define MM_WEIGHTS_FP8_F128 2
MM_API mm_status_t mm_set_weight_format(mm_handle_t h, int format);

/* Weight-scale transform ("MegaMoE research report" sec. 6.4, the SM100
 * kernel's transform_weights_for_mega_moe, which transposes the UE8M0 scale
 * factors for the tensor core's scale copy ahead of time; "MEGAMOE_SM90_DESIGN"
 * sec. 15.2 Weight SF Layout, SM100: UE8M0, 4 x 32 transposed, per 32 along
 * K). The transformed copy holds, for every 128-row block of a weight tensor
 * and every 128-long K step, the 512 bytes that the grouped GEMM copies into
 * TMEM for that block and step: byte 16 * l + 4 * i + b is the scale byte b
 * (32-element block b of the step) of row 32 * i + l of the block. Each such
 * piece then arrives in shared memory as one 512-byte bulk copy instead of
 * 128 strided 16-byte rows.
 *   mm_transformed_scale_bytes(h, &bytes): device bytes of the copy for both
 *     weight scale tensors ([E+S][2I][H/32] + [E+S][H][I/32] bytes, the same as
 *     the two inputs).
 *   mm_transform_weight_scales(h, w1_sf, w2_sf, dst, dst_bytes, stream): writes
 *     the copy of w1_sf and w2_sf (device, read only) into dst (device, caller
 *     owned, at least mm_transformed_scale_bytes, 16-byte aligned) on stream,
 *     and registers it on the handle: a later mm_run (on a stream ordered
 *     after this one) whose w1_sf and w2_sf arguments are these two pointers
 *     reads the copy instead; a run with other scale pointers reads its
 *     arguments. Rewrite the copy (call again) whenever the scales' contents
 *     change; dst = NULL unregisters. The transform is weight preparation, not
 *     part of a forward. UE8M0 formats only (MXFP4, MXFP8), H and I multiples of
 *     512, both scale tensors 16-byte aligned (else MM_ERR_UNSUPPORTED); runs on
 *     CTA pairs, and runs after a switch to MM_WEIGHTS_FP8_F128, read the
 *     arguments.
 *     Errors: MM_ERR_INVALID_ARG for a null handle, null scale pointers, an
 *     unaligned dst or dst_bytes too small; MM_ERR_CUDA if the launch fails. */
MM_API mm_status_t mm_transformed_scale_bytes(mm_handle_t h, size_t* bytes);
MM_API mm_status_t mm_transform_weight_scales(mm_handle_t h, const void* w1_sf, const void* w2_sf, void* dst,
                                              size_t dst_bytes, mm_stream_t stream);

/* Expert-parallel-ready routing outputs ("MegaMoE research report" sec. 4.1,
 * the dispatch warps' expert counts and source metadata; "MEGAMOE_SM90_DESIGN"
 * sec. 16.1, the cumulative_local_expert_recv_stats argument, and sec. 21
 * Phase 2 step 2.3, the per-rank receive counts; here every expert is local
 * and nothing is sent).
 *
 * mm_set_ep_ranks: the routed experts are owned by num_ranks destination
 * ranks in contiguous blocks of E / num_ranks (rank g owns experts
 * [g*E/num_ranks, (g+1)*E/num_ranks)); E % num_ranks must be 0
 * (MM_ERR_UNSUPPORTED otherwise), 1 <= num_ranks <= E (MM_ERR_INVALID_ARG
 * otherwise). Default 1. Because the routing order is expert-major with the
 * experts of a rank contiguous, it is also ordered by destination rank: after
 * each mm_run, the workspace holds rank_offsets[num_ranks + 1] (see
 * mm_debug_views_t) with rows [rank_offsets[g], rank_offsets[g+1]) of the
 * sorted order bound for rank g; rank_offsets[num_ranks] is the number of
 * routed rows, the shared experts' rows (replicated on every rank) follow.
 *
 * mm_set_expert_stats: a caller-owned device array of E + S int32 (4-byte
 * aligned; NULL disables). Every mm_run adds each expert's routed row count of
 * that call to it on the device, in stream order after routing; the library
 * never reads it otherwise, never clears it and never frees it. The pointer
 * must stay valid while calls that use it are in flight. */
MM_API mm_status_t mm_set_ep_ranks(mm_handle_t h, int num_ranks);
MM_API mm_status_t mm_set_expert_stats(mm_handle_t h, int32_t* cumulative_counts);

/* Bytes of device workspace mm_run needs for T tokens (T >= 0): the local
 * form of the symmetric buffer whose layout get_symm_buffer_size_for_mega_moe
 * computes ("MegaMoE research report" sec. 6.4; "MEGAMOE_SM90_DESIGN" sec. 16.1).
 * The workspace holds the routing tables, the gathered FP8 L1 operand, the FP8 L2
 * operand, the BF16 per-slot L2 output and a status word. Host only; MM_OK, or
 * MM_ERR_INVALID_ARG for a null handle or pointer or T < 0. */
MM_API mm_status_t mm_workspace_bytes(mm_handle_t h, int T, size_t* bytes);

/* Runs the path for T tokens, asynchronously on `stream`: the local form of
 * fp8_fp4_mega_moe ("MegaMoE research report" sec. 6.4 and sec. 4.1) and of the
 * fp8_mega_moe argument list of "MEGAMOE_SM90_DESIGN" sec. 16.1 (activations,
 * the L1 and L2 weight tuples, the workspace, top-k); the workspace is
 * re-initialised by the call itself, as the design's sec. 21 Phase 2 step 2.2
 * and Phase 6 step 6.6 require of two calls in a row.
 *   x_fp8    device, [T][H] E4M3                                  (16-byte aligned)
 *   x_sf     device, [T][H/32] UE8M0                               (4-byte aligned)
 *            (MM_WEIGHTS_FP8_F128: [T][H/128] float32)
 *   topk_idx device, [T][topk] int32, each in [0, E) or -1 (slot disabled);
 *            other values disable the slot and set MM_DEV_BAD_ROUTING
 *   topk_w   device, [T][topk] float32 (need not sum to 1)
 *   w1       device, [E+S][2I][H/2] E2M1 packed; rows [0,I) gate, [I,2I) up   (32-byte aligned)
 *            (MM_WEIGHTS_MXFP8, MM_WEIGHTS_FP8_F128: [E+S][2I][H] E4M3)
 *   w1_sf    device, [E+S][2I][H/32] UE8M0                                     (4-byte aligned)
 *            (MM_WEIGHTS_FP8_F128: [E+S][2I/128][H/128] float32)
 *   w2       device, [E+S][H][I/2] E2M1 packed                                  (32-byte aligned)
 *            (MM_WEIGHTS_MXFP8, MM_WEIGHTS_FP8_F128: [E+S][H][I] E4M3)
 *   w2_sf    device, [E+S][H][I/32] UE8M0                                      (4-byte aligned)
 *            (MM_WEIGHTS_FP8_F128: [E+S][H/128][I/128] float32)
 *   out_bf16 device, [T][H] bfloat16, fully overwritten               (16-byte aligned)
 *   ws       device workspace of ws_bytes >= mm_workspace_bytes(T) (256-byte aligned),
 *            fully re-initialised by every call, so it can be reused; two calls that
 *            share a workspace must be ordered on the device (same stream).
 * All buffers are owned by the caller and must stay valid until the work on
 * `stream` completes. T == 0 is valid: only the status word is reset.
 * Returns synchronous argument errors only; device-side errors are read with
 * mm_get_status. */
MM_API mm_status_t mm_run(mm_handle_t h, int T, const void* x_fp8, const void* x_sf, const int32_t* topk_idx,
                   const float* topk_w, const void* w1, const void* w1_sf, const void* w2, const void* w2_sf,
                   void* out_bf16, void* ws, size_t ws_bytes, mm_stream_t stream);

/* Synchronises `stream` and returns in *device_status the MM_DEV_* bits the
 * last mm_run on this workspace recorded (0 = none). The pages' kernels poll
 * arrival counters until the other side completes (the "SM90 FP8 x MXFP4
 * MegaMoE" pull request #411 page's review of the dispatch completion
 * protocol: a waiter polls and eventually times out; "MEGAMOE_SM90_DESIGN"
 * sec. 21, the no-hang criteria of Phase 2 step 2.6 and Phase 3 step 3.8);
 * here every wait is bounded and an expiry is reported through this word
 * instead of a hang. Returns MM_ERR_INVALID_ARG for null arguments and
 * MM_ERR_CUDA if the copy or the synchronisation fails. */
MM_API mm_status_t mm_get_status(mm_handle_t h, const void* ws, mm_stream_t stream, uint32_t* device_status);

/* Number of kernel launches one mm_run for T tokens enqueues (host only). The
 * pages have no counterpart; it states the split into kernels that
 * "MegaMoE research report" sec. 4.1 (one fused kernel) and sec. 4.3 (pr-352's
 * split L1/L2 kernels) compare. */
MM_API mm_status_t mm_launches_per_run(mm_handle_t h, int T, int* launches);

/* Device pointers into a workspace after mm_run for T tokens (contents valid
 * once the stream has reached them):
 *   counts [E+S] int32, offsets [E+S+1] int32, perm [T(k+S)] int32 (pool row -> slot
 *   t*(k+S)+j), pos [T(k+S)] int32 (slot -> pool row or -1), row_w [T(k+S)] float,
 *   pool_x [rows][H] u8, pool_sf [rows][H/32] u8, l2a [rows][I] u8 (E4M3),
 *   l2a_sf [rows][I/32] u8 (UE8M0; MM_WEIGHTS_FP8_F128: [rows][I/128] float32, the
 *   same bytes), z [rows][H] bf16, status (uint32). Rows are in
 *   pool order (expert-sorted); only the first offsets[E+S] rows are defined. */
typedef struct {
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* pos;
  float* row_w;
  uint8_t* pool_x;
  uint8_t* pool_sf;
  uint8_t* l2a;
  uint8_t* l2a_sf;
  uint16_t* z;
  uint32_t* status;
  int rows_capacity;
  int32_t* rank_offsets; /* [ep_ranks + 1], see mm_set_ep_ranks */
} mm_debug_views_t;

/* Test views (mm_debug_views_t above) into a workspace used by mm_run for T
 * tokens: the local form of the verification views of "MEGAMOE_SM90_DEV" (the
 * 2026-06-18 00:46 entry, l1_accum_debug for single-tile accumulator checks)
 * and of the dispatch products that "MEGAMOE_SM90_DESIGN" sec. 21 Phase 2
 * checks against the routing reference. Host only (pointer arithmetic on ws);
 * MM_ERR_INVALID_ARG for null arguments or T < 0. */
MM_API mm_status_t mm_debug_views(mm_handle_t h, void* ws, int T, mm_debug_views_t* views);

/* Test hook for the bounded-wait machinery behind mm_get_status (the pages'
 * no-hang criteria, "MEGAMOE_SM90_DESIGN" sec. 21 Phase 3 steps 3.2 and 3.8):
 * launches one CTA that waits on an
 * mbarrier nothing ever arrives on, gives up after timeout_ns nanoseconds,
 * sets MM_DEV_TIMEOUT in the workspace status word and returns. The GPU stays
 * usable. ws must hold at least 256 bytes. */
MM_API mm_status_t mm_debug_timeout_probe(void* ws, uint64_t timeout_ns, mm_stream_t stream);

/* Test hook for the SiLU division of "MEGAMOE_SM90_DESIGN" sec. 10.1 (silu =
 * gate / (1 + exp(-gate)), fast_math off): the L1 epilogue divides the gate by
 * 1 + exp(-gate) with a branch-free Newton-Raphson reciprocal and Markstein's
 * residual correction instead of the IEEE division routine. This compares it
 * with __frcp_rn / __fdiv_rn on the GPU. counts: device memory, 5 x uint64,
 * 8-byte aligned, zeroed here, then
 *   [0] significands of y in [1, 2) (all 2^23) whose refined reciprocal is not
 *       the correctly rounded one,
 *   [1] of `pairs` pseudo-random (x, y >= 1) pairs (splitmix64 stream `seed`),
 *       those with a normal IEEE quotient where the two differ,
 *   [2] those with a subnormal or zero IEEE quotient where they differ,
 *   [3] pairs checked,
 *   [4] pairs where they differ by more than one unit in the last place.
 * pairs <= 2^40. Asynchronous on `stream`. */
MM_API mm_status_t mm_debug_div_check(uint64_t pairs, uint64_t seed, unsigned long long* counts, mm_stream_t stream);

/* Per-launch timing for measurement, the local form of the pages' per-phase
 * profiling switch ("MEGAMOE_SM90_DESIGN" sec. 18, DG_SM90_MOE_PHASE_PROFILE,
 * and sec. 19.4): with profiling on, mm_run records a CUDA
 * event on its stream before each launch and after the last one. mm_profile_last
 * waits for the last recorded event and writes up to n durations in
 * milliseconds into ms, one per launch of the last profiled mm_run (route,
 * gather, then "l1_gemm", "l2_gemm" or the fused "gemm", then combine),
 * returning the count in *written; mm_profile_name(h, i) names the i-th
 * (NULL past the end). Events are created on the handle's device and freed by
 * mm_destroy or mm_profile_enable(h, 0). */
MM_API mm_status_t mm_profile_enable(mm_handle_t h, int on);
MM_API mm_status_t mm_profile_last(mm_handle_t h, float* ms, int n, int* written);
MM_API const char* mm_profile_name(mm_handle_t h, int i);

/* Allocation-free variant of mm_run (the pages have no counterpart; this is a
 * convenience of this library). Some callers cannot allocate device memory
 * where they run the layer: plugin hosts that own every device allocation and
 * forbid allocating inside their execute callback, and latency-critical loops
 * that avoid cudaMalloc/cudaFree because those calls can synchronise the
 * device. mm_run_noalloc computes exactly what mm_run computes, with the
 * workspace taken from a fixed 32 MiB array of device memory inside this
 * library instead of a caller buffer; every GPU that loads the library holds
 * that array until the process exits. The caller still passes the inputs and
 * the output, with the layouts and alignments of mm_run.
 *   - Calls whose workspace (mm_workspace_bytes(h, T)) exceeds 32 MiB are
 *     rejected with MM_ERR_WORKSPACE_TOO_SMALL before anything is enqueued
 *     (up to T = 143 tokens at H = 7168, I = 2048, E = 256, top-8).
 *   - mm_create looks up the array's device address (cudaGetSymbolAddress,
 *     on the device current at creation; that first use of the library's
 *     device code on the device is also when the driver backs the array) and
 *     keeps it in the handle, so this call does no set-up of its own. A handle
 *     serves only the device it was created on (MM_ERR_CUDA otherwise) and
 *     must be recreated after a cudaDeviceReset on that device.
 *   - Nothing is allocated or freed: no cudaMalloc, cudaFree or allocating
 *     library routine is called.
 *   - All calls in the process share the one array, which keeps the last
 *     call's contents. Nothing in it has to start at zero (every call rewrites
 *     the routing tables and the status word before use), but calls that
 *     overlap on the GPU (different streams, or different handles without
 *     ordering between them) race on it and give undefined results. */
MM_API mm_status_t mm_run_noalloc(mm_handle_t h, int T, const void* x_fp8, const void* x_sf, const int32_t* topk_idx,
                                  const float* topk_w, const void* w1, const void* w1_sf, const void* w2,
                                  const void* w2_sf, void* out_bf16, mm_stream_t stream);

/* Destroys a handle made by mm_create (the same set-up passages:
 * "MegaMoE research report" sec. 6.4; "MEGAMOE_SM90_DESIGN" sec. 16.1).
 * NULL is ignored. Frees only the handle's host memory and its profiling
 * events; the caller's buffers and workspaces are untouched. */
MM_API void mm_destroy(mm_handle_t h);

#ifdef __cplusplus
}
#endif
#endif /* MEGAMOE_H */
