/*
 * Oracle for the MegaMoE expert path: a plain, slow CPU restatement used only
 * as test infrastructure (tests, the smoke check and the CPU baseline timing).
 * It shares no code with the CUDA library.
 */
#ifndef MEGAMOE_ORACLE_H
#define MEGAMOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int T;          /* tokens                                  */
  int H;          /* hidden size (K of L1, N of L2)          */
  int I;          /* intermediate size (N of L1 is 2I)       */
  int E;          /* routed experts                          */
  int k;          /* routed slots per token                  */
  int S;          /* shared experts (0 or more), weight 1    */
  float clamp;    /* SwiGLU clamp c (<= 0: off)              */
  int weight_in_combine; /* diagnosis only: apply top-k weight in the combine instead of L1 */
  int w_fmt;      /* weight elements: 0 = E2M1 packed two per byte (MXFP4),
                     1 = E4M3 one per byte (MXFP8); both with UE8M0 per 32 along K;
                     2 = the float-scale FP8 recipe (1, 128, 128): E4M3 weights,
                     one float32 scale per 128 x 128 weight block, activations
                     and L2 activations with one float32 scale per (row, 128
                     along K); H and I multiples of 128 */
} orc_dims;

/* Format decoders / encoders (OCP Microscaling v1.0, OCP FP8, bfloat16). */
float orc_e4m3_to_float(uint8_t b);
float orc_e2m1_to_float(uint8_t nibble);
float orc_ue8m0_to_float(uint8_t b);
uint8_t orc_float_to_e4m3(float v);      /* nearest even, saturating to +-448 */
uint16_t orc_float_to_bf16(float v);     /* nearest even */
float orc_bf16_to_float(uint16_t h);
uint8_t orc_requant_code(float amax);    /* UE8M0 code for the L2-activation scale */

void orc_decode_e4m3(const uint8_t* in, float* out, long n);
void orc_decode_e2m1(const uint8_t* in, float* out, long n);
void orc_decode_ue8m0(const uint8_t* in, float* out, long n);
void orc_encode_e4m3(const float* in, uint8_t* out, long n);
void orc_encode_bf16(const float* in, uint16_t* out, long n);
void orc_requant_codes(const float* amax, uint8_t* out, long n);

/* Routing: counting sort of the T*(k+S) slots by expert, stable in slot order.
 * counts[E+S], offsets[E+S+1], perm[T*(k+S)] (pool row -> slot), pos[T*(k+S)]
 * (slot -> pool row or -1). Returns the number of out-of-range expert ids
 * (treated as disabled slots). */
int orc_route(int T, int k, int S, int E, const int32_t* topk_idx,
              int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos);

/* Whole path. Optional intermediates (pool order, NULL to skip):
 *   acc1 [R][2I] float   L1 accumulators (gate | up)
 *   q    [R][I]  uint8   E4M3 L2 activations;  qsf [R][I/32] UE8M0 codes
 *   z    [R][H]  uint16  BF16 L2 outputs per slot row
 * with R = T*(k+S). Rows beyond the valid count are left untouched.
 * With w_fmt 2 the scale arguments hold float32 values (passed as bytes):
 *   x_sf [T][H/128], w1_sf [E+S][2I/128][H/128], w2_sf [E+S][H/128][I/128],
 *   qsf  [R][I/128] (output).
 * Returns the out-of-range count from orc_route, or a negative error. */
int orc_forward(const orc_dims* d, const uint8_t* x, const uint8_t* x_sf, const int32_t* topk_idx,
                const float* topk_w, const uint8_t* w1, const uint8_t* w1_sf, const uint8_t* w2,
                const uint8_t* w2_sf, uint16_t* out, float* acc1, uint8_t* q, uint8_t* qsf, uint16_t* z,
                int nthreads);

/* L2 alone from given E4M3 activations ("MegaMoE on SM100/SM90" research
 * report sec. 4.1, Linear2 phase; "MEGAMOE_SM90_DESIGN" sec. 11.1):
 * acc2[r][h] = sum_i deq(q[r][i]) * deq(W2[e_r][h][i]), float, ascending i;
 * w_fmt as in orc_dims (with w_fmt 2, qsf is float32 [R][I/128] and w2_sf
 * float32 [E][H/128][I/128], and the sum runs per 128-block as in orc_forward).
 * The L2 step of orc_forward computes the same sums, so the BF16 of acc2
 * equals orc_forward's per-slot rows z. */
void orc_l2_rows(int R, int H, int I, int w_fmt, const int32_t* expert_of_row, const uint8_t* q,
                 const uint8_t* qsf, const uint8_t* w2, const uint8_t* w2_sf, float* acc2);

#ifdef __cplusplus
}
#endif
#endif
