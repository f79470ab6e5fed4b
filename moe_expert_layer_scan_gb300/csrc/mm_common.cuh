// Device helpers shared by the GEMM kernels: the tile decode of the grouped
// GEMMs' tile tables, 16-byte shared-memory stores and the UE8M0 requantiser.
#pragma once

#include <cstdint>

#include "mm_ptx.cuh"

namespace mm {

struct Tile {
  int e, fb, row0, nrows;
  bool active;  // this CTA has a weight tile (fb < fb_total)
};

// Tile index -> expert, token tile and weight tile. The tile table (in tile
// order: position j holds expert eorder[j]) and the row offsets are
// shared-memory copies. An expert's rows are
// split into the fewest token tiles of at most bn rows, all of one size
// rounded up to 16 (the last takes the rest): 256 rows with bn = 224 give two
// tiles of 128, not 224 + 32 (a tile costs its weight stream and a per-K-step
// instruction floor whatever its row count).
static __device__ __noinline__ Tile decode_tile(int tile, const int* tstart, const int32_t* eorder, const int* offs,
                                           int Ep, int fb_total, int bn) {
  int lo = 0, hi = Ep - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tstart[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  Tile t;
  t.e = eorder ? eorder[lo] : lo;  // (null: the tile order is the expert order)
  const int local = tile - tstart[lo];
  const int cnt = offs[t.e + 1] - offs[t.e];
  const int ntt = (cnt + bn - 1) / bn;
  t.fb = local / ntt;
  const int tt = local - t.fb * ntt;
  t.active = t.fb < fb_total;
  const int per = ((cnt + ntt - 1) / ntt + 15) & ~15;  // <= bn, and (ntt - 1) * per < cnt
  t.row0 = offs[t.e] + tt * per;
  t.nrows = min(per, cnt - tt * per);
  return t;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int c) {
  return c == 0 ? v.x : (c == 1 ? v.y : (c == 2 ? v.z : v.w));
}

__device__ __forceinline__ void st_shared_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// One byte per (row, feature) from a chunk held feature-per-lane: lane l's
// w[c] packs the bytes of feature f0 + l for rows c0 + 4c .. c0 + 4c + 3
// (byte i: row c0 + 4c + i). Each group of four lanes transposes its 4 x 4
// blocks (two exchange steps, byte permutes) so that lane 4a + r writes
// features f0 + 4a .. f0 + 4a + 3 of row c0 + 4c + r as one 4-byte store.
// Rows at or beyond c0 + nvalid are not written. All 32 lanes call it.
template <int NW>
__device__ __forceinline__ void store_u8_rows_4x4(uint8_t* q, size_t ld, int row0, int c0, int nvalid, int f0,
                                                  const uint32_t (&w)[NW]) {
  const int lane = threadIdx.x & 31;
  const bool odd = (lane & 1) != 0, hi = (lane & 2) != 0;
#pragma unroll
  for (int c = 0; c < NW; ++c) {
    // step 1 (lanes 2m, 2m + 1): the even lane keeps rows 0 and 2 of the
    // group, the odd lane rows 1 and 3, each with both lanes' features
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, w[c], 1);
    const uint32_t x = odd ? __byte_perm(w[c], r1, 0x3715) : __byte_perm(w[c], r1, 0x6240);
    // step 2 (lanes 4a + b, 4a + b + 2): the lower lane keeps row b, the
    // upper row b + 2, each with all four features
    const uint32_t r2 = __shfl_xor_sync(0xffffffffu, x, 2);
    const uint32_t out = hi ? __byte_perm(x, r2, 0x3276) : __byte_perm(x, r2, 0x5410);
    const int row = 4 * c + (lane & 3);
    if (row < nvalid) *reinterpret_cast<uint32_t*>(q + (size_t)(row0 + c0 + row) * ld + f0 + (lane & ~3)) = out;
  }
}

// UE8M0 code of the smallest power of two >= amax / 448 (IEEE quotient),
// 127 for amax == 0, clamped to [1, 254].
__device__ __forceinline__ uint32_t requant_code(float amax) {
  if (!(amax > 0.0f)) return 127u;
  const uint32_t b = __float_as_uint(__fdiv_rn(amax, 448.0f));
  const int e = (int)(b >> 23);
  int code = (e == 0) ? 1 : (((b & 0x7FFFFFu) == 0u) ? e : e + 1);
  code = code < 1 ? 1 : (code > 254 ? 254 : code);
  return (uint32_t)code;
}

// 2^(127 - code) exactly (a normal or subnormal float for code in [1, 254]).
__device__ __forceinline__ float inv_scale(uint32_t code) {
  const int n = 127 - (int)code;
  return n >= -126 ? __uint_as_float((uint32_t)(n + 127) << 23) : __uint_as_float(1u << (n + 149));
}

}  // namespace mm
