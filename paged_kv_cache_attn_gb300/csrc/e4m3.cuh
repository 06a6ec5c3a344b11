// Device helpers for e4m3 pools: the scale exponent rule, the tile byte
// layouts, element conversions and the warp-wide quantising tile write.
//
// Format and rule (kv_pool_desc in pagedkv.h): a stored value is
// code value x 2^e, one e per (layer, block, kv-head) and tensor, the
// smallest e in [-126, 120] with max|x| <= 448 x 2^e.  A write that starts a
// block (slot 0) takes the exponent of its own rows; a later write keeps the
// block's exponent unless its rows need a larger one, and then re-encodes the
// rows already stored.  Codes are the nearest e4m3 value of x x 2^-e, ties to
// the even mantissa (the hardware conversion with satfinite).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace pkv {

constexpr int kE4m3EMin = -126;
constexpr int kE4m3EMax = 120;

// Smallest e in [-126, 120] with amax <= 448 * 2^e, from the bits of amax:
// amax = (1 + M / 2^23) 2^(E - 127) = m 2^k with m = (1 + M / 2^23) / 2 and
// k = E - 126; 448 = 0.875 x 2^9, so e = k - 9 when m <= 0.875
// (M <= 0x600000), else k - 8.  Zero and subnormal amax (< 2^-126) take the
// lower bound.
__device__ __forceinline__ int e4m3_exponent_for(float amax) {
  const uint32_t bits = __float_as_uint(amax) & 0x7fffffffu;
  const int E = (int)(bits >> 23);
  if (E == 0) return kE4m3EMin;
  const int e = (bits & 0x7fffffu) <= 0x600000u ? E - 135 : E - 134;
  return e < kE4m3EMin ? kE4m3EMin : (e > kE4m3EMax ? kE4m3EMax : e);
}

// 2^e as a float, e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) {
  return __uint_as_float((uint32_t)(e + 127) << 23);
}

// Exponent of a stored scale 2^e (a normal float).
__device__ __forceinline__ int scale_exponent(float s) {
  return (int)((__float_as_uint(s) >> 23) & 0xff) - 127;
}

__device__ __forceinline__ uint8_t e4m3_encode(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_decode(uint8_t c) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

// Four codes (bytes 0..3 of w) -> two f16x2, exactly: lo = (byte 0, byte 1),
// hi = (byte 2, byte 3), the lower byte in the lower half.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo,
                                                  uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Byte offset of (slot t, dimension c) inside a K tile / a V tile.
__device__ __forceinline__ int k_tile_offset(int t, int c, int d) {
  if (d == 128) return t * 128 + ((((c >> 4) ^ (t & 7))) << 4) + (c & 15);
  return t * d + c;
}
__device__ __forceinline__ int v_tile_offset(int t, int c) { return c * 16 + t; }

// Warp-wide: write rows[0 .. s1 - s0) (bf16, row r at rows + r * row_stride,
// d values) into slots [s0, s1) of one e4m3 tile `codes` whose scale is
// *scale.  Applies the block rule; every lane must call it.
__device__ inline void e4m3_tile_write(uint8_t* codes, float* scale, int s0,
                                       int s1, const __nv_bfloat16* rows,
                                       int64_t row_stride, int d, bool is_v,
                                       int lane) {
  const int n = s1 - s0;
  const int lg = d == 128 ? 7 : 6;
  float amax = 0.f;
  for (int i = lane; i < n * d; i += 32) {
    const int r = i >> lg, c = i & (d - 1);
    amax = fmaxf(amax, fabsf(__bfloat162float(rows[r * row_stride + c])));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e_req = e4m3_exponent_for(amax);
  int e = e_req;
  if (s0 > 0) {
    const int e_old = scale_exponent(*scale);
    if (e_old >= e_req) {
      e = e_old;
    } else {
      // Re-encode the stored rows under the larger scale: a pure exponent
      // shift of their stored values (exact while they stay normal).
      const int sh = e_old - e;
      for (int i = lane; i < s0 * d; i += 32) {
        const int t = i >> lg, c = i & (d - 1);
        const int off = is_v ? v_tile_offset(t, c) : k_tile_offset(t, c, d);
        codes[off] = e4m3_encode(ldexpf(e4m3_decode(codes[off]), sh));
      }
    }
  }
  const float inv = pow2f(-e);
  for (int i = lane; i < n * d; i += 32) {
    const int r = i >> lg, c = i & (d - 1);
    const int t = s0 + r;
    const int off = is_v ? v_tile_offset(t, c) : k_tile_offset(t, c, d);
    codes[off] = e4m3_encode(__bfloat162float(rows[r * row_stride + c]) * inv);
  }
  __syncwarp();
  if (lane == 0) *scale = pow2f(e);
  __syncwarp();
}

}  // namespace pkv
