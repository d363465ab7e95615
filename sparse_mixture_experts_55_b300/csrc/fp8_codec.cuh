// fp8_codec.cuh -- the e4m3 encoding of the quantisers (fp8.cu): from a row's
// or column's largest magnitude a, the dequantisation scale s = a / 448 and
// the quantisation factor u = 448 / a (both 1 when a is 0; a nonzero a below
// 2^-100 counts as 2^-100 so that u stays finite), and code = e4m3(v * u)
// rounded to nearest, ties to even, saturating at 448.  The two divisions are
// fp32 IEEE divisions made once per row or column; the product that decides
// each code is one fp32 multiply.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace moe {

constexpr float kE4M3Max = 448.0f;
// e4m3 weight banks are stored in kFp8Tile x kFp8Tile tiles (fp8.cu).
constexpr int kFp8Tile = 128;

constexpr float kAmaxFloor = 0x1p-100f;

__device__ __forceinline__ float amax_used(float absmax) {
  return absmax > 0.f ? fmaxf(absmax, kAmaxFloor) : kE4M3Max;
}
__device__ __forceinline__ float scale_of(float absmax) { return amax_used(absmax) / kE4M3Max; }
__device__ __forceinline__ float inverse_scale_of(float absmax) { return kE4M3Max / amax_used(absmax); }

__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// 8 values (16 bytes of bf16) to 8 e4m3 codes, u the quantisation factor.
__device__ __forceinline__ uint2 quant8(uint4 u, float inv) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
  uint32_t w[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    const uint32_t q = static_cast<uint32_t>(to_e4m3(__fmul_rn(f.x, inv))) |
                       (static_cast<uint32_t>(to_e4m3(__fmul_rn(f.y, inv))) << 8);
    w[i >> 1] |= q << (16 * (i & 1));
  }
  return make_uint2(w[0], w[1]);
}

}  // namespace moe
