// fp8_codec.cuh -- the e4m3 encoding shared by the quantisers (fp8.cu) and the
// expert GEMM epilogue that quantises H at decode sizes (gemm_tc.cu), so both
// produce the same codes: scale = max |v| / 448 over the row or column (1 when
// that maximum is 0), code = e4m3(v / scale) rounded to nearest, ties to even,
// saturating at 448; the division is an fp32 IEEE division.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace moe {

constexpr float kE4M3Max = 448.0f;
// e4m3 weight banks are stored in kFp8Tile x kFp8Tile tiles (fp8.cu).
constexpr int kFp8Tile = 128;

__device__ __forceinline__ float scale_of(float absmax) { return absmax > 0.f ? absmax / kE4M3Max : 1.0f; }

__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// 8 values (16 bytes of bf16) to 8 e4m3 codes.
__device__ __forceinline__ uint2 quant8(uint4 u, float s) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
  uint32_t w[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    const uint32_t q = static_cast<uint32_t>(to_e4m3(f.x / s)) | (static_cast<uint32_t>(to_e4m3(f.y / s)) << 8);
    w[i >> 1] |= q << (16 * (i & 1));
  }
  return make_uint2(w[0], w[1]);
}

}  // namespace moe
