// fp8.cu -- the e4m3 pieces of the FP8-weight variant of the layer: weight
// quantisation (one fp32 scale per output column, codes stored K-contiguous),
// the row gather that quantises each grouped activation row with its own
// scale, and the per-row quantisation of the SwiGLU output H.
//
// Scheme (the pages name FP8 only as deployment work -- paper-graph-ui
// summary, "Inference and Deployment Infrastructure" -- so it is this
// library's): from a = max |v| over the column (weights) or row
// (activations), the dequantisation scale a / 448 and the quantisation factor
// u = 448 / a (both 1 where a is 0, a nonzero a below 2^-100 taken as
// 2^-100); code = e4m3(v * u) rounded to nearest, ties to even, saturating at
// 448 (fp8_codec.cuh).
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "fp8_codec.cuh"
#include "internal.h"
#include "stamps.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// amax[e, n] = max_k |W[e, k, n]| (written into the scales array, which
// scales_from_amax_kernel turns into the scales once the codes are out).
// Block: 64 columns x 4 row phases.
__global__ void __launch_bounds__(256) weight_absmax_kernel(const __nv_bfloat16 *__restrict__ W, int K, int N,
                                                            float *__restrict__ amax) {
  __shared__ float red[4][64];
  const int e = blockIdx.y;
  const int j = threadIdx.x & 63, ph = threadIdx.x >> 6;
  const int n = blockIdx.x * 64 + j;
  float m = 0.f;
  if (n < N) {
    const __nv_bfloat16 *col = W + static_cast<size_t>(e) * K * N + n;
    for (int k = ph; k < K; k += 4) m = fmaxf(m, fabsf(__bfloat162float(col[static_cast<size_t>(k) * N])));
  }
  red[ph][j] = m;
  __syncthreads();
  if (ph == 0 && n < N) {
    const float a = fmaxf(fmaxf(red[0][j], red[1][j]), fmaxf(red[2][j], red[3][j]));
    amax[static_cast<size_t>(e) * N + n] = a;
  }
}

// scales[i] = amax[i] / 448 in place (1 for an all-zero column).
__global__ void __launch_bounds__(256) scales_from_amax_kernel(float *__restrict__ scales, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    scales[i] = scale_of(scales[i]);
}

// Wq holds e4m3(W[e, k, n] * u[e, n]) in 128 x 128 tiles, u = 448 / amax[e, n]: tile (nt, kt)
// of expert e is the contiguous 16 KiB block ((e * Nt + nt) * Kt + kt), inside
// it row n % 128 holds the 128 codes of k = kt*128 .. kt*128 + 127 (zero past
// N or K).  64x64 pieces through shared memory so that both the reads (along
// n) and the writes (along k) coalesce; the grid covers whole tiles.
__global__ void __launch_bounds__(256) weight_quant_kernel(const __nv_bfloat16 *__restrict__ W, int K, int N,
                                                           const float *__restrict__ amax, uint8_t *__restrict__ Wq) {
  __shared__ uint8_t tile[64][65];
  const int e = blockIdx.z;
  const int k0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  const int Nt = (N + kFp8Tile - 1) / kFp8Tile, Kt = (K + kFp8Tile - 1) / kFp8Tile;
  const __nv_bfloat16 *Wb = W + static_cast<size_t>(e) * K * N;
  const int n = n0 + tx;
  const float u = n < N ? inverse_scale_of(amax[static_cast<size_t>(e) * N + n]) : 1.0f;
  for (int i = ty; i < 64; i += 4) {
    const int k = k0 + i;
    uint8_t q = 0;
    if (k < K && n < N) q = to_e4m3(__fmul_rn(__bfloat162float(Wb[static_cast<size_t>(k) * N + n]), u));
    tile[tx][i] = q;  // [n][k]
  }
  __syncthreads();
  for (int i = ty; i < 64; i += 4) {
    const int nn = n0 + i, k = k0 + tx;
    const size_t t = (static_cast<size_t>(e) * Nt + nn / kFp8Tile) * Kt + k / kFp8Tile;
    Wq[t * kFp8Tile * kFp8Tile + (nn % kFp8Tile) * kFp8Tile + k % kFp8Tile] = tile[i][tx];
  }
}

// Rows are processed by teams: one warp per row when there are many rows,
// the whole block per row when there are few (decode), so that either way
// the row's loads spread over many threads.
template <bool BLOCK_TEAM>
struct Team {
  int rank, size, first, stride;  // thread's rank in the team, team size, first row, row stride
  __device__ Team() {
    if (BLOCK_TEAM) {
      rank = threadIdx.x; size = blockDim.x; first = blockIdx.x; stride = gridDim.x;
    } else {
      rank = threadIdx.x & 31; size = 32;
      first = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
      stride = (gridDim.x * blockDim.x) >> 5;
    }
  }
};

// Maximum of v over the team (a warp, or the block: blockDim.x a multiple of
// 32, at most 256).
template <bool BLOCK_TEAM>
__device__ __forceinline__ float team_max(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (!BLOCK_TEAM) return v;
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();  // red is free (an earlier row's readers are done)
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float m = 0.f;
  for (int i = 0; i < nw; ++i) m = fmaxf(m, red[i]);
  return m;
}

__device__ __forceinline__ float absmax8(uint4 u) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

// X_perm8[r, :] = e4m3(x[perm_tok[r], :] * u_r) with xs[r] the row's scale;
// pad rows are zero with scale 0.  One team per grouped row (grid-stride).
template <bool BLOCK_TEAM>
__global__ void __launch_bounds__(256) gather_quant_kernel(const __nv_bfloat16 *__restrict__ x, int T, int d,
                                                           const int32_t *__restrict__ perm_tok,
                                                           const int32_t *__restrict__ poffsets, int E,
                                                           uint8_t *__restrict__ xq, float *__restrict__ xs,
                                                           int *status, unsigned long long *stamps) {
  __shared__ float red[8];
  pdl_wait();
  pdl_trigger();
  stamp_begin(stamps, ST_GATHER);
  const Team<BLOCK_TEAM> tm;
  const int rows = poffsets[E];
  const int nchunk = d / 8;  // 8 bf16 in, 8 codes out
  for (int r = tm.first; r < rows; r += tm.stride) {
    int tok = perm_tok[r];
    if (tok >= T) {
      if (tm.rank == 0) atomicCAS(status, 0, MOE_ERR_DEVICE_BOUNDS);
      tok = -1;
    }
    uint8_t *dst = xq + static_cast<size_t>(r) * d;
    if (tok < 0) {
      for (int c = tm.rank; c < nchunk; c += tm.size) *reinterpret_cast<uint2 *>(dst + 8 * c) = make_uint2(0, 0);
      if (tm.rank == 0) xs[r] = 0.f;
      continue;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(tok) * d);
    float m = 0.f;
    for (int c = tm.rank; c < nchunk; c += tm.size) m = fmaxf(m, absmax8(__ldg(src + c)));
    const float a = team_max<BLOCK_TEAM>(m, red);
    const float u = inverse_scale_of(a);
    for (int c = tm.rank; c < nchunk; c += tm.size) *reinterpret_cast<uint2 *>(dst + 8 * c) = quant8(__ldg(src + c), u);
    if (tm.rank == 0) xs[r] = scale_of(a);
  }
  stamp_end(stamps, ST_GATHER);
}

// Hq[r, :] = e4m3(H[r, :] * u_r) for every real grouped row, with a_r the
// largest of the row's tile maxima habs[r, :] written by the gate/up epilogue
// (the maxima of the bf16 H values), u_r = 448 / a_r and hs[r] = a_r / 448.  One team per
// real row (grid-stride over the T*K real rows, each mapped to its padded
// position; padding rows are left alone, the down projection drops their
// output).  With few rows a row's chunks are split over gridDim.y blocks,
// each taking the row's scale from the tile maxima itself.
template <bool BLOCK_TEAM>
__global__ void __launch_bounds__(256) quant_h_kernel(const __nv_bfloat16 *__restrict__ H, int f,
                                                      const float *__restrict__ habs, int n_tiles,
                                                      const int32_t *__restrict__ offsets,
                                                      const int32_t *__restrict__ poffsets, int E,
                                                      uint8_t *__restrict__ hq, float *__restrict__ hs,
                                                      unsigned long long *stamps) {
  __shared__ float red[8];
  pdl_wait();
  pdl_trigger();
  stamp_begin(stamps, ST_QUANT_H);
  const Team<BLOCK_TEAM> tm;
  const int real_rows = offsets[E];
  const int nchunk = f / 8;
  const int per = (nchunk + gridDim.y - 1) / gridDim.y;
  const int c0 = blockIdx.y * per, c1 = min(nchunk, c0 + per);
  for (int u = tm.first; u < real_rows; u += tm.stride) {
    int e = 0;
    while (e < E - 1 && u >= offsets[e + 1]) ++e;
    const int r = poffsets[e] + (u - offsets[e]);  // padded grouped row
    float m = 0.f;
    for (int t = tm.rank; t < n_tiles; t += tm.size) m = fmaxf(m, habs[static_cast<size_t>(r) * n_tiles + t]);
    const float a = team_max<BLOCK_TEAM>(m, red);
    const float inv = inverse_scale_of(a);
    const uint4 *src = reinterpret_cast<const uint4 *>(H + static_cast<size_t>(r) * f);
    uint8_t *dst = hq + static_cast<size_t>(r) * f;
#pragma unroll 4
    for (int c = c0 + tm.rank; c < c1; c += tm.size) *reinterpret_cast<uint2 *>(dst + 8 * c) = quant8(src[c], inv);
    if (tm.rank == 0 && blockIdx.y == 0) hs[r] = scale_of(a);
  }
  stamp_end(stamps, ST_QUANT_H);
}

}  // namespace

cudaError_t launch_quantize_weights_fp8(const void *W, int E, int K, int N, void *Wq, float *scales,
                                        cudaStream_t s) {
  const dim3 g1((N + 63) / 64, E);
  weight_absmax_kernel<<<g1, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(W), K, N, scales);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // every 64 x 64 piece of the whole tiles (padding included)
  const dim3 g2(2 * ((N + kFp8Tile - 1) / kFp8Tile), 2 * ((K + kFp8Tile - 1) / kFp8Tile), E);
  weight_quant_kernel<<<g2, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(W), K, N, scales,
                                         static_cast<uint8_t *>(Wq));
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t n = static_cast<size_t>(E) * N;
  scales_from_amax_kernel<<<static_cast<unsigned>(std::min<size_t>((n + 255) / 256, 4096)), 256, 0, s>>>(scales, n);
  return cudaGetLastError();
}

cudaError_t launch_gather_quant(const void *x, int T, int d, int E, int R, const Ptrs &P, int num_sms,
                                cudaStream_t s) {
  // A block per row until there are enough rows to give every resident warp
  // about half a row (prefill sizes); a lone warp per row is slow on the few,
  // long rows of decode batches.
  const bool block_team = R <= num_sms * 32;
  int blocks = block_team ? R : (R + 7) / 8;
  if (blocks > num_sms * 8) blocks = num_sms * 8;
  if (blocks < 1) blocks = 1;
  return launch_kernel(block_team ? gather_quant_kernel<true> : gather_quant_kernel<false>, dim3(blocks), dim3(256),
                       0, s, true,
                       static_cast<const __nv_bfloat16 *>(x), T, d, static_cast<const int32_t *>(P.perm_tok),
                       static_cast<const int32_t *>(P.poffsets), E, static_cast<uint8_t *>(P.xperm), P.xscale,
                       P.status, P.stamps);
}

cudaError_t launch_quant_h(int f, int E, int TK, int n_tiles, const Ptrs &P, int num_sms, cudaStream_t s) {
  const bool block_team = TK <= num_sms * 32;  // as launch_gather_quant
  int blocks = block_team ? TK : (TK + 7) / 8;
  if (blocks > num_sms * 8) blocks = num_sms * 8;
  if (blocks < 1) blocks = 1;
  // few rows: split each row over up to 16 blocks, about two blocks per SM in all
  const int parts = block_team ? std::max(1, std::min(16, (2 * num_sms + blocks - 1) / blocks)) : 1;
  return launch_kernel(block_team ? quant_h_kernel<true> : quant_h_kernel<false>, dim3(blocks, parts), dim3(256), 0,
                       s, true,
                       static_cast<const __nv_bfloat16 *>(P.hbuf), f, static_cast<const float *>(P.habs), n_tiles,
                       static_cast<const int32_t *>(P.offsets), static_cast<const int32_t *>(P.poffsets), E,
                       static_cast<uint8_t *>(P.hq), P.hscale, P.stamps);
}

}  // namespace moe
