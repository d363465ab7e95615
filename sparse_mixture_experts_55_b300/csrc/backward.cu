// backward.cu -- the non-GEMM steps of the MoE layer's backward pass (bf16
// layer, fp32 gradients), around the grouped GEMMs of gemm_bwd.cu.
//
// The forward computes y = sum_k G_k O_k with O_k = E_{e_k}(x) the expert
// output of slot k and G = softmax over the K kept router logits l = x Wg
// (section 3.4 "MoE Layer Formulation"; routing of "Sparse Mixture of Experts
// Architecture", Mixtral of Experts summary pages).  The selected set has no
// gradient.  With the saved gate-scaled outputs P_k = G_k O_k and dy = dL/dy:
//   dL/dG_k = <dy, O_k>, so G_k dL/dG_k = <dy, P_k>, and the softmax backward
//   dL/dl_k = G_k (dL/dG_k - sum_j G_j dL/dG_j) = <dy, P_k> - G_k <dy, sum_j P_j>
//   needs no division by a gate;
//   dL/dE_{e_k}(x) = G_k dy is the expert's output gradient dY (bf16, the A
//   operand of the expert dgrad and the B operand of the W2 wgrad);
//   dx = sum_k dX_k + dL/dl Wg^T, dWg = x^T dL/dl.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void unpack8(const uint4 w, float (&v)[8]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ws[j]));
    v[2 * j] = p.x;
    v[2 * j + 1] = p.y;
  }
}

// One warp per token: dL/dl for its row of [T, E] (zero off the selected
// experts) and the rows dY = G_k dy of its K grouped rows; then the padding
// rows of dY are cleared.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ dy, int T, int d, int E,
                                                       int K, int S, long long split_stride,
                                                       const float *__restrict__ obuf, const float *__restrict__ gate,
                                                       const int32_t *__restrict__ idx, const int32_t *__restrict__ pos,
                                                       const int32_t *__restrict__ offsets,
                                                       const int32_t *__restrict__ poffsets, float *__restrict__ dl,
                                                       __nv_bfloat16 *__restrict__ dye, int *status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int nchunk = d / 8;
  for (int t = gw; t < T; t += nw) {
    int ek[kMaxK], uk[kMaxK], prow[kMaxK];
    float gk[kMaxK], p[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      ek[k] = -1;
      uk[k] = 0;
      prow[k] = -1;
      gk[k] = 0.f;
      p[k] = 0.f;
      if (k >= K) continue;
      const int e = idx[t * K + k], u = pos[t * K + k];
      if (e < 0 || e >= E || u < offsets[e] || u >= offsets[e + 1]) {
        if (lane == 0) atomicCAS(status, 0, MOE_ERR_DEVICE_BOUNDS);
        continue;
      }
      ek[k] = e;
      uk[k] = u;
      prow[k] = poffsets[e] + (u - offsets[e]);
      gk[k] = gate[t * K + k];
    }
    const uint4 *dyr = reinterpret_cast<const uint4 *>(dy + static_cast<size_t>(t) * d);
    for (int c = lane; c < nchunk; c += 32) {
      float dv[8];
      unpack8(__ldg(dyr + c), dv);
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        if (ek[k] < 0) continue;
        const float *o = obuf + static_cast<size_t>(uk[k]) * d + 8 * c;
        float4 o0 = __ldg(reinterpret_cast<const float4 *>(o));
        float4 o1 = __ldg(reinterpret_cast<const float4 *>(o + 4));
        for (int s = 1; s < S; ++s) {  // the down projection's split partials, in split order
          const float4 a = __ldg(reinterpret_cast<const float4 *>(o + s * split_stride));
          const float4 b = __ldg(reinterpret_cast<const float4 *>(o + s * split_stride + 4));
          o0.x += a.x; o0.y += a.y; o0.z += a.z; o0.w += a.w;
          o1.x += b.x; o1.y += b.y; o1.z += b.z; o1.w += b.w;
        }
        p[k] += dv[0] * o0.x + dv[1] * o0.y + dv[2] * o0.z + dv[3] * o0.w + dv[4] * o1.x + dv[5] * o1.y +
                dv[6] * o1.z + dv[7] * o1.w;
      }
    }
    float yy = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) p[k] += __shfl_xor_sync(0xffffffffu, p[k], o);
      yy += p[k];
    }
    for (int e = lane; e < E; e += 32) {
      float v = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxK; ++k)
        if (ek[k] == e) v = p[k] - gk[k] * yy;
      dl[static_cast<size_t>(t) * E + e] = v;
    }
    for (int c = lane; c < nchunk; c += 32) {
      float dv[8];
      unpack8(__ldg(dyr + c), dv);
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) {
        if (ek[k] < 0) continue;
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(gk[k] * dv[2 * j], gk[k] * dv[2 * j + 1]);
          w[j] = *reinterpret_cast<const uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(dye + static_cast<size_t>(prow[k]) * d + 8 * c) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  // padding rows of every segment: zeros (the weight gradients contract over them)
  const int rows = poffsets[E];
  for (int r = gw; r < rows; r += nw) {
    int e = 0;
    while (e < E - 1 && r >= poffsets[e + 1]) ++e;
    if (r - poffsets[e] < offsets[e + 1] - offsets[e]) continue;
    uint4 *dst = reinterpret_cast<uint4 *>(dye + static_cast<size_t>(r) * d);
    for (int c = lane; c < nchunk; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
  }
}

// dx[t, :] = sum_k dX[u_k, :] + sum_e dl[t, e] Wg[:, e]; one thread per four columns.
__global__ void __launch_bounds__(256) bwd_dx_kernel(const float *__restrict__ dxc, const int32_t *__restrict__ pos,
                                                     const float *__restrict__ dl, const __nv_bfloat16 *__restrict__ Wg,
                                                     int T, int d, int E, int K, int TK, float *__restrict__ dx,
                                                     int accumulate, int *status) {
  pdl_wait();
  pdl_trigger();
  const int q = d >> 2;
  const long long total = static_cast<long long>(T) * q;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / q);
    const int c = static_cast<int>(i - static_cast<long long>(t) * q) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; ++k) {
      const int u = pos[t * K + k];
      if (u < 0 || u >= TK) {
        atomicCAS(status, 0, MOE_ERR_DEVICE_BOUNDS);
        continue;
      }
      const float4 v = __ldg(reinterpret_cast<const float4 *>(dxc + static_cast<size_t>(u) * d + c));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    for (int e = 0; e < E; ++e) {
      const float g = dl[static_cast<size_t>(t) * E + e];
      if (g == 0.f) continue;  // the experts a token did not select
      const __nv_bfloat16 *w = Wg + static_cast<size_t>(c) * E + e;
      acc.x += g * __bfloat162float(w[0]);
      acc.y += g * __bfloat162float(w[E]);
      acc.z += g * __bfloat162float(w[2 * E]);
      acc.w += g * __bfloat162float(w[3 * E]);
    }
    float4 *dst = reinterpret_cast<float4 *>(dx + static_cast<size_t>(t) * d + c);
    if (accumulate) {
      const float4 o = *dst;
      acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
    }
    *dst = acc;
  }
}

constexpr int kDwgThreads = 128;  // two columns each
constexpr int kDwgStage = 64;     // tokens of dl staged in shared memory at a time

// part[ch, i, e] = sum over the tokens of chunk ch of x[t, i] dl[t, e].
__global__ void __launch_bounds__(kDwgThreads) bwd_dwg_part_kernel(const __nv_bfloat16 *__restrict__ x,
                                                                   const float *__restrict__ dl, int T, int d, int E,
                                                                   int tokens_per_chunk, float *__restrict__ part) {
  __shared__ float sdl[kDwgStage * kMaxE];
  pdl_wait();
  pdl_trigger();
  const int i0 = 2 * (blockIdx.x * kDwgThreads + threadIdx.x);
  const int ch = blockIdx.y;
  const int t0 = ch * tokens_per_chunk;
  const int t1 = min(T, t0 + tokens_per_chunk);
  float a0[kMaxE], a1[kMaxE];
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) { a0[e] = 0.f; a1[e] = 0.f; }
  for (int tb = t0; tb < t1; tb += kDwgStage) {
    const int n = min(kDwgStage, t1 - tb);
    __syncthreads();
    for (int j = threadIdx.x; j < n * E; j += kDwgThreads) sdl[j] = dl[static_cast<size_t>(tb) * E + j];
    __syncthreads();
    if (i0 < d) {
      for (int tt = 0; tt < n; ++tt) {
        const float2 xv =
            __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(x + static_cast<size_t>(tb + tt) * d + i0));
#pragma unroll
        for (int e = 0; e < kMaxE; ++e) {
          if (e < E) {
            const float g = sdl[tt * E + e];
            a0[e] = fmaf(xv.x, g, a0[e]);
            a1[e] = fmaf(xv.y, g, a1[e]);
          }
        }
      }
    }
  }
  if (i0 < d) {
    float *dst = part + (static_cast<size_t>(ch) * d + i0) * E;
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) {
      if (e < E) {
        dst[e] = a0[e];
        dst[E + e] = a1[e];
      }
    }
  }
}

// dWg[i, e] = sum over chunks, in order, of part[ch, i, e].
__global__ void __launch_bounds__(256) bwd_dwg_reduce_kernel(const float *__restrict__ part, int d, int E, int chunks,
                                                             float *__restrict__ dWg, int accumulate) {
  pdl_wait();
  pdl_trigger();
  const int n = d * E;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int ch = 0; ch < chunks; ++ch) s += part[static_cast<size_t>(ch) * n + i];
    if (accumulate) s += dWg[i];
    dWg[i] = s;
  }
}

}  // namespace

cudaError_t launch_bwd_prep(const void *dy, int T, int d, int E, int K, int S, const WsLayout &L, const Ptrs &P,
                            int num_sms, cudaStream_t s) {
  const int rows_warps = T > L.R ? T : L.R;  // one warp per token, then per grouped row
  int blocks = (rows_warps + 7) / 8;
  if (blocks > num_sms * 8) blocks = num_sms * 8;
  if (blocks < 1) blocks = 1;
  const long long split_stride = static_cast<long long>(T) * K * d;
  return launch_kernel(bwd_prep_kernel, dim3(blocks), dim3(256), 0, s, true, static_cast<const __nv_bfloat16 *>(dy), T,
                       d, E, K, S, split_stride, static_cast<const float *>(P.obuf), static_cast<const float *>(P.gate),
                       static_cast<const int32_t *>(P.idx), static_cast<const int32_t *>(P.pos),
                       static_cast<const int32_t *>(P.offsets), static_cast<const int32_t *>(P.poffsets), P.dl,
                       static_cast<__nv_bfloat16 *>(P.dye), P.status);
}

cudaError_t launch_bwd_input(const void *x, const void *Wg, void *dx, void *dWg, int T, int d, int E, int K,
                             bool accumulate, const WsLayout &L, const Ptrs &P, int num_sms, cudaStream_t s,
                             void *const *events) {
  const long long total = static_cast<long long>(T) * (d / 4);
  long long blocks = (total + 255) / 256;
  if (blocks > num_sms * 16LL) blocks = num_sms * 16LL;
  if (blocks < 1) blocks = 1;
  cudaError_t err = launch_kernel(bwd_dx_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, true,
                                  static_cast<const float *>(P.dxc), static_cast<const int32_t *>(P.pos),
                                  static_cast<const float *>(P.dl), static_cast<const __nv_bfloat16 *>(Wg), T, d, E, K,
                                  T * K, static_cast<float *>(dx), accumulate ? 1 : 0, P.status);
  if (err == cudaSuccess && events) err = cudaEventRecord(static_cast<cudaEvent_t>(events[0]), s);
  if (err != cudaSuccess) return err;
  const int chunks = L.dwg_chunks;
  const int tpc = (T + chunks - 1) / chunks;
  const dim3 g1((d / 2 + kDwgThreads - 1) / kDwgThreads, chunks);
  err = launch_kernel(bwd_dwg_part_kernel, g1, dim3(kDwgThreads), 0, s, true, static_cast<const __nv_bfloat16 *>(x),
                      static_cast<const float *>(P.dl), T, d, E, tpc, P.dwg_part);
  if (err != cudaSuccess) return err;
  int rb = (d * E + 255) / 256;
  if (rb > num_sms * 8) rb = num_sms * 8;
  err = launch_kernel(bwd_dwg_reduce_kernel, dim3(rb), dim3(256), 0, s, true, static_cast<const float *>(P.dwg_part),
                      d, E, chunks, static_cast<float *>(dWg), accumulate ? 1 : 0);
  if (err == cudaSuccess && events) err = cudaEventRecord(static_cast<cudaEvent_t>(events[1]), s);
  return err;
}

}  // namespace moe
