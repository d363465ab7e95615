// gemm_simt.cu -- the expert FFN of the fp32 path on the CUDA cores (plain
// fp32 FMA, no TF32), for the exact-arithmetic small configurations.
//
//   gate/up:  H[r, n] = SiLU(sum_k X[r,k] W1[e,k,n]) * sum_k X[r,k] W3[e,k,n]
//   down:     O[u, n] = gate[r] * sum_k H[r,k] W2[e,k,n]
// ("Expert Network Structure (SwiGLU)", Mixtral of Experts summary pages), for
// every grouped row r of expert e's padded segment; the down projection stores
// only real rows, at their unpadded grouped row u (compact output).
#include <cuda_runtime.h>

#include "internal.h"
#include "stamps.cuh"

namespace moe {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

template <bool GATE_UP>
__global__ void __launch_bounds__(256) ffn_f32_kernel(const float *__restrict__ A, const float *__restrict__ B0,
                                                      const float *__restrict__ B1, int k_total, int n_out,
                                                      const int32_t *__restrict__ poffsets,
                                                      const int32_t *__restrict__ offsets, int E,
                                                      const float *__restrict__ perm_gate, float *__restrict__ out,
                                                      unsigned long long *stamps) {
  __shared__ float As[TK][TM];
  __shared__ float Bs0[TK][TN];
  __shared__ float Bs1[GATE_UP ? TK : 1][GATE_UP ? TN : 1];
  const int row0 = blockIdx.y * TM;
  if (row0 >= poffsets[E]) return;  // whole block
  stamp_begin(stamps, GATE_UP ? ST_GATE_UP : ST_DOWN);
  int e = 0;
  while (row0 >= poffsets[e + 1]) ++e;
  const int n0 = blockIdx.x * TN;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const float *W0 = B0 + static_cast<size_t>(e) * k_total * n_out;
  const float *W1 = GATE_UP ? B1 + static_cast<size_t>(e) * k_total * n_out : nullptr;
  float acc0[4][4] = {}, acc1[4][4] = {};
  for (int k0 = 0; k0 < k_total; k0 += TK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * 256;
      const int r = idx / TK, kk = idx % TK;
      As[kk][r] = (k0 + kk < k_total) ? A[static_cast<size_t>(row0 + r) * k_total + k0 + kk] : 0.f;
      const int kb = idx / TN, n = idx % TN;
      const bool in = (k0 + kb < k_total) && (n0 + n < n_out);
      Bs0[kb][n] = in ? W0[static_cast<size_t>(k0 + kb) * n_out + n0 + n] : 0.f;
      if (GATE_UP) Bs1[kb][n] = in ? W1[static_cast<size_t>(k0 + kb) * n_out + n0 + n] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b0[4], b1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b0[j] = Bs0[kk][tx * 4 + j];
        if (GATE_UP) b1[j] = Bs1[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc0[i][j] = fmaf(a[i], b0[j], acc0[i][j]);
          if (GATE_UP) acc1[i][j] = fmaf(a[i], b1[j], acc1[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    const int seg_row = r - poffsets[e];
    if (!GATE_UP && seg_row >= offsets[e + 1] - offsets[e]) continue;  // padding row
    const int r_out = GATE_UP ? r : offsets[e] + seg_row;
    const float gsc = GATE_UP ? 1.f : perm_gate[r];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= n_out) continue;
      float v;
      if (GATE_UP) {
        const float g = acc0[i][j];
        v = g / (1.0f + expf(-g)) * acc1[i][j];
      } else {
        v = acc0[i][j] * gsc;
      }
      out[static_cast<size_t>(r_out) * n_out + n] = v;
    }
  }
  stamp_end(stamps, GATE_UP ? ST_GATE_UP : ST_DOWN);
}

}  // namespace

cudaError_t launch_expert_ffn_f32(const void *W1, const void *W3, const void *W2, int d, int f, int E,
                                  const WsLayout &L, const Ptrs &P, cudaStream_t s) {
  const dim3 g1((f + TN - 1) / TN, L.R / TM);
  ffn_f32_kernel<true><<<g1, 256, 0, s>>>(static_cast<const float *>(P.xperm), static_cast<const float *>(W1),
                                          static_cast<const float *>(W3), d, f, P.poffsets, P.offsets, E, P.perm_gate,
                                          static_cast<float *>(P.hbuf), P.stamps);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const dim3 g2((d + TN - 1) / TN, L.R / TM);
  ffn_f32_kernel<false><<<g2, 256, 0, s>>>(static_cast<const float *>(P.hbuf), static_cast<const float *>(W2),
                                           nullptr, f, d, P.poffsets, P.offsets, E, P.perm_gate, P.obuf, P.stamps);
  return cudaGetLastError();
}

}  // namespace moe
