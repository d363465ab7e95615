// routing.cu -- the router (logits, top-K with lower-index ties, softmax over
// the kept logits), the stable grouping of (token, slot) pairs by expert, the
// row gather into the grouped activation buffer, the deterministic two-slot
// combine, and RMSNorm.
//
// Method: Mixtral of Experts (arXiv 2401.04088), paper-graph-ui summary,
// section 3.4 "MoE Layer Formulation" (G(x) = Softmax(TopK(x . W_g)),
// y = sum_i G(x)_i E_i(x)) and "Top-K Gating Mechanism and Routing" (the
// three-step Top-2 procedure); grouping tokens by expert follows
// "Inference and Deployment Infrastructure" (all experts' inputs packed into
// one matrix).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "stamps.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void set_status(int *status, int code) { atomicCAS(status, 0, code); }

// Programmatic dependent launch: wait for the previous kernel in the stream
// before touching its outputs, and let the next kernel start its prologue.
// Both are no-ops when the kernel was launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename Tin>
struct Vec;  // one 16-byte vector of inputs
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16 *p, float (&v)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void load(const float *p, float (&v)[4]) {
    float4 u = __ldg(reinterpret_cast<const float4 *>(p));
    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
  }
};

// Router rows of this thread's d-slice: w[c][e] = W_g[j0 + c, e] as fp32.
template <typename Tin, int EP>
__device__ __forceinline__ void load_router_rows(const Tin *__restrict__ Wg, int j0, int E, bool valid,
                                                 float (&w)[Vec<Tin>::N][EP]) {
  constexpr int NV = Vec<Tin>::N;
#pragma unroll
  for (int c = 0; c < NV; ++c)
#pragma unroll
    for (int e = 0; e < EP; ++e) w[c][e] = 0.f;
  if (!valid) return;
  if (sizeof(Tin) == 2 && EP == 8 && E == 8) {
#pragma unroll
    for (int c = 0; c < NV; ++c) {  // one 16-byte row per d index
      float r[8];
      Vec<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16 *>(Wg) + static_cast<size_t>(j0 + c) * 8, r);
#pragma unroll
      for (int e = 0; e < 8; ++e) w[c][e] = r[e];
    }
  } else {
#pragma unroll
    for (int c = 0; c < NV; ++c)
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (e < E) w[c][e] = to_f(Wg[static_cast<size_t>(j0 + c) * E + e]);
  }
}

template <typename Tin>
__device__ __forceinline__ uint4 load_raw(const Tin *p, bool valid) {
  return valid ? __ldg(reinterpret_cast<const uint4 *>(p)) : make_uint4(0, 0, 0, 0);
}

template <typename Tin>
__device__ __forceinline__ void unpack(uint4 raw, float (&xv)[Vec<Tin>::N]) {
  if constexpr (sizeof(Tin) == 2) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      xv[2 * i] = f.x;
      xv[2 * i + 1] = f.y;
    }
  } else {
    xv[0] = __uint_as_float(raw.x); xv[1] = __uint_as_float(raw.y);
    xv[2] = __uint_as_float(raw.z); xv[3] = __uint_as_float(raw.w);
  }
}

// a[e] += sum_c x[c] * w[c][e] for one 16-byte chunk of x.
template <typename Tin, int EP>
__device__ __forceinline__ void dot_chunk(uint4 raw, const float (&w)[Vec<Tin>::N][EP], float (&a)[EP]) {
  constexpr int NV = Vec<Tin>::N;
  float xv[NV];
  unpack<Tin>(raw, xv);
#pragma unroll
  for (int c = 0; c < NV; ++c)
#pragma unroll
    for (int e = 0; e < EP; ++e) a[e] = fmaf(xv[c], w[c][e], a[e]);
}

// The same with the W_g rows streamed from L1 one at a time (no register copy).
template <typename Tin, int EP>
__device__ __forceinline__ void dot_chunk_streamed(uint4 raw, const Tin *__restrict__ Wg, int j0, int E,
                                                   float (&a)[EP]) {
  constexpr int NV = Vec<Tin>::N;
  float xv[NV];
  unpack<Tin>(raw, xv);
#pragma unroll
  for (int c = 0; c < NV; ++c) {
    const Tin *row = Wg + static_cast<size_t>(j0 + c) * E;
#pragma unroll
    for (int e = 0; e < EP; ++e)
      if (e < E) a[e] = fmaf(xv[c], to_f(__ldg(row + e)), a[e]);
  }
}

// Warp reduce-scatter of EP partial logits: afterwards lane l holds the warp's
// sum for expert `expert` (32 / EP lanes per expert hold the same value).
// log2(EP) halving steps, then full reduction over the remaining lane bits.
template <int EP>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[EP], int lane, int &expert) {
  int base = 0;
#pragma unroll
  for (int w = EP, m = 16; w > 1; w >>= 1, m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < w / 2; ++i) {
      const float send = upper ? v[i] : v[i + w / 2];
      const float keep = upper ? v[i + w / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
    if (upper) base += w / 2;
  }
#pragma unroll
  for (int m = 16 / EP; m > 0; m >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
  expert = base;
  return v[0];
}

// Top-K (K <= 2) of the E logits with lower-index tie-break, softmax over the
// kept logits, and the per-block expert histogram.
template <int EP>
__device__ __forceinline__ void select_and_store(const float (&l)[EP], int t, int E, int K, unsigned flags,
                                                 int32_t *idx, float *gate, int *s_cnt, int *status) {
  if (flags & MOE_DEBUG_CHECKS) {
#pragma unroll
    for (int e = 0; e < EP; ++e)
      if (e < E && !isfinite(l[e])) set_status(status, MOE_ERR_NONFINITE);
  }
  int i1 = 0;
  float v1 = l[0];
#pragma unroll
  for (int e = 1; e < EP; ++e)
    if (e < E && l[e] > v1) { v1 = l[e]; i1 = e; }
  if (K == 1) {
    idx[t] = i1;
    gate[t] = 1.0f;
    atomicAdd(&s_cnt[i1], 1);
    return;
  }
  int i2 = -1;
  float v2 = 0.f;
#pragma unroll
  for (int e = 0; e < EP; ++e)
    if (e < E && e != i1 && (i2 < 0 || l[e] > v2)) { v2 = l[e]; i2 = e; }
  // softmax over {v1, v2}: g1 = e^v1 / (e^v1 + e^v2) = 1 / (1 + e^(v2 - v1)), g2 = 1 - g1
  const float g1 = 1.0f / (1.0f + expf(v2 - v1));
  idx[2 * t] = i1;
  idx[2 * t + 1] = i2;
  gate[2 * t] = g1;
  gate[2 * t + 1] = 1.0f - g1;
  atomicAdd(&s_cnt[i1], 1);
  atomicAdd(&s_cnt[i2], 1);
}

// One block routes tpb consecutive tokens.  Thread i owns the i-th 16-byte slice
// of d (8 bf16 or 4 fp32 columns).  With up to 8 experts it keeps its rows of
// W_g in registers for all the block's tokens.  The tokens go by in chunks of
// CH: every warp runs through a chunk's tokens with the x slices of the next
// kRouteGroup tokens in flight, reduce-scatters each token's partial logits
// and parks its warp sums in shared memory; one barrier per chunk, then the
// warp sums of each logit are added in a fixed order (so the logits are
// deterministic) and the chunk's tokens are selected.
template <typename Tin, int EP>
__device__ __forceinline__ void route_body(const Tin *__restrict__ x, const Tin *__restrict__ Wg, int T, int d,
                                           int E, int K, int tpb, unsigned flags, int32_t *__restrict__ idx,
                                           float *__restrict__ gate, int32_t *__restrict__ blockcounts, int *status,
                                           unsigned long long *stamps) {
  constexpr int NV = Vec<Tin>::N;
  constexpr int NW = kRouteThreads / 32;
  constexpr int G = kRouteGroup;       // x slices in flight per thread
  constexpr int CH = EP <= 8 ? 32 : 8;  // tokens per chunk (partials in shared memory)
  constexpr bool kCached = EP == 8;
  __shared__ float s_red[CH][NW][EP];
  __shared__ float s_log[CH][EP];
  __shared__ int s_cnt[kMaxE];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * tpb;
  const int nt = min(tpb, T - t0);
  const int nchunks = d / NV;
  if (tid < kMaxE) s_cnt[tid] = 0;
  pdl_wait();
  pdl_trigger();
  stamp_begin(stamps, ST_ROUTE);

  const bool own = tid < nchunks;
  float w[kCached ? NV : 1][kCached ? EP : 1];
  if constexpr (kCached) load_router_rows<Tin, EP>(Wg, tid * NV, E, own, w);
  const Tin *xb = x + static_cast<size_t>(t0) * d + tid * NV;
  uint4 xr[G];
#pragma unroll
  for (int i = 0; i < G; ++i) xr[i] = load_raw(xb + static_cast<size_t>(i) * d, own && i < nt);

  for (int c0 = 0; c0 < nt; c0 += CH) {
    const int nc = min(CH, nt - c0);  // uniform over the block
    for (int i0 = 0; i0 < nc; i0 += G) {
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const int i = i0 + j;  // token c0 + i of the block
        if (i < nc) {
          float a[EP];
#pragma unroll
          for (int e = 0; e < EP; ++e) a[e] = 0.f;
          if constexpr (kCached) {
            dot_chunk<Tin, EP>(xr[j], w, a);
          } else {
            if (own) dot_chunk_streamed<Tin, EP>(xr[j], Wg, tid * NV, E, a);
          }
          // d wider than one slice per thread: further slices with W_g rows from L1
          for (int c = tid + kRouteThreads; c < nchunks; c += kRouteThreads)
            dot_chunk_streamed<Tin, EP>(load_raw(x + static_cast<size_t>(t0 + c0 + i) * d + c * NV, true), Wg,
                                        c * NV, E, a);
          int e;
          const float v = warp_reduce_scatter<EP>(a, lane, e);
          if ((lane & (32 / EP - 1)) == 0) s_red[i][warp][e] = v;
        }
        // the slice kRouteGroup tokens ahead (across chunk ends)
        const int nxt = c0 + i + G;
        xr[j] = load_raw(xb + static_cast<size_t>(nxt) * d, own && nxt < nt);
      }
    }
    __syncthreads();
    if (tid < nc * EP) {
      const int i = tid / EP, e = tid % EP;
      float sum = 0.f;
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) sum += s_red[i][ww][e];
      s_log[i][e] = sum;
    }
    __syncthreads();
    if (tid < nc) select_and_store<EP>(s_log[tid], t0 + c0 + tid, E, K, flags, idx, gate, s_cnt, status);
  }
  __syncthreads();
  if (tid < E) blockcounts[blockIdx.x * E + tid] = s_cnt[tid];
  stamp_end(stamps, ST_ROUTE);
}

template <typename Tin, int EP>
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_kernel(const Tin *__restrict__ x, const Tin *__restrict__ Wg, int T, int d, int E, int K, int tpb,
                 unsigned flags, int32_t *__restrict__ idx, float *__restrict__ gate,
                 int32_t *__restrict__ blockcounts, int *status, unsigned long long *stamps) {
  route_body<Tin, EP>(x, Wg, T, d, E, K, tpb, flags, idx, gate, blockcounts, status, stamps);
}

// Stable grouping.  Block b (of nb) ranks the (token, slot) entries of tokens
// [b*kGroupTokens, (b+1)*kGroupTokens) in flat t*K + k order: rank = entries of
// that expert in earlier router blocks + in earlier warps of this block + in
// earlier lanes of this warp.  Each expert's segment in the padded grouped
// buffers (X_perm, H) starts at a multiple of kSegPad; pad rows get token -1
// and gate 0.  pos[t, k] is the entry's row in the unpadded grouped order
// (offsets[e] + rank), which indexes the compact expert-output buffer.  The
// router's outputs are read through L2 (ld.cg): in the fused router the block
// that runs this has not written most of them itself.
__device__ __forceinline__ void group_body(int b, int nb, int T, int E, int K, int nb_route, int tpb,
                                           const int32_t *__restrict__ idx, const float *__restrict__ gate,
                                           const int32_t *__restrict__ blockcounts, int32_t *offsets,
                                           int32_t *poffsets, int32_t *pos, int32_t *perm_tok, float *perm_gate,
                                           int *status) {
  constexpr int NT = kGroupTokens * kMaxK;
  constexpr int NW = NT / 32;
  __shared__ int s_base[kMaxE], s_tot[kMaxE], s_off[kMaxE + 1], s_poff[kMaxE + 1];
  __shared__ int s_wcnt[NW][kMaxE];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid < kMaxE) { s_base[tid] = 0; s_tot[tid] = 0; }
  for (int i = tid; i < NW * kMaxE; i += NT) (&s_wcnt[0][0])[i] = 0;
  __syncthreads();
  // entries ahead of this chunk: whole router blocks from their histograms,
  // plus the part of the router block it starts in, counted from idx
  const int tok0 = b * kGroupTokens;
  const int rb_full = tok0 / tpb;
  for (int i = tid; i < nb_route * E; i += NT) {
    const int rb = i / E, e = i - rb * E;
    const int c = __ldcg(blockcounts + i);
    atomicAdd(&s_tot[e], c);
    if (rb < rb_full) atomicAdd(&s_base[e], c);
  }
  for (int i = rb_full * tpb * K + tid; i < tok0 * K; i += NT) {
    const int e = __ldcg(idx + i);
    if (e >= 0 && e < E) atomicAdd(&s_base[e], 1);
  }
  __syncthreads();
  if (tid == 0) {
    int off = 0, poff = 0;
    for (int e = 0; e < E; ++e) {
      s_off[e] = off;
      s_poff[e] = poff;
      off += s_tot[e];
      poff += (s_tot[e] + kSegPad - 1) / kSegPad * kSegPad;
    }
    s_off[E] = off;
    s_poff[E] = poff;
  }
  __syncthreads();
  if (b == 0 && tid <= E) { offsets[tid] = s_off[tid]; poffsets[tid] = s_poff[tid]; }

  const int flat0 = b * kGroupTokens * K;
  const int n_entries = min(kGroupTokens, T - b * kGroupTokens) * K;
  bool active = tid < n_entries;
  int e = active ? __ldcg(idx + flat0 + tid) : -1;
  if (active && (e < 0 || e >= E)) {
    set_status(status, MOE_ERR_DEVICE_BOUNDS);
    active = false;
    e = -1;
  }
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (active && rank_w == 0) s_wcnt[warp][e] = __popc(peers);
  __syncthreads();
  if (active) {
    int r = s_base[e] + rank_w;
    for (int w = 0; w < warp; ++w) r += s_wcnt[w][e];
    const int rp = s_poff[e] + r;
    perm_tok[rp] = (flat0 + tid) / K;
    perm_gate[rp] = __ldcg(gate + flat0 + tid);
    pos[flat0 + tid] = s_off[e] + r;  // unpadded grouped row
  }
  for (int ee = b; ee < E; ee += nb) {
    const int start = s_poff[ee] + s_tot[ee], end = s_poff[ee + 1];
    for (int r = start + tid; r < end; r += NT) {
      perm_tok[r] = -1;
      perm_gate[r] = 0.f;
    }
  }
}

// Grouping of at most 32 (token, slot) entries (T * K <= 32) by the block
// that has just routed them: one warp ranks the entries with
// __match_any_sync in flat t*K + k order within each expert -- the order of
// group_body, so the permutation is the same -- reading idx and gate back
// from this block's own stores; then the block marks the padding rows.
__device__ __forceinline__ void group_tiny(int T, int E, int K, const int32_t *idx, const float *gate,
                                           int32_t *offsets, int32_t *poffsets, int32_t *pos, int32_t *perm_tok,
                                           float *perm_gate, int *status) {
  __shared__ int s_cnt[kMaxE], s_off[kMaxE + 1], s_poff[kMaxE + 1];
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = T * K;
  for (int i = tid; i < E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  if (tid < 32) {
    bool active = lane < n;
    int e = active ? idx[lane] : -1;
    if (active && (e < 0 || e >= E)) {
      set_status(status, MOE_ERR_DEVICE_BOUNDS);
      active = false;
      e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (active && rank == 0) s_cnt[e] = __popc(peers);
    __syncwarp();
    if (lane == 0) {
      int off = 0, poff = 0;
      for (int ee = 0; ee < E; ++ee) {
        s_off[ee] = off;
        s_poff[ee] = poff;
        off += s_cnt[ee];
        poff += (s_cnt[ee] + kSegPad - 1) / kSegPad * kSegPad;
      }
      s_off[E] = off;
      s_poff[E] = poff;
    }
    __syncwarp();
    for (int i = lane; i <= E; i += 32) {
      offsets[i] = s_off[i];
      poffsets[i] = s_poff[i];
    }
    if (active) {
      const int rp = s_poff[e] + rank;
      perm_tok[rp] = lane / K;
      perm_gate[rp] = gate[lane];
      pos[lane] = s_off[e] + rank;  // unpadded grouped row
    }
  }
  __syncthreads();
  for (int ee = 0; ee < E; ++ee)
    for (int r = s_poff[ee] + s_cnt[ee] + tid; r < s_poff[ee + 1]; r += blockDim.x) {
      perm_tok[r] = -1;
      perm_gate[r] = 0.f;
    }
}

__global__ void __launch_bounds__(kGroupTokens *kMaxK)
    group_kernel(int T, int E, int K, int nb_route, int tpb, unsigned flags, const int32_t *__restrict__ idx,
                 const float *__restrict__ gate, const int32_t *__restrict__ blockcounts, int32_t *offsets,
                 int32_t *poffsets, int32_t *pos, int32_t *perm_tok, float *perm_gate, int *status,
                 unsigned long long *stamps) {
  pdl_wait();
  pdl_trigger();
  stamp_begin(stamps, ST_GROUP);
  group_body(blockIdx.x, gridDim.x, T, E, K, nb_route, tpb, idx, gate, blockcounts, offsets, poffsets, pos,
             perm_tok, perm_gate, status);
  (void)flags;
  stamp_end(stamps, ST_GROUP);
}

// Router and grouping in one launch, for batches that one grouping block
// covers (T <= kGroupTokens): every block routes its tokens as route_kernel
// does (same arithmetic, same results), then the block that finishes last --
// the one whose arrival on the ticket counter (zero at launch) completes the
// count -- groups all the tokens.
template <typename Tin, int EP>
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_group_kernel(const Tin *__restrict__ x, const Tin *__restrict__ Wg, int T, int d, int E, int K, int tpb,
                       unsigned flags, int32_t *idx, float *gate, int32_t *blockcounts, int32_t *offsets,
                       int32_t *poffsets, int32_t *pos, int32_t *perm_tok, float *perm_gate, int *status,
                       int *ticket, unsigned long long *stamps) {
  route_body<Tin, EP>(x, Wg, T, d, E, K, tpb, flags, idx, gate, blockcounts, status, stamps);
  __shared__ int s_last;
  __syncthreads();  // this block's routing stores precede its arrival
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // the other blocks' routing stores are visible to this one
  stamp_begin(stamps, ST_GROUP);
  group_body(0, 1, T, E, K, gridDim.x, tpb, idx, gate, blockcounts, offsets, poffsets, pos, perm_tok, perm_gate,
             status);
  stamp_end(stamps, ST_GROUP);
}

// Router and grouping of a small batch (T <= kSingleRouteT) in one block,
// launched with programmatic dependent launch: the block first waits for the
// previous work in the stream to finish, then clears the call's status words
// and split / slot counters (n_zero ints from `status`, which that work may
// have been using), then routes every token as route_kernel does (same
// arithmetic) and groups them in one warp (group_tiny).
template <typename Tin, int EP>
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_single_kernel(const Tin *__restrict__ x, const Tin *__restrict__ Wg, int T, int d, int E, int K, int tpb,
                        unsigned flags, int32_t *idx, float *gate, int32_t *blockcounts, int32_t *offsets,
                        int32_t *poffsets, int32_t *pos, int32_t *perm_tok, float *perm_gate, int *status, int n_zero,
                        unsigned long long *stamps) {
  pdl_wait();
  for (int i = threadIdx.x; i < n_zero; i += blockDim.x) status[i] = 0;
  __syncthreads();
  route_body<Tin, EP>(x, Wg, T, d, E, K, tpb, flags, idx, gate, blockcounts, status, stamps);
  __syncthreads();
  __threadfence_block();
  stamp_begin(stamps, ST_GROUP);
  static_assert(kSingleRouteT * kMaxK <= 32, "group_tiny ranks all entries in one warp");
  group_tiny(T, E, K, idx, gate, offsets, poffsets, pos, perm_tok, perm_gate, status);
  stamp_end(stamps, ST_GROUP);
}

// X_perm[r, :] = x[perm_tok[r], :] for every grouped row; pad rows are zeroed
// when zero_pads (the training forward: the weight gradients contract over
// whole segments) and left as they are otherwise (every product row depends
// on its own input row only, and the rows of padding are never stored to the
// layer's output).  One warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_kernel(const uint4 *__restrict__ x, int T, int vec_per_row,
                                                     const int32_t *__restrict__ perm_tok,
                                                     const int32_t *__restrict__ poffsets, int E,
                                                     uint4 *__restrict__ xperm, int zero_pads, int *status,
                                                     unsigned long long *stamps) {
  pdl_wait();
  pdl_trigger();
  stamp_begin(stamps, ST_GATHER);
  const int rows = poffsets[E];
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int r = gw; r < rows; r += nw) {
    int tok = perm_tok[r];
    if (tok >= T) {
      set_status(status, MOE_ERR_DEVICE_BOUNDS);
      tok = -1;
    }
    uint4 *dst = xperm + static_cast<size_t>(r) * vec_per_row;
    if (tok >= 0) {
      // eight 16-byte loads per lane in flight (a 4096-wide bf16 row is 16 per lane)
      const uint4 *src = x + static_cast<size_t>(tok) * vec_per_row;
      int v = lane;
      for (; v + 224 < vec_per_row; v += 256) {
        uint4 a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = __ldg(src + v + 32 * i);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[v + 32 * i] = a[i];
      }
      for (; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
    } else if (zero_pads) {
      for (int v = lane; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    }
  }
  stamp_end(stamps, ST_GATHER);
}

__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&a);
  u.y = *reinterpret_cast<uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p) = u;
}
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
  uint2 u = *reinterpret_cast<const uint2 *>(p);
  float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&u.x));
  float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// y[t] = sum_k (sum_s O[s][pos[t,k]]): slot 0 then slot 1, splits in order,
// with O the compact [splits, T*K, d] output of the down projection (pos is an
// unpadded grouped row).  The gate was applied by the down projection's
// epilogue.  No atomics.
template <typename Tout>
__global__ void __launch_bounds__(256) combine_kernel(Tout *__restrict__ y, int T, int d, int K, int S,
                                                      long long split_stride, const float *__restrict__ obuf,
                                                      const int32_t *__restrict__ pos, int rows_bound,
                                                      unsigned flags, int *status, unsigned long long *stamps) {
  pdl_wait();
  pdl_trigger();
  stamp_begin(stamps, ST_COMBINE);
  const int q = d >> 2;
  const long long total = static_cast<long long>(T) * q;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / q);
    const int c = static_cast<int>(i - static_cast<long long>(t) * q) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; ++k) {
      int r = pos[t * K + k];
      if (r < 0 || r >= rows_bound) {
        set_status(status, MOE_ERR_DEVICE_BOUNDS);
        continue;
      }
      const float *src = obuf + static_cast<size_t>(r) * d + c;
      float4 sk = __ldg(reinterpret_cast<const float4 *>(src));
      for (int s = 1; s < S; ++s) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(src + s * split_stride));
        sk.x += v.x; sk.y += v.y; sk.z += v.z; sk.w += v.w;
      }
      if (k == 0) {
        acc = sk;
      } else {
        acc.x += sk.x; acc.y += sk.y; acc.z += sk.z; acc.w += sk.w;
      }
    }
    Tout *dst = y + static_cast<size_t>(t) * d + c;
    if (flags & MOE_ACCUMULATE) {
      float4 old = load4(dst);
      acc.x = old.x + acc.x; acc.y = old.y + acc.y; acc.z = old.z + acc.z; acc.w = old.w + acc.w;
    }
    store4(dst, acc);
  }
  stamp_end(stamps, ST_COMBINE);
}

// Unpadded copies of the routing results for moe_route.
__global__ void route_export_kernel(int T, int E, int K, const int32_t *__restrict__ idx_ws,
                                    const float *__restrict__ gate_ws, const int32_t *__restrict__ pos_ws,
                                    const int32_t *__restrict__ offsets_ws, const int32_t *__restrict__ poffsets_ws,
                                    int32_t *idx, float *gate, int32_t *perm_tok, int32_t *offsets, int32_t *pos) {
  pdl_wait();
  pdl_trigger();
  const int n = T * K;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int e = idx_ws[i];
    const int ru = pos_ws[i];
    idx[i] = e;
    gate[i] = gate_ws[i];
    perm_tok[ru] = i / K;
    if (pos) pos[i] = ru;
  }
  if (blockIdx.x == 0 && threadIdx.x <= E) offsets[threadIdx.x] = offsets_ws[threadIdx.x];
}

// out = x / sqrt(mean(x^2) + eps) per row; one block per row, fp32 sums.
// The general form: any d, any alignment (element loads).
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const T *__restrict__ x, T *__restrict__ out, int d, float eps,
                                                      unsigned long long *stamps) {
  __shared__ float s_red[8];
  pdl_wait();
  pdl_trigger();
  stamp_begin(stamps, ST_NORM);
  const T *row = x + static_cast<size_t>(blockIdx.x) * d;
  T *orow = out + static_cast<size_t>(blockIdx.x) * d;
  float ss = 0.f;
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    const float v = to_f(row[j]);
    ss = fmaf(v, v, ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += s_red[w];
  const float inv = 1.0f / sqrtf(tot / static_cast<float>(d) + eps);
  __syncthreads();  // every thread has read s_red before any write below (in-place safe)
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    const float v = to_f(row[j]) * inv;
    if constexpr (sizeof(T) == 2) orow[j] = __float2bfloat16_rn(v);
    else orow[j] = v;
  }
  stamp_end(stamps, ST_NORM);
}

// Sum of squares of one 16-byte chunk (8 bf16 or 4 fp32 values), in order.
template <typename T>
__device__ __forceinline__ float chunk_sumsq(uint4 u, float ss) {
  if constexpr (sizeof(T) == 2) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      ss = fmaf(f.x, f.x, ss);
      ss = fmaf(f.y, f.y, ss);
    }
  } else {
    const float f[4] = {__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) ss = fmaf(f[i], f[i], ss);
  }
  return ss;
}

template <typename T>
__device__ __forceinline__ uint4 chunk_scale(uint4 u, float inv) {
  if constexpr (sizeof(T) == 2) {
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      h[i] = __floats2bfloat162_rn(f.x * inv, f.y * inv);
    }
    return u;
  } else {
    return make_uint4(__float_as_uint(__uint_as_float(u.x) * inv), __float_as_uint(__uint_as_float(u.y) * inv),
                      __float_as_uint(__uint_as_float(u.z) * inv), __float_as_uint(__uint_as_float(u.w) * inv));
  }
}

// The same for rows of whole 16-byte chunks at 16-byte aligned addresses:
// 16-byte loads and stores, and each thread keeps its first kNormRegChunks
// chunks in registers between the sum and the scaling, so a row of up to
// 256 * kNormRegChunks chunks (8192 bf16 values) is read from memory once.
constexpr int kNormRegChunks = 4;
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_vec_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ out,
                                                          int nch, int d, float eps, unsigned long long *stamps) {
  __shared__ float s_red[8];
  pdl_wait();
  pdl_trigger();
  stamp_begin(stamps, ST_NORM);
  const uint4 *row = x + static_cast<size_t>(blockIdx.x) * nch;
  uint4 *orow = out + static_cast<size_t>(blockIdx.x) * nch;
  uint4 v[kNormRegChunks];
#pragma unroll
  for (int i = 0; i < kNormRegChunks; ++i) {
    const int c = threadIdx.x + i * 256;
    v[i] = c < nch ? row[c] : make_uint4(0u, 0u, 0u, 0u);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormRegChunks; ++i) ss = chunk_sumsq<T>(v[i], ss);
  for (int c = threadIdx.x + kNormRegChunks * 256; c < nch; c += 256) ss = chunk_sumsq<T>(row[c], ss);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += s_red[w];
  const float inv = 1.0f / sqrtf(tot / static_cast<float>(d) + eps);
  // each thread writes back only the chunks it read, so out may equal x
#pragma unroll
  for (int i = 0; i < kNormRegChunks; ++i) {
    const int c = threadIdx.x + i * 256;
    if (c < nch) orow[c] = chunk_scale<T>(v[i], inv);
  }
  for (int c = threadIdx.x + kNormRegChunks * 256; c < nch; c += 256) orow[c] = chunk_scale<T>(row[c], inv);
  stamp_end(stamps, ST_NORM);
}

}  // namespace

cudaError_t launch_route(const void *x, const void *Wg, int T, int d, int E, int K, int dtype, unsigned flags,
                         const WsLayout &L, const Ptrs &P, cudaStream_t s) {
  // First kernel of a forward pass: an ordinary launch, ordered after all
  // earlier work in the stream.
  const dim3 grid(L.n_route_blocks), block(kRouteThreads);
  const int tpb = L.route_tpb;
  if (dtype == MOE_BF16) {
    auto *xx = static_cast<const __nv_bfloat16 *>(x);
    auto *ww = static_cast<const __nv_bfloat16 *>(Wg);
    if (E <= 8)
      return launch_kernel(route_kernel<__nv_bfloat16, 8>, grid, block, 0, s, false, xx, ww, T, d, E, K, tpb, flags,
                           P.idx, P.gate, P.blockcounts, P.status, P.stamps);
    return launch_kernel(route_kernel<__nv_bfloat16, 32>, grid, block, 0, s, false, xx, ww, T, d, E, K, tpb, flags,
                         P.idx, P.gate, P.blockcounts, P.status, P.stamps);
  }
  auto *xx = static_cast<const float *>(x);
  auto *ww = static_cast<const float *>(Wg);
  if (E <= 8)
    return launch_kernel(route_kernel<float, 8>, grid, block, 0, s, false, xx, ww, T, d, E, K, tpb, flags, P.idx,
                         P.gate, P.blockcounts, P.status, P.stamps);
  return launch_kernel(route_kernel<float, 32>, grid, block, 0, s, false, xx, ww, T, d, E, K, tpb, flags, P.idx,
                       P.gate, P.blockcounts, P.status, P.stamps);
}

cudaError_t launch_route_group(const void *x, const void *Wg, int T, int d, int E, int K, int dtype, unsigned flags,
                               const WsLayout &L, const Ptrs &P, cudaStream_t s) {
  if (L.route_single) {
    const int n_zero = static_cast<int>(L.zero_bytes / sizeof(int));
    const int tpb = L.route_tpb;
    if (dtype == MOE_BF16) {
      auto *xx = static_cast<const __nv_bfloat16 *>(x);
      auto *ww = static_cast<const __nv_bfloat16 *>(Wg);
      auto kern = E <= 8 ? route_single_kernel<__nv_bfloat16, 8> : route_single_kernel<__nv_bfloat16, 32>;
      return launch_kernel(kern, dim3(1), dim3(kRouteThreads), 0, s, true, xx, ww, T, d, E, K, tpb, flags, P.idx,
                           P.gate, P.blockcounts, P.offsets, P.poffsets, P.pos, P.perm_tok, P.perm_gate, P.status,
                           n_zero, P.stamps);
    }
    auto *xx = static_cast<const float *>(x);
    auto *ww = static_cast<const float *>(Wg);
    auto kern = E <= 8 ? route_single_kernel<float, 8> : route_single_kernel<float, 32>;
    return launch_kernel(kern, dim3(1), dim3(kRouteThreads), 0, s, true, xx, ww, T, d, E, K, tpb, flags, P.idx, P.gate,
                         P.blockcounts, P.offsets, P.poffsets, P.pos, P.perm_tok, P.perm_gate, P.status, n_zero,
                         P.stamps);
  }
  if (T > kGroupTokens) {
    const cudaError_t err = launch_route(x, Wg, T, d, E, K, dtype, flags, L, P, s);
    return err == cudaSuccess ? launch_group(T, E, K, L, flags, P, s) : err;
  }
  // one launch: the router blocks, then the grouping in the block that finishes last
  const dim3 grid(L.n_route_blocks), block(kRouteThreads);
  static_assert(kRouteThreads == kGroupTokens * kMaxK, "the fused kernel's blocks run both bodies");
  const int tpb = L.route_tpb;
  int *ticket = P.status + 1;  // zero at launch, like the rest of the status words
  if (dtype == MOE_BF16) {
    auto *xx = static_cast<const __nv_bfloat16 *>(x);
    auto *ww = static_cast<const __nv_bfloat16 *>(Wg);
    auto kern = E <= 8 ? route_group_kernel<__nv_bfloat16, 8> : route_group_kernel<__nv_bfloat16, 32>;
    return launch_kernel(kern, grid, block, 0, s, false, xx, ww, T, d, E, K, tpb, flags, P.idx, P.gate,
                         P.blockcounts, P.offsets, P.poffsets, P.pos, P.perm_tok, P.perm_gate, P.status, ticket,
                         P.stamps);
  }
  auto *xx = static_cast<const float *>(x);
  auto *ww = static_cast<const float *>(Wg);
  auto kern = E <= 8 ? route_group_kernel<float, 8> : route_group_kernel<float, 32>;
  return launch_kernel(kern, grid, block, 0, s, false, xx, ww, T, d, E, K, tpb, flags, P.idx, P.gate, P.blockcounts,
                       P.offsets, P.poffsets, P.pos, P.perm_tok, P.perm_gate, P.status, ticket, P.stamps);
}

cudaError_t launch_group(int T, int E, int K, const WsLayout &L, unsigned flags, const Ptrs &P, cudaStream_t s) {
  const dim3 grid((T + kGroupTokens - 1) / kGroupTokens), block(kGroupTokens * kMaxK);
  return launch_kernel(group_kernel, grid, block, 0, s, true, T, E, K, L.n_route_blocks, L.route_tpb, flags, P.idx,
                       P.gate, P.blockcounts, P.offsets, P.poffsets, P.pos, P.perm_tok, P.perm_gate, P.status,
                       P.stamps);
}

cudaError_t launch_gather(const void *x, int T, int d, int E, int dtype, int R, const Ptrs &P, int num_sms,
                          cudaStream_t s, bool zero_pads) {
  const int elem = dtype == MOE_BF16 ? 2 : 4;
  const int vec_per_row = d * elem / 16;
  int blocks = (R + 7) / 8;  // 8 warps (rows) per block
  if (blocks > num_sms * 8) blocks = num_sms * 8;
  if (blocks < 1) blocks = 1;
  return launch_kernel(gather_kernel, dim3(blocks), dim3(256), 0, s, true, static_cast<const uint4 *>(x), T,
                       vec_per_row, static_cast<const int32_t *>(P.perm_tok), static_cast<const int32_t *>(P.poffsets),
                       E, static_cast<uint4 *>(P.xperm), zero_pads ? 1 : 0, P.status, P.stamps);
}

cudaError_t launch_combine(void *y, int T, int d, int K, int S, int dtype, unsigned flags, const Ptrs &P,
                           int num_sms, cudaStream_t s) {
  const long long total = static_cast<long long>(T) * (d / 4);
  long long blocks = (total + 255) / 256;
  if (blocks > num_sms * 16LL) blocks = num_sms * 16LL;
  if (blocks < 1) blocks = 1;
  const long long split_stride = static_cast<long long>(T) * K * d;  // compact [S, T*K, d]
  const dim3 grid(static_cast<unsigned>(blocks)), block(256);
  if (dtype == MOE_BF16)
    return launch_kernel(combine_kernel<__nv_bfloat16>, grid, block, 0, s, true, static_cast<__nv_bfloat16 *>(y), T,
                         d, K, S, split_stride, static_cast<const float *>(P.obuf), static_cast<const int32_t *>(P.pos),
                         T * K, flags, P.status, P.stamps);
  return launch_kernel(combine_kernel<float>, grid, block, 0, s, true, static_cast<float *>(y), T, d, K, S,
                       split_stride, static_cast<const float *>(P.obuf), static_cast<const int32_t *>(P.pos), T * K,
                       flags, P.status, P.stamps);
}

cudaError_t launch_route_export(int T, int E, int K, const Ptrs &P, int32_t *idx, float *gate, int32_t *perm_tok,
                                int32_t *offsets, int32_t *pos, cudaStream_t s) {
  int blocks = (T * K + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 1024) blocks = 1024;
  return launch_kernel(route_export_kernel, dim3(blocks), dim3(256), 0, s, true, T, E, K,
                       static_cast<const int32_t *>(P.idx), static_cast<const float *>(P.gate),
                       static_cast<const int32_t *>(P.pos), static_cast<const int32_t *>(P.offsets),
                       static_cast<const int32_t *>(P.poffsets), idx, gate, perm_tok, offsets, pos);
}

cudaError_t launch_rmsnorm(const void *x, void *out, int T, int d, float eps, int dtype, cudaStream_t s,
                           unsigned long long *stamps) {
  if (T == 0) return cudaSuccess;
  // Launched with programmatic dependent launch: each block waits for the
  // previous kernel in the stream before it reads x.
  const size_t eb = dtype == MOE_BF16 ? 2 : 4;
  const bool vec = (d * eb) % 16 == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  const int nch = static_cast<int>(d * eb / 16);
  if (vec && dtype == MOE_BF16)
    return launch_kernel(rmsnorm_vec_kernel<__nv_bfloat16>, dim3(T), dim3(256), 0, s, true,
                         static_cast<const uint4 *>(x), static_cast<uint4 *>(out), nch, d, eps, stamps);
  if (vec)
    return launch_kernel(rmsnorm_vec_kernel<float>, dim3(T), dim3(256), 0, s, true, static_cast<const uint4 *>(x),
                         static_cast<uint4 *>(out), nch, d, eps, stamps);
  if (dtype == MOE_BF16)
    return launch_kernel(rmsnorm_kernel<__nv_bfloat16>, dim3(T), dim3(256), 0, s, true,
                         static_cast<const __nv_bfloat16 *>(x), static_cast<__nv_bfloat16 *>(out), d, eps, stamps);
  return launch_kernel(rmsnorm_kernel<float>, dim3(T), dim3(256), 0, s, true, static_cast<const float *>(x),
                       static_cast<float *>(out), d, eps, stamps);
}

}  // namespace moe
