// gemm_bwd.cu -- the grouped GEMMs of the MoE layer's backward pass on
// 5th-generation tensor cores (bf16 operands, fp32 accumulators in TMEM,
// operands staged by TMA).
//
// For expert e with grouped rows X_e (its padded segment of X_perm), saved
// pre-activations a = X_e W1[e], b = X_e W3[e], H_e = SiLU(a) (.) b and
// dY_e = gate (.) dy on the same rows (built by the prep kernel), the chain
// rule through "Expert Network Structure (SwiGLU)" and the gate-weighted sum
// of section 3.4 "MoE Layer Formulation" (Mixtral of Experts summary pages)
// gives four grouped products:
//   dgrad H    dH = dY_e W2[e]^T; epilogue da = dH (.) b (.) SiLU'(a),
//              db = dH (.) SiLU(a)                    -> dAB [R, 2f] bf16
//   dgrad X    dX_e = [da | db] [W1[e] | W3[e]]^T      -> fp32 [T*K, d], unpadded rows
//   wgrad W2   dW2[e] = H_e^T dY_e                     -> fp32 [E, f, d]
//   wgrad W13  [dW1[e] | dW3[e]] = X_e^T [da | db]     -> fp32 [E, d, f] twice
//
// One persistent kernel per product: one CTA of 192 threads per SM, 128 x 256
// output tiles, cta_group::1 MMAs (M128 N256 K16), a 4-stage ring of 48 KiB
// and two 256-column TMEM accumulators, so the epilogue of one tile overlaps
// the MMAs of the next.  Roles: warp 0 TMA producer, warp 1 TMEM allocator +
// MMA issuer, warps 2..5 epilogue (one 32-lane TMEM quarter each).
// Shared-memory operand layouts (128-byte swizzle throughout):
//   dgrad  A K-major: one 128-row x 64-column box of the grouped activations;
//          B K-major: 256 weight rows x 64 contraction elements in one box of
//          the bank's [E, N, K] view (W2 [E, f, d] for dH; W1, W3 [E, d, f]
//          for dX, whose contraction runs over W1's f/64 k-blocks, then W3's);
//   wgrad  the contraction runs over grouped rows, so both operands are
//          MN-major row panels: 64-column x 64-row boxes, two for A's 128
//          columns and four for B's 256, 8 KiB apart.
// Weight-gradient tiles cover every expert; the tiles of an expert with no
// rows write zeros (or leave the output alone when accumulating).  Padding
// rows of X_perm, H, dY and dAB are zeros, so whole segments are contracted.
//
// Every mbarrier wait is bounded (about one second); on expiry the CTA records
// MOE_ERR_DEVICE_TIMEOUT, stops issuing work, waits (bounded) for its own
// copies and MMAs in flight, frees TMEM and returns.  MOE_DEBUG_FORCE_TIMEOUT
// makes the dH product's MMA thread first wait on a barrier that nothing
// signals, which runs that path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;   // 16 KiB
constexpr int B_BYTES = BN * BK * 2;   // 32 KiB
constexpr int BOX_BYTES = 64 * 64 * 2; // one MN-major 64 x 64 box
constexpr int STAGES = 4;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
// Epilogue staging: one 32 x 33 fp32 tile per epilogue warp (the odd row
// pitch keeps both the row-per-lane and the segment-per-lane accesses free of
// bank conflicts).
constexpr int STAGE_PITCH = 33;
constexpr int EPI_WARP_BYTES = 32 * STAGE_PITCH * 4;
constexpr int SMEM = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + 1024 /*Ctrl*/ + 4 * EPI_WARP_BYTES;
static_assert(SMEM <= 232448, "shared memory budget");
constexpr int ACC_COLS = BN;
constexpr int TMEM_COLS = 2 * ACC_COLS;
constexpr int NUM_THREADS = 192;

enum { KIND_DGRAD_H = 0, KIND_DGRAD_X = 1, KIND_WGRAD_W2 = 2, KIND_WGRAD_W13 = 3 };

struct BwdArgs {
  const int32_t *poffsets;  // [E+1] padded segment starts
  const int32_t *offsets;   // [E+1] unpadded segment starts
  int E;
  int rows_bound;           // R: rows of the padded grouped buffers
  int f;
  int m_total;              // weight gradients: rows of one expert's gradient (f or d)
  int n_out;                // output columns: f (dH), d (dX, dW2), 2f (dW1 | dW3)
  int num_n_tiles;
  int num_kb;               // dgrad: 64-deep k-blocks of the contraction
  int kb_bank;              // dX: k-blocks per weight bank (f / 64)
  const __nv_bfloat16 *ab;  // dH: saved pre-activations [R, 2f]
  __nv_bfloat16 *dab;       // dH: output dL/da | dL/db [R, 2f]
  float *out0;              // dX [T*K, d]; dW2 [E, f, d]; dW1 [E, d, f]
  float *out1;              // dW3 [E, d, f]
  int accumulate;           // weight gradients: add to out0 / out1
  int force_timeout;        // failure-path test: wait on a barrier nothing signals first
  int *status;
};

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t stall;  // never signalled (failure-path test)
  uint32_t tmem_base;
  int abort;
  int total_units;
  int ustart[kMaxE + 1];
  int mtiles[kMaxE];
  int poff[kMaxE + 1];
  int uoff[kMaxE + 1];
};
static_assert(sizeof(Ctrl) <= 1024, "control block too large");

struct BTile {
  int e, mt, nt;
  int krow0;  // weight gradients: first grouped row of the contraction
  int nkb;    // k-blocks of this tile
};

template <int KIND>
__device__ __forceinline__ BTile decode_tile(int u, const Ctrl &c, const BwdArgs &a) {
  BTile t;
  int e = 0;
  while (u >= c.ustart[e + 1]) ++e;
  const int r = u - c.ustart[e];
  t.e = e;
  if (KIND == KIND_DGRAD_H || KIND == KIND_DGRAD_X) {
    // m-tiles fastest: CTAs running together share the weight panel
    const int mt_e = c.mtiles[e];
    t.nt = r / mt_e;
    t.mt = r - t.nt * mt_e;
    t.krow0 = 0;
    t.nkb = a.num_kb;
  } else {
    const int MT = (a.m_total + BM - 1) / BM;
    t.nt = r / MT;
    t.mt = r - t.nt * MT;
    t.krow0 = c.poff[e];
    t.nkb = (c.poff[e + 1] - c.poff[e]) / BK;
  }
  return t;
}

// Logistic function with the fast reciprocal division (a few fp32 ulps; its
// results are rounded to bf16).
__device__ __forceinline__ float sigmoid_f(float v) { return __fdividef(1.0f, 1.0f + __expf(-v)); }

// The epilogue holds a 32 x 32 block as one row per lane (what tcgen05.ld
// 32x32b returns); global memory wants each instruction to cover whole row
// segments.  These helpers move the block through the warp's staging tile.
//
// Rows r < rows_valid of the block to fp32 rows at dst + r * ld (32 floats
// each): every instruction writes four 128-byte row segments.  With
// accumulate the old values are added.
__device__ __forceinline__ void store_block_f32(float *st, const uint32_t (&v)[32], float *dst, size_t ld,
                                                int rows_valid, bool accumulate, int lane) {
#pragma unroll
  for (int c = 0; c < 32; ++c) st[lane * STAGE_PITCH + c] = __uint_as_float(v[c]);
  __syncwarp();
  const int cq = 4 * (lane & 7);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int r = 4 * k + (lane >> 3);
    if (r < rows_valid) {
      const float *sr = st + r * STAGE_PITCH + cq;
      float4 val = make_float4(sr[0], sr[1], sr[2], sr[3]);
      float4 *p = reinterpret_cast<float4 *>(dst + r * ld + cq);
      if (accumulate) {
        const float4 o = *p;
        val.x += o.x; val.y += o.y; val.z += o.z; val.w += o.w;
      }
      *p = val;
    }
  }
  __syncwarp();
}

// A bf16 block of 32 rows x 32 columns (src + r * ld) in segment layout:
// lane l holds the 8 columns 8 (l & 3) .. +7 of rows 8 k + (l >> 2), k < 4, so
// every load instruction reads eight 64-byte row segments.
__device__ __forceinline__ void load_segments_bf16(const __nv_bfloat16 *src, size_t ld, uint4 (&w)[4], int lane) {
#pragma unroll
  for (int k = 0; k < 4; ++k) w[k] = *reinterpret_cast<const uint4 *>(src + (8 * k + (lane >> 2)) * ld + 8 * (lane & 3));
}

// bf16 blocks move through the staging tile as 16-byte pieces, rows
// ROW_BYTES apart (80: every 8 lanes of a row-per-lane access hit distinct
// banks).
constexpr int ROW_BYTES = 80;
static_assert(32 * ROW_BYTES <= EPI_WARP_BYTES, "bf16 staging tile");

// The block loaded by load_segments_bf16 as fp32, one row (32 columns) per lane.
__device__ __forceinline__ void segments_to_rows(uint8_t *st, const uint4 (&w)[4], float (&v)[32], int lane) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4 *>(st + (8 * k + (lane >> 2)) * ROW_BYTES + 16 * (lane & 3)) = w[k];
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 r = *reinterpret_cast<const uint4 *>(st + lane * ROW_BYTES + 16 * j);
    const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&rw[i]));
      v[8 * j + 2 * i] = f2.x;
      v[8 * j + 2 * i + 1] = f2.y;
    }
  }
  __syncwarp();
}

// v (one row per lane) to bf16 rows 0..31 at dst + r * ld, rounded to nearest
// even: every store instruction writes eight 64-byte row segments.
__device__ __forceinline__ void store_block_bf16(uint8_t *st, const float (&v)[32], __nv_bfloat16 *dst, size_t ld,
                                                 int lane) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(st + lane * ROW_BYTES + 16 * j) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = 8 * k + (lane >> 2);
    *reinterpret_cast<uint4 *>(dst + r * ld + 8 * (lane & 3)) =
        *reinterpret_cast<const uint4 *>(st + r * ROW_BYTES + 16 * (lane & 3));
  }
  __syncwarp();
}

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const BwdArgs args) {
  constexpr bool WG = KIND == KIND_WGRAD_W2 || KIND == KIND_WGRAD_W13;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = base;
  uint8_t *sB = base + STAGES * A_BYTES;
  Ctrl &c = *reinterpret_cast<Ctrl *>(sB + STAGES * B_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = args.num_n_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&c.full[s], 1);
      ptx::mbar_init(&c.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&c.tfull[a], 1);
      ptx::mbar_init(&c.tempty[a], 4);  // one arrival per epilogue warp
    }
    ptx::mbar_init(&c.drain, 1);
    ptx::mbar_init(&c.stall, 1);
    ptx::fence_barrier_init();
  }
  ptx::grid_dependency_wait();  // the previous kernel's outputs are read below
  ptx::allow_dependent_launch();
  if (threadIdx.x == 0) {
    int acc = 0;
    bool bad = false;
    const int MT = (args.m_total + BM - 1) / BM;
    for (int e = 0; e < args.E; ++e) {
      const int p0 = args.poffsets[e], p1 = args.poffsets[e + 1];
      if (p1 < p0 || (p1 - p0) % BM != 0 || p1 > args.rows_bound) bad = true;
      const int mt = bad ? 0 : (p1 - p0) / BM;
      c.poff[e] = p0;
      c.uoff[e] = args.offsets[e];
      c.mtiles[e] = mt;
      c.ustart[e] = acc;
      acc += WG ? MT * NT : mt * NT;
    }
    c.poff[args.E] = args.poffsets[args.E];
    c.uoff[args.E] = args.offsets[args.E];
    if (bad) {
      atomicCAS(args.status, 0, MOE_ERR_DEVICE_BOUNDS);
      for (int e = 0; e <= args.E; ++e) { c.ustart[e] = 0; c.poff[e] = 0; }
      acc = 0;
    }
    c.ustart[args.E] = acc;
    c.total_units = acc;
    c.abort = 0;
  }
  __syncthreads();
  const int total = c.total_units;
  if (static_cast<int>(blockIdx.x) >= total) return;

  if (warp == 1) {
    ptx::tmem_alloc(&c.tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB0);
    if (KIND == KIND_DGRAD_X) ptx::prefetch_tmap(&tmB1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  uint32_t issued = 0, last_par = 0;
  int p_stage = 0;
  uint32_t p_phase = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_normal();
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
        const BTile t = decode_tile<KIND>(u, c, args);
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!wait_bounded(&c.empty[p_stage], p_phase ^ 1u, c, args.status, true)) { ok = false; break; }
          uint8_t *a_dst = sA + p_stage * A_BYTES;
          uint8_t *b_dst = sB + p_stage * B_BYTES;
          uint64_t *bar = &c.full[p_stage];
          ptx::mbar_arrive_expect_tx(bar, STAGE_BYTES);
          if (!WG) {
            const int row0 = c.poff[t.e] + t.mt * BM;
            ptx::tma_load_2d(a_dst, &tmA, bar, kb * BK, row0, pol);
            if (KIND == KIND_DGRAD_H) {
              ptx::tma_load_3d(b_dst, &tmB0, bar, kb * BK, t.nt * BN, t.e, pol);
            } else {
              const bool second = kb >= args.kb_bank;
              ptx::tma_load_3d(b_dst, second ? &tmB1 : &tmB0, bar, (second ? kb - args.kb_bank : kb) * BK,
                               t.nt * BN, t.e, pol);
            }
          } else {
            const int krow = t.krow0 + kb * BK;
            const int m0 = t.mt * BM, n0 = t.nt * BN;
            // column-block views: the two 64-column blocks of A and the four
            // of B each in one copy
            ptx::tma_load_3d(a_dst, &tmA, bar, 0, krow, m0 / 64, pol);
            ptx::tma_load_3d(b_dst, &tmB0, bar, 0, krow, n0 / 64, pol);
          }
          issued |= 1u << p_stage;
          last_par = (last_par & ~(1u << p_stage)) | (p_phase << p_stage);
          if (++p_stage == STAGES) { p_stage = 0; p_phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, /*A MN-major*/ WG, /*B MN-major*/ WG);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      // failure-path test: this wait expires, raising the CTA's abort flag
      if (args.force_timeout) ok = wait_bounded(&c.stall, 0, c, args.status, true);
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
        const BTile t = decode_tile<KIND>(u, c, args);
        const int acc = local & 1;
        const uint32_t apar = (local >> 1) & 1;
        if (!wait_bounded(&c.tempty[acc], apar ^ 1u, c, args.status, true)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * ACC_COLS;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!wait_bounded(&c.full[stage], phase, c, args.status, true)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(sA + stage * A_BYTES);
          const uint32_t b_addr = ptx::smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            uint64_t ad, bd;
            if (WG) {
              // MN-major: 64-column boxes 8 KiB apart (LBO), 8-row K groups
              // 1024 B apart (SBO); a K step of 16 rows is 2048 B.
              ad = ptx::smem_desc_sw128(a_addr + ks * 2048, BOX_BYTES, 1024);
              bd = ptx::smem_desc_sw128(b_addr + ks * 2048, BOX_BYTES, 1024);
            } else {
              // K-major: 128 B rows, 8-row groups 1024 B apart; a K step of 16
              // elements is 32 B.
              ad = ptx::smem_desc_sw128(a_addr + ks * 32, 16, 1024);
              bd = ptx::smem_desc_sw128(b_addr + ks * 32, 16, 1024);
            }
            ptx::mma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&c.empty[stage]);  // frees the stage once these MMAs have read it
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit(&c.tfull[acc]);  // (a tile with no k-blocks signals at once)
        ++local;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint8_t *stage_bytes = reinterpret_cast<uint8_t *>(&c) + 1024 + q * EPI_WARP_BYTES;  // 16-byte aligned
    float *stage_tile = reinterpret_cast<float *>(stage_bytes);
    int local = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const BTile t = decode_tile<KIND>(u, c, args);
      const int acc = local & 1;
      const uint32_t apar = (local >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = wait_bounded(&c.tfull[acc], apar, c, args.status, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      const int n0 = t.nt * BN;
      if (KIND == KIND_DGRAD_H) {
        // every row of the segment, padding included (its dH is zero, and so
        // are its a and b: the weight gradients read these rows)
        const int row0 = c.poff[t.e] + t.mt * BM + q * 32;  // the warp's first row
        const size_t rstride = 2 * static_cast<size_t>(args.f);
        const __nv_bfloat16 *pa = args.ab + row0 * rstride;
        __nv_bfloat16 *pd = args.dab + row0 * rstride;
        // a and b of the next chunk are in flight while this one is computed
        uint4 wa[4], wb[4];
        if (n0 < args.n_out) {
          load_segments_bf16(pa + n0, rstride, wa, lane);
          load_segments_bf16(pa + args.f + n0, rstride, wb, lane);
        }
#pragma unroll 1
        for (int cc = 0; cc < BN / 32; ++cc) {
          const int col = n0 + cc * 32;
          if (col >= args.n_out) break;  // f is a multiple of 64: a chunk is all in or all out
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tbase + cc * 32, v);
          float a[32], b[32];
          segments_to_rows(stage_bytes, wa, a, lane);
          segments_to_rows(stage_bytes, wb, b, lane);
          if (cc + 1 < BN / 32 && col + 32 < args.n_out) {
            load_segments_bf16(pa + col + 32, rstride, wa, lane);
            load_segments_bf16(pa + args.f + col + 32, rstride, wb, lane);
          }
          ptx::tmem_wait_ld();
          // SiLU(a) = a s, SiLU'(a) = s (1 + a (1 - s)), s = sigmoid(a):
          // da = dH b SiLU'(a) into a, db = dH SiLU(a) into b
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float dh = __uint_as_float(v[j]);
            const float sg = sigmoid_f(a[j]);
            const float da = dh * b[j] * sg * (1.f + a[j] * (1.f - sg));
            b[j] = dh * a[j] * sg;
            a[j] = da;
          }
          store_block_bf16(stage_bytes, a, pd + col, rstride, lane);
          store_block_bf16(stage_bytes, b, pd + args.f + col, rstride, lane);
        }
      } else if (KIND == KIND_DGRAD_X) {
        // real rows (a prefix of the segment) to their unpadded grouped rows;
        // padding rows are dropped
        const int seg0 = t.mt * BM + q * 32;  // the warp's first segment row
        const int rows_valid = min(32, c.uoff[t.e + 1] - c.uoff[t.e] - seg0);
        if (rows_valid > 0) {
          float *dst = args.out0 + static_cast<size_t>(c.uoff[t.e] + seg0) * args.n_out;
#pragma unroll 1
          for (int cc = 0; cc < BN / 32; ++cc) {
            const int col = n0 + cc * 32;
            if (col >= args.n_out) break;
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tbase + cc * 32, v);
            ptx::tmem_wait_ld();
            store_block_f32(stage_tile, v, dst + col, args.n_out, rows_valid, false, lane);
          }
        }
      } else {
        // weight gradient rows m0.. of expert e (fp32, n contiguous)
        const int m0 = t.mt * BM + q * 32;  // the warp's first row
        const int rows_valid = min(32, args.m_total - m0);
        const bool empty = t.nkb == 0;
        if (!(empty && args.accumulate) && rows_valid > 0) {
#pragma unroll 1
          for (int cc = 0; cc < BN / 32; ++cc) {
            const int col = n0 + cc * 32;
            if (col >= args.n_out) break;
            uint32_t v[32];
            if (!empty) {
              ptx::tmem_ld_32x32b_x32(tbase + cc * 32, v);
              ptx::tmem_wait_ld();
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0u;
            }
            float *dst;
            size_t ld;
            if (KIND == KIND_WGRAD_W2) {
              ld = args.n_out;
              dst = args.out0 + (static_cast<size_t>(t.e) * args.m_total + m0) * ld + col;
            } else {
              // columns [0, f) are dW1's, [f, 2f) dW3's (f a multiple of 64)
              const bool w3 = col >= args.f;
              ld = args.f;
              dst = (w3 ? args.out1 : args.out0) + (static_cast<size_t>(t.e) * args.m_total + m0) * ld +
                    (w3 ? col - args.f : col);
            }
            store_block_f32(stage_tile, v, dst, ld, rows_valid, args.accumulate != 0, lane);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&c.tempty[acc]);
      ++local;
    }
  }

  // Producer tail: every stage's last release has arrived, so no commit can
  // still land in this CTA's barriers.
  if (warp == 0 && lane == 0 && !*reinterpret_cast<volatile int *>(&c.abort)) {
    for (int i = 0; i < STAGES; ++i) {
      wait_bounded(&c.empty[p_stage], p_phase ^ 1u, c, args.status, false);
      if (++p_stage == STAGES) { p_stage = 0; p_phase ^= 1u; }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (*reinterpret_cast<volatile int *>(&c.abort)) {
    // some role gave up: wait (bounded) for this CTA's MMAs and copies in flight
    if (warp == 1 && lane == 0) {
      ptx::mma_commit(&c.drain);
      wait_bounded(&c.drain, 0, c, args.status, false);
    }
    if (warp == 0 && lane == 0) {
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) wait_bounded(&c.full[s], (last_par >> s) & 1u, c, args.status, false);
    }
    ptx::tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
template <int KIND>
cudaError_t launch_one(int num_sms, cudaStream_t s, const CUtensorMap &a, const CUtensorMap &b0,
                       const CUtensorMap &b1, const BwdArgs &args) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(bwd_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  return launch_kernel(bwd_gemm_kernel<KIND>, dim3(num_sms), dim3(NUM_THREADS), SMEM, s, true, a, b0, b1, args);
}

}  // namespace

cudaError_t launch_bwd_gemms(const void *W1, const void *W3, const void *W2, void *dW1, void *dW3, void *dW2, int d,
                             int f, int E, bool accumulate, bool force_timeout, const WsLayout &L, const Ptrs &P,
                             int num_sms, cudaStream_t s, void *const *events) {
  // events (optional): recorded after each of the four products
  auto mark = [&](int i) -> cudaError_t {
    return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) : cudaSuccess;
  };
  CUtensorMap tm_dye_k, tm_w2_k, tm_dab_k, tm_w1_k, tm_w3_k, tm_h_mn, tm_dye_mn, tm_x_mn, tm_dab_mn;
  const uint64_t R = static_cast<uint64_t>(L.R);
  if (!tmap_2d(&tm_dye_k, P.dye, d, R, BM) || !tmap_3d(&tm_w2_k, W2, d, f, E, BN) ||
      !tmap_2d(&tm_dab_k, P.dab, 2 * static_cast<uint64_t>(f), R, BM) || !tmap_3d(&tm_w1_k, W1, f, d, E, BN) ||
      !tmap_3d(&tm_w3_k, W3, f, d, E, BN) || !tmap_blocks_2d(&tm_h_mn, P.hbuf, f, R, BM / 64) ||
      !tmap_blocks_2d(&tm_dye_mn, P.dye, d, R, BN / 64) || !tmap_blocks_2d(&tm_x_mn, P.xperm, d, R, BM / 64) ||
      !tmap_blocks_2d(&tm_dab_mn, P.dab, 2 * static_cast<uint64_t>(f), R, BN / 64))
    return cudaErrorInvalidValue;

  BwdArgs a{};
  a.poffsets = P.poffsets;
  a.offsets = P.offsets;
  a.E = E;
  a.rows_bound = L.R;
  a.f = f;
  a.status = P.status;
  a.accumulate = accumulate ? 1 : 0;

  // dH = dY W2^T with the SwiGLU backward epilogue
  BwdArgs g = a;
  g.n_out = f;
  g.num_n_tiles = (f + BN - 1) / BN;
  g.num_kb = d / BK;
  g.ab = static_cast<const __nv_bfloat16 *>(P.ab);
  g.dab = static_cast<__nv_bfloat16 *>(P.dab);
  g.force_timeout = force_timeout ? 1 : 0;
  cudaError_t err = launch_one<KIND_DGRAD_H>(num_sms, s, tm_dye_k, tm_w2_k, tm_w2_k, g);
  if (err == cudaSuccess) err = mark(0);
  if (err != cudaSuccess) return err;

  // dW2 = H^T dY (needs only dY: it runs before dX so H leaves L2 late)
  g = a;
  g.m_total = f;
  g.n_out = d;
  g.num_n_tiles = (d + BN - 1) / BN;
  g.out0 = static_cast<float *>(dW2);
  err = launch_one<KIND_WGRAD_W2>(num_sms, s, tm_h_mn, tm_dye_mn, tm_dye_mn, g);
  if (err == cudaSuccess) err = mark(1);
  if (err != cudaSuccess) return err;

  // dX = [da | db] [W1 | W3]^T over K = 2f
  g = a;
  g.n_out = d;
  g.num_n_tiles = (d + BN - 1) / BN;
  g.num_kb = 2 * f / BK;
  g.kb_bank = f / BK;
  g.out0 = P.dxc;
  err = launch_one<KIND_DGRAD_X>(num_sms, s, tm_dab_k, tm_w1_k, tm_w3_k, g);
  if (err == cudaSuccess) err = mark(2);
  if (err != cudaSuccess) return err;

  // [dW1 | dW3] = X^T [da | db]
  g = a;
  g.m_total = d;
  g.n_out = 2 * f;
  g.num_n_tiles = (2 * f + BN - 1) / BN;
  g.out0 = static_cast<float *>(dW1);
  g.out1 = static_cast<float *>(dW3);
  err = launch_one<KIND_WGRAD_W13>(num_sms, s, tm_x_mn, tm_dab_mn, tm_dab_mn, g);
  if (err == cudaSuccess) err = mark(3);
  return err;
}

}  // namespace moe
