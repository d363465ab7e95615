// gemm_tc.cu -- the two grouped expert GEMMs of the bf16 path on 5th-generation
// tensor cores (tcgen05.mma, accumulators in TMEM, operands staged by TMA).
//
//   gate/up:  for each expert e and its grouped rows X_e (padded segment of
//             X_perm):  H_e = SiLU(X_e W1[e]) (.) (X_e W3[e])      (bf16 out)
//   down:     O_e = gate (.) (H_e W2[e]), fp32, optionally split over K
//             ("Expert Network Structure (SwiGLU)" and the gate-weighted sum of
//             section 3.4 "MoE Layer Formulation", Mixtral of Experts summary
//             pages).
//
// One persistent kernel per GEMM, one 192-thread CTA per SM:
//   warp 0      TMA producer (one elected thread): A tile 128x64 (K-major,
//               128-byte swizzle) and B tile 64x256 (four 64-column boxes,
//               N-major since the weights are stored [E, K, N]) per stage;
//   warp 1      TMEM allocator + MMA issuer (one thread): 4 x (M128 N256 K16)
//               per 64-deep k-block into one of two 256-column accumulators;
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, SwiGLU or gate
//               scale, global stores; the second accumulator lets the next
//               tile's MMAs run under this tile's epilogue.
// For gate/up the 256 accumulator columns hold 128 columns of X W1 followed by
// the same 128 columns of X W3, so one MMA feeds both SwiGLU branches.
//
// Every mbarrier wait is bounded (about one second); on expiry the CTA records
// MOE_ERR_DEVICE_TIMEOUT in the status word, stops issuing work, waits (again
// bounded) for its own copies and MMAs in flight, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;    // 16 KiB
constexpr int B_CHUNK = 64 * BK * 2;    // 8 KiB: 64 N-columns x 64 K-rows
constexpr int B_BYTES = 4 * B_CHUNK;    // 32 KiB
constexpr int STAGE_TX = A_BYTES + B_BYTES;
constexpr int ACC_COLS = BN;
constexpr int TMEM_COLS = 2 * ACC_COLS;  // 512: the whole TMEM of the SM
constexpr int NUM_THREADS = 192;
constexpr int GROUP_M = 8;               // m-tiles rastered together (weight reuse in L2)
constexpr uint64_t kTimeoutNs = 1000000000ull;

enum { MODE_GATE_UP = 0, MODE_DOWN = 1 };

struct GemmArgs {
  const int32_t *poffsets;  // [E+1] padded segment starts (device)
  const float *perm_gate;   // [R] gate of each grouped row (down only)
  void *out;                // gate/up: bf16 H [R, n_out]; down: fp32 O [splits, R, n_out]
  long long out_split_stride;
  int E;
  int rows_bound;           // R: rows of the grouped buffers
  int n_out;                // output columns: f (gate/up) or d (down)
  int num_n_tiles;
  int num_kb;               // k-blocks of 64 over the contraction
  int splits;
  int kb_per_split;
  int *status;
};

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int tstart[kMaxE + 1];
  int mtiles[kMaxE];
  int poff[kMaxE + 1];
};

constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * (A_BYTES + B_BYTES) + 1024 /*Ctrl*/;
static_assert(sizeof(Ctrl) <= 1024, "control block too large");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct Tile {
  int e, mt, nt, s;
};

// Tiles of expert e are ordered (m-group, split, n-tile, m-tile within group)
// with the m-tile fastest, so CTAs running together share one weight panel.
__device__ __forceinline__ Tile decode_tile(int tile, const Ctrl &c, int NT, int S) {
  Tile t;
  int e = 0;
  while (tile >= c.tstart[e + 1]) ++e;
  int r = tile - c.tstart[e];
  const int mt_e = c.mtiles[e];
  const int per_m = NT * S;
  const int full_groups = mt_e / GROUP_M;
  const int group_tiles = GROUP_M * per_m;
  int g, gs;
  if (r < full_groups * group_tiles) {
    g = r / group_tiles;
    r -= g * group_tiles;
    gs = GROUP_M;
  } else {
    g = full_groups;
    r -= full_groups * group_tiles;
    gs = mt_e - full_groups * GROUP_M;
  }
  const int mi = r % gs;
  r /= gs;
  t.e = e;
  t.nt = r % NT;
  t.s = r / NT;
  t.mt = g * GROUP_M + mi;
  return t;
}

// Bounded mbarrier wait.  Returns false if the CTA is aborting (when
// honor_abort) or the wait expired; expiry records MOE_ERR_DEVICE_TIMEOUT and
// raises the CTA's abort flag.
__device__ __noinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, Ctrl &c, int *status, bool honor_abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (honor_abort && *reinterpret_cast<volatile int *>(&c.abort)) return false;
      if (ptx::globaltimer_ns() - t0 > kTimeoutNs) {
        *reinterpret_cast<volatile int *>(&c.abort) = 1;
        atomicCAS(status, 0, MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = base;
  uint8_t *sB = base + STAGES * A_BYTES;
  Ctrl &c = *reinterpret_cast<Ctrl *>(sB + STAGES * B_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = args.num_n_tiles, S = args.splits;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&c.full[s], 1);
      ptx::mbar_init(&c.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&c.tfull[a], 1);
      ptx::mbar_init(&c.tempty[a], 4);  // one arrive per epilogue warp
    }
    ptx::mbar_init(&c.drain, 1);
    ptx::fence_barrier_init();
  }
  // Everything above overlaps the previous kernel's tail (programmatic
  // dependent launch); its outputs are read only after this wait.
  ptx::grid_dependency_wait();
  ptx::allow_dependent_launch();
  if (threadIdx.x == 0) {
    // Tile table from the padded segment offsets written by the grouping kernel.
    int acc = 0;
    bool bad = false;
    for (int e = 0; e < args.E; ++e) {
      const int p0 = args.poffsets[e], p1 = args.poffsets[e + 1];
      if (p1 < p0 || (p1 - p0) % BM != 0 || p1 > args.rows_bound) bad = true;
      const int mt = bad ? 0 : (p1 - p0) / BM;
      c.poff[e] = p0;
      c.mtiles[e] = mt;
      c.tstart[e] = acc;
      acc += mt * NT * S;
    }
    if (bad) {
      atomicCAS(args.status, 0, MOE_ERR_DEVICE_BOUNDS);
      for (int e = 0; e < args.E; ++e) { c.mtiles[e] = 0; c.tstart[e] = 0; }
      acc = 0;
    }
    c.poff[args.E] = args.poffsets[args.E];
    c.tstart[args.E] = acc;
    c.total_tiles = acc;
    c.abort = 0;
  }
  __syncthreads();
  const int total = c.total_tiles;
  if (static_cast<int>(blockIdx.x) >= total) return;  // uniform exit, nothing allocated

  if (warp == 1) {
    ptx::tmem_alloc(&c.tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB0);
    if (MODE == MODE_GATE_UP) ptx::prefetch_tmap(&tmB1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  // Producer bookkeeping for the abort drain: stages ever filled and the
  // phase parity of each one's latest fill.
  uint32_t issued = 0, last_par = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_a = ptx::policy_evict_last();
      const uint64_t pol_b = ptx::policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const Tile t = decode_tile(tile, c, NT, S);
        const int row0 = c.poff[t.e] + t.mt * BM;
        const int kb0 = t.s * args.kb_per_split;
        const int kb1 = min(args.num_kb, kb0 + args.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded(&c.empty[stage], phase ^ 1u, c, args.status, true)) { ok = false; break; }
          uint64_t *bar = &c.full[stage];
          ptx::mbar_arrive_expect_tx(bar, STAGE_TX);
          uint8_t *a_dst = sA + stage * A_BYTES;
          uint8_t *b_dst = sB + stage * B_BYTES;
          ptx::tma_load_2d(a_dst, &tmA, bar, kb * BK, row0, pol_a);
          if (MODE == MODE_GATE_UP) {
            const int n0 = t.nt * (BN / 2);
            ptx::tma_load_3d(b_dst, &tmB0, bar, n0, kb * BK, t.e, pol_b);
            ptx::tma_load_3d(b_dst + B_CHUNK, &tmB0, bar, n0 + 64, kb * BK, t.e, pol_b);
            ptx::tma_load_3d(b_dst + 2 * B_CHUNK, &tmB1, bar, n0, kb * BK, t.e, pol_b);
            ptx::tma_load_3d(b_dst + 3 * B_CHUNK, &tmB1, bar, n0 + 64, kb * BK, t.e, pol_b);
          } else {
            const int n0 = t.nt * BN;
#pragma unroll
            for (int j = 0; j < 4; ++j) ptx::tma_load_3d(b_dst + j * B_CHUNK, &tmB0, bar, n0 + 64 * j, kb * BK, t.e, pol_b);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, /*A MN-major*/ false, /*B MN-major*/ true);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const Tile t = decode_tile(tile, c, NT, S);
        const int kb0 = t.s * args.kb_per_split;
        const int kb1 = min(args.num_kb, kb0 + args.kb_per_split);
        const int acc = local & 1;
        const uint32_t apar = (local >> 1) & 1;
        if (!wait_bounded(&c.tempty[acc], apar ^ 1u, c, args.status, true)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * ACC_COLS;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded(&c.full[stage], phase, c, args.status, true)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(sA + stage * A_BYTES);
          const uint32_t b_addr = ptx::smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            // A: K-major, 128 B rows, 8-row groups 1024 B apart; K step = 32 B.
            const uint64_t ad = ptx::smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            // B: N-major, 64-column chunks 8 KiB apart (LBO), 8-row K groups 1024 B apart (SBO); K step = 16 rows.
            const uint64_t bd = ptx::smem_desc_sw128(b_addr + ks * 2048, B_CHUNK, 1024);
            ptx::mma_bf16(d_tmem, ad, bd, idesc, (kb > kb0 || ks > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&c.empty[stage]);  // frees the stage once these MMAs have read it
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit(&c.tfull[acc]);      // accumulator ready for the epilogue
        ++local;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode_tile(tile, c, NT, S);
      const int acc = local & 1;
      const uint32_t apar = (local >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = wait_bounded(&c.tfull[acc], apar, c, args.status, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      const int row = c.poff[t.e] + t.mt * BM + q * 32 + lane;
      const uint32_t tbase = tmem + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      if (MODE == MODE_GATE_UP) {
        __nv_bfloat16 *H = static_cast<__nv_bfloat16 *>(args.out);
        const int n0 = t.nt * (BN / 2);
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t g[32], u[32];
          ptx::tmem_ld_32x32b_x32(tbase + cc * 32, g);
          ptx::tmem_ld_32x32b_x32(tbase + BN / 2 + cc * 32, u);
          ptx::tmem_wait_ld();
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float h0 = silu_f(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
            const float h1 = silu_f(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
            __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
            packed[j] = *reinterpret_cast<uint32_t *>(&hb);
          }
          const int col = n0 + cc * 32;
          __nv_bfloat16 *dst = H + static_cast<size_t>(row) * args.n_out + col;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            if (col + v * 8 < args.n_out)
              *reinterpret_cast<uint4 *>(dst + v * 8) =
                  make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      } else {
        float *O = static_cast<float *>(args.out) + static_cast<size_t>(t.s) * args.out_split_stride;
        const float gsc = args.perm_gate[row];
        const int n0 = t.nt * BN;
#pragma unroll 1
        for (int cc = 0; cc < BN / 32; ++cc) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tbase + cc * 32, v);
          ptx::tmem_wait_ld();
          const int col = n0 + cc * 32;
          float *dst = O + static_cast<size_t>(row) * args.n_out + col;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (col + 4 * j < args.n_out)
              *reinterpret_cast<float4 *>(dst + 4 * j) =
                  make_float4(__uint_as_float(v[4 * j]) * gsc, __uint_as_float(v[4 * j + 1]) * gsc,
                              __uint_as_float(v[4 * j + 2]) * gsc, __uint_as_float(v[4 * j + 3]) * gsc);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&c.tempty[acc]);
      ++local;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*reinterpret_cast<volatile int *>(&c.abort)) {
    // Some role gave up: before TMEM and shared memory are released, wait
    // (bounded) for this CTA's MMAs and for every copy it issued.
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
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 row-major [rows, cols] matrix, box = 64 columns x box_rows rows, 128-byte swizzle.
bool tmap_2d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 bank [E, rows, cols] (cols contiguous), box = 64 x 64 x 1, 128-byte swizzle.
bool tmap_3d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t E) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, E};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_smem_attrs() {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  static std::mutex mu;
  static bool done[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  err = cudaFuncSetAttribute(expert_gemm_kernel<MODE_GATE_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(expert_gemm_kernel<MODE_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES);
  if (err == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return err;
}

}  // namespace

cudaError_t launch_expert_gemms_bf16(const void *W1, const void *W3, const void *W2, int d, int f, int E,
                                     const WsLayout &L, const Ptrs &P, unsigned flags, int num_sms,
                                     cudaStream_t s, void *const *mid_event) {
  (void)flags;
  cudaError_t err = set_smem_attrs();
  if (err != cudaSuccess) return err;
  CUtensorMap tm_x, tm_w1, tm_w3, tm_h, tm_w2;
  if (!tmap_2d(&tm_x, P.xperm, d, L.R, BM) || !tmap_3d(&tm_w1, W1, f, d, E) || !tmap_3d(&tm_w3, W3, f, d, E) ||
      !tmap_2d(&tm_h, P.hbuf, f, L.R, BM) || !tmap_3d(&tm_w2, W2, d, f, E))
    return cudaErrorInvalidValue;

  GemmArgs g1{};
  g1.poffsets = P.poffsets;
  g1.perm_gate = P.perm_gate;
  g1.out = P.hbuf;
  g1.out_split_stride = 0;
  g1.E = E;
  g1.rows_bound = L.R;
  g1.n_out = f;
  g1.num_n_tiles = (f + BN / 2 - 1) / (BN / 2);
  g1.num_kb = (d + BK - 1) / BK;
  g1.splits = 1;
  g1.kb_per_split = g1.num_kb;
  g1.status = P.status;
  err = launch_kernel(expert_gemm_kernel<MODE_GATE_UP>, dim3(num_sms), dim3(NUM_THREADS), SMEM_BYTES, s, true, tm_x,
                      tm_w1, tm_w3, g1);
  if (err == cudaSuccess && mid_event) err = cudaEventRecord(static_cast<cudaEvent_t>(*mid_event), s);
  if (err != cudaSuccess) return err;

  GemmArgs g2 = g1;
  g2.out = P.obuf;
  g2.out_split_stride = static_cast<long long>(L.R) * d;
  g2.n_out = d;
  g2.num_n_tiles = (d + BN - 1) / BN;
  g2.num_kb = (f + BK - 1) / BK;
  g2.splits = L.S;
  g2.kb_per_split = L.kb_per_split;
  return launch_kernel(expert_gemm_kernel<MODE_DOWN>, dim3(num_sms), dim3(NUM_THREADS), SMEM_BYTES, s,
                       mid_event == nullptr, tm_h, tm_w2, tm_w2, g2);
}

}  // namespace moe
