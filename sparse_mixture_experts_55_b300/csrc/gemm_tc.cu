// gemm_tc.cu -- the two grouped expert GEMMs of the forward pass on
// 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM, operands
// staged by TMA), for bf16 weights and for e4m3 weights (FP8).
//
//   gate/up:  for each expert e and its grouped rows X_e (padded segment of
//             X_perm):  H_e = SiLU(X_e W1[e]) (.) (X_e W3[e])      (bf16 out)
//   down:     O_e = gate (.) (H_e W2[e]), fp32, optionally split over K; when
//             not split, the epilogue also adds each token's K slot rows and
//             stores y (the combine)
//             ("Expert Network Structure (SwiGLU)" and the gate-weighted sum of
//             section 3.4 "MoE Layer Formulation", Mixtral of Experts summary
//             pages).
//
// One persistent kernel per GEMM, launched as clusters (one CTA of 192
// threads per SM), in one of three forms chosen per call (all compute every
// tile in the same order, so their results are bitwise identical):
//
// Pair MMA (FORM_PAIR; default once experts average 16 or more 128-row tiles,
//   8 with e4m3 weights):
//   the two CTAs run one 256x256 tile together with tcgen05.mma.cta_group::2:
//   rows 128r..128r+127 come from CTA r's A tile and CTA r holds half of the
//   256 B columns, so each CTA stages 16 KiB of A and 16 KiB of B per
//   64-deep k-block (6-stage ring) and its TMEM receives its own 128 rows x
//   256 columns.  Copies of both CTAs complete on the first CTA's stage
//   barrier; that CTA's single MMA thread issues M256 N256 K16 MMAs and its
//   commits release the stage (and hand the accumulator to the epilogue) in
//   both CTAs.  An expert with an odd tile count pairs its last tile with a
//   phantom tile whose rows are computed but never stored.
// Multicast pairs (FORM_MC2; default below that): each CTA computes its own
//   128x256 tile with cta_group::1 MMAs; the two CTAs work on a pair of
//   tiles that share an operand, and each loads half of the shared operand
//   and multicasts it to both:
//   M-pair  tiles (m, n) and (m+1, n) of one expert share the 64x256 weight
//           tile: each CTA loads its own 128x64 A tile and two of the four
//           64-column B boxes, multicast (32 KiB per CTA per k-block
//           instead of 48);
//   N-pair  for the last m-tile of an expert with an odd count, tiles
//           (m, n) and (m, n+1) share the A tile: each CTA loads 64 of its
//           128 rows multicast and its own B tile.
//   A stage is refilled only after both CTAs' MMAs have read it (4 stages).
// 2x2 multicast (FORM_MC4; MOE_GEMM_QUAD only): 4-CTA clusters, CTA (i, j)
//   runs tile (2p+i, 2q+j); rows share A and columns share B, each CTA
//   loading half of both.
// Roles per CTA:
//   warp 0      TMA producer (one elected thread), shared-memory ring
//               (A 128x64 K-major; bf16 B in 64x64 N-major blocks since the
//               weights are stored [E, K, N], two blocks per copy when N is a
//               multiple of 128; e4m3 B K-major; 128-byte swizzle); weight banks are addressed by slot (wslot[e]) so
//               that an expert cache can hold them in any order;
//   warp 1      TMEM allocator + MMA issuer (one thread) into one of two
//               256-column accumulators;
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, SwiGLU or gate
//               scale, global stores; the second accumulator lets the next
//               tile's MMAs run under this tile's epilogue.
// For gate/up the 256 accumulator columns hold 128 columns of X W1 followed by
// the same 128 columns of X W3, so one MMA feeds both SwiGLU branches.  The
// training forward also stores a = X W1 and b = X W3 (save_ab).
//
// Launch overlap: the kernel is launched with programmatic dependent launch.
// Before its grid-dependency wait each producer builds the unit table and
// issues the weight (B) copies of its first ring stages, which depend on
// nothing the previous kernel writes; the activation (A) copies follow the
// wait.
// Tail split (multicast pairs, unsplit contractions of 8192 or more
// elements, three or more waves): the units of the last, partial wave run as
// two halves of the contraction on twice as many clusters.  The first-half
// CTA stores its fp32 sums into a workspace slot and raises a counter; the
// second-half CTA waits for it (bounded), adds the slot to its own
// accumulator in a fixed order and runs the tile's normal epilogue, so the
// result does not depend on which half finishes first.
//
// Every mbarrier wait is bounded (about one second); on expiry the CTA records
// MOE_ERR_DEVICE_TIMEOUT in the status word, stops issuing work, waits (again
// bounded) for its own copies and MMAs in flight, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "fp8_codec.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "stamps.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;    // 16 KiB
constexpr int B_CHUNK = 64 * BK * 2;    // 8 KiB: 64 N-columns x 64 K-rows
constexpr int MAX_STAGES = 6;
// Ring geometry of the two forms (stages, B bytes per CTA and stage).
template <bool PAIR>
struct Ring {
  static constexpr int STAGES = PAIR ? 6 : 4;
  static constexpr int B_BYTES = (PAIR ? 2 : 4) * B_CHUNK;  // half or all of the 256 B columns
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // bytes that complete one stage: both CTAs' copies (pair MMA: on the first
  // CTA's barrier) or this CTA's A plus all four B boxes (multicast pairs)
  static constexpr int STAGE_TX = PAIR ? 2 * STAGE_BYTES : A_BYTES + 4 * B_CHUNK;
  static constexpr int SMEM = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + 1024 /*Ctrl*/;
};
static_assert(Ring<true>::SMEM <= 232448 && Ring<false>::SMEM <= 232448, "shared memory budget");
constexpr int ACC_COLS = BN;
constexpr int TMEM_COLS = 2 * ACC_COLS;  // 512: the whole TMEM of the SM
constexpr int NUM_THREADS = 192;
constexpr uint16_t kBothCtas = 0x3;
constexpr int GROUP_PAIRS = 16;          // M-pairs rastered together (weight reuse in L2)

// The three forms of the kernel (see the file comment).
enum { FORM_MC2 = 0, FORM_PAIR = 1, FORM_MC4 = 2 };
template <int FORM>
struct FormInfo {
  static constexpr bool PAIR = FORM == FORM_PAIR;  // cta_group::2 MMAs
  static constexpr bool QUAD = FORM == FORM_MC4;   // 2x2 tiles per cluster
  static constexpr int CL = QUAD ? 4 : 2;           // CTAs per cluster
  static constexpr uint16_t ALL = QUAD ? 0xF : 0x3;
};

enum { MODE_GATE_UP = 0, MODE_DOWN = 1 };

struct GemmArgs {
  const int32_t *poffsets;  // [E+1] padded segment starts (device)
  const int32_t *offsets;   // [E+1] unpadded segment starts (device)
  const float *perm_gate;   // [R] gate of each grouped row (down only)
  void *out;                // gate/up: bf16 H [R, n_out]; down: fp32 O [splits, T*K, n_out]
  long long out_split_stride;
  float *part;              // gate/up with splits > 1: fp32 partial sums [splits, T*K, 2*n_out]
  int *tile_cnt;            // gate/up with splits > 1: arrivals per (m-tile, n-tile, lane quarter), zero at launch
  int E;
  int rows_bound;           // R: rows of the padded grouped buffers
  int tk;                   // T*K: rows of the compact buffers
  int n_out;                // output columns: f (gate/up) or d (down)
  int num_n_tiles;
  int num_kb;               // k-blocks of 64 over the contraction
  int splits;
  int kb_per_split;
  int force_timeout;        // failure-path test: wait on a barrier nothing signals first
  // e4m3 operands only: per-row scale of A (indexed by padded row), per-column
  // scales of B ([E, n_out]; col_scale1 is the W3 bank's for gate/up), and
  // the per-(row, n-tile) maxima of the bf16 H values the gate/up writes
  const float *row_scale;
  const float *col_scale0;
  const float *col_scale1;
  float *habs;
  // e4m3 weight banks in 128 x 128 tiles: tiles per expert along N and K
  int b_nt, b_kt;
  // training forward (bf16 gate/up without splits): also store the
  // pre-activations a = X W1 and b = X W3 as bf16 [R, 2 n_out] (a in columns
  // [0, n_out), b after), for every row of the segments including padding
  __nv_bfloat16 *save_ab;
  int *status;
  // weight banks indexed by slot: expert e's matrices are slot wslot[e] of
  // the banks (use_slots; otherwise slot e)
  int use_slots;
  int wslot[kMaxE];
  // fused combine: y [T, n_out] bf16 gets, per token and 256-column tile,
  // the sum over its K slot rows of O in slot order, formed by whichever
  // slot's epilogue arrives last on tok_cnt
  __nv_bfloat16 *y;
  int y_accumulate;
  int keep_o;               // store every slot row of O (the training forward's backward reads them)
  int b4d;                  // bf16 weights through the 4-D map: one copy per 128 columns
  const int32_t *pos;       // [T*K] unpadded grouped row of each (token, slot)
  const int32_t *perm_tok;  // [R] token of each padded grouped row
  int *tok_cnt;             // [T, num_n_tiles], zero at launch
  int T, K;
  unsigned long long *stamps;  // profiling calls: stage begin/end times (stamps.cuh), else null
  // tail split (multicast pairs, unsplit contraction): scratch for the fp32
  // first halves of the last wave's tiles, [tail_slots][2][BM][BN], and one
  // arrival counter per (slot, CTA), zero at launch; null disables it
  float *tail_part;
  int *tail_flag;
  int tail_slots;
};

struct Ctrl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t stall;           // never signalled (failure-path test)
  uint64_t exit_bar;        // the peer CTA's "done issuing" arrival
  uint32_t tmem_base;
  int abort;
  int total_units;
  int total_items;  // work items: units, with the last wave's units split in two halves when tail_base >= 0
  int tail_base;
  int ustart[kMaxE + 1];
  int mtiles[kMaxE];
  int poff[kMaxE + 1];
  int uoff[kMaxE + 1];
  int wslot[kMaxE];
};

static_assert(sizeof(Ctrl) <= 1024, "control block too large");

struct Tile {
  int e, mt, nt, s;
  bool npair;  // the pair shares A (N-pair) rather than B (M-pair)
};

// Units of expert e: its M-pairs ordered (pair group, split, n-tile, pair in
// group) with the pair fastest, so clusters running together share weight
// panels; then, for an odd m-tile count, the N-pairs of its last m-tile
// (multicast pairs; interleaved with the M-pairs of their n-tiles when the
// expert has one pair group) or one more M-pair with a phantom second tile
// (pair MMA).
template <int FORM>
__device__ __forceinline__ int units_of(int mt_e, int NT, int S) {
  if (FORM == FORM_PAIR) return ((mt_e + 1) >> 1) * NT * S;
  if (FORM == FORM_MC4) return (mt_e >> 1) * ((NT + 1) >> 1) * S + (mt_e & 1) * ((NT + 3) >> 2) * S;
  return (mt_e >> 1) * NT * S + (mt_e & 1) * ((NT + 1) >> 1) * S;
}

template <int FORM>
__device__ __forceinline__ Tile decode_unit(int u, const Ctrl &c, int NT, int S, int rank) {
  Tile t;
  int e = 0;
  while (u >= c.ustart[e + 1]) ++e;
  int r = u - c.ustart[e];
  const int mt_e = c.mtiles[e];
  const int mp = FORM == FORM_PAIR ? (mt_e + 1) >> 1 : mt_e >> 1;
  if (FORM == FORM_MC2 && (mt_e & 1) && mp <= GROUP_PAIRS) {
    // Multicast pairs, odd tile count, one pair group: per split, blocks of
    // the M-pairs of n-tiles 2j and 2j+1 (pair fastest) followed by the
    // N-pair of those two n-tiles on the last m-tile, so the N-pair reads the
    // weight panels while the M-pairs still hold them in L2.
    const int per_s = NT * mp + ((NT + 1) >> 1);
    t.e = e;
    t.s = r / per_s;
    r -= t.s * per_s;
    const int blk = 2 * mp + 1;
    const int j = r / blk;
    const int w = r - j * blk;
    if (w < min(2, NT - 2 * j) * mp) {
      const int q = w / mp;  // mp > 0 here
      t.nt = 2 * j + q;
      t.mt = 2 * (w - q * mp) + rank;
      t.npair = false;
    } else {
      t.nt = 2 * j + rank;  // may reach NT: all its loads and stores fall outside
      t.mt = mt_e - 1;
      t.npair = true;
    }
    return t;
  }
  // n positions per M-pair unit: every n-tile, or n-tile pairs for 2x2 tiles
  const int nu = FORM == FORM_MC4 ? (NT + 1) >> 1 : NT;
  const int per = nu * S;
  t.e = e;
  if (r < mp * per) {
    const int full_groups = mp / GROUP_PAIRS;
    const int group_units = GROUP_PAIRS * per;
    int g, gs;
    if (r < full_groups * group_units) {
      g = r / group_units;
      r -= g * group_units;
      gs = GROUP_PAIRS;
    } else {
      g = full_groups;
      r -= full_groups * group_units;
      gs = mp - full_groups * GROUP_PAIRS;
    }
    const int pi = r % gs;
    r /= gs;
    if (FORM == FORM_MC4) {
      // CTA (i, j) = (rank >> 1, rank & 1) takes m-tile 2p + i, n-tile 2q + j
      t.nt = 2 * (r % nu) + (rank & 1);  // may equal NT for odd NT: all its loads and stores fall outside
      t.s = r / nu;
      t.mt = 2 * (g * GROUP_PAIRS + pi) + (rank >> 1);
    } else {
      t.nt = r % NT;
      t.s = r / NT;
      t.mt = 2 * (g * GROUP_PAIRS + pi) + rank;
    }
    t.npair = false;
  } else {
    // the last m-tile of an odd count: the cluster's CTAs take consecutive
    // n-tiles of it and share its A tile
    r -= mp * per;
    const int nc = FORM == FORM_MC4 ? 4 : 2;
    const int ntg = (NT + nc - 1) / nc;
    t.nt = nc * (r % ntg) + rank;  // may reach NT: all its loads and stores fall outside
    t.s = r / ntg;
    t.mt = mt_e - 1;
    t.npair = true;
  }
  return t;
}

// Work item `it` of the persistent schedule: a whole unit, or (the tail
// split) one k-half of one of the last wave's units.  Items before tail_base
// are units; item tail_base + j is half (j & 1) of unit tail_base + (j >> 1),
// both halves computing the same tiles: the first half (role 1) stores its
// fp32 sums, the second (role 2, the owner) adds them and runs the epilogue.
struct Work {
  Tile t;
  int kb0, kb1, role, slot;
};

template <int FORM>
__device__ __forceinline__ Work work_item(int it, const Ctrl &c, int NT, int S, int rank, int kb_per_split, int num_kb) {
  Work w;
  int unit = it;
  w.role = 0;
  w.slot = 0;
  if (c.tail_base >= 0 && it >= c.tail_base) {
    const int j = it - c.tail_base;
    unit = c.tail_base + (j >> 1);
    w.role = 1 + (j & 1);
    w.slot = j >> 1;
  }
  w.t = decode_unit<FORM>(unit, c, NT, S, rank);
  w.kb0 = w.t.s * kb_per_split;
  w.kb1 = min(num_kb, w.kb0 + kb_per_split);
  if (w.role) {
    const int mid = w.kb0 + (w.kb1 - w.kb0) / 2;
    if (w.role == 1) w.kb1 = mid;
    else w.kb0 = mid;
  }
  return w;
}

// Bounded wait until *p reaches target (a counter other CTAs raise); records
// MOE_ERR_DEVICE_TIMEOUT and returns false after about one second.
__device__ __noinline__ bool wait_count(const int *p, int target, int *status) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (*reinterpret_cast<const volatile int *>(p) < target) {
    if (ptx::globaltimer_ns() - t0 > kTimeoutNs) {
      atomicCAS(status, 0, MOE_ERR_DEVICE_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Bounded wait until the high 16 bits of *p (the signals of a token's slot
// rows whose O stores are out) reach target; as wait_count otherwise.
__device__ __noinline__ bool wait_signals(const int *p, int target, int *status) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while ((*reinterpret_cast<const volatile int *>(p) >> 16) < target) {
    if (ptx::globaltimer_ns() - t0 > kTimeoutNs) {
      atomicCAS(status, 0, MOE_ERR_DEVICE_TIMEOUT);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

// SiLU(g) = g / (1 + e^-g) with CUDA's fast exponential and fast division
// intrinsics (a few ulp of fp32; the result is rounded to bf16 next).  An
// IEEE division's longer dependent chain made this the epilogue's cost at
// decode sizes, where one warp holds a tile's real rows.  For g below about
// -88, e^-g is infinite and the quotient is 0, SiLU's limit.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

template <int MODE, int FORM, bool FP8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA_half,
                       const __grid_constant__ CUtensorMap tmA_quarter, const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, const GemmArgs args) {
  constexpr bool PAIR = FormInfo<FORM>::PAIR;
  constexpr bool QUAD = FormInfo<FORM>::QUAD;
  constexpr int CL = FormInfo<FORM>::CL;
  constexpr uint16_t kAll = FormInfo<FORM>::ALL;  // every CTA of the cluster
  using RG = Ring<PAIR>;
  constexpr int STAGES = RG::STAGES;
  // a k-block is one 128-byte row of A and of B in shared memory: 64 bf16 or
  // 128 e4m3 elements of the contraction
  constexpr int KB_ELEMS = FP8 ? 128 : BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = base;
  uint8_t *sB = base + STAGES * A_BYTES;
  Ctrl &c = *reinterpret_cast<Ctrl *>(sB + STAGES * RG::B_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = args.num_n_tiles, S = args.splits;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const int cluster = static_cast<int>(ptx::cluster_id_x());
  const int nclusters = static_cast<int>(ptx::num_clusters_x());
  // Pair MMA: CTA 0 of the pair issues every MMA and owns the stage-full and
  // accumulator-empty barriers that both CTAs signal.
  const bool leader = !PAIR || rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&c.full[s], 1);
      // multicast forms: every CTA's MMAs release a stage; pair MMA: one commit
      ptx::mbar_init(&c.empty[s], PAIR ? 1 : CL);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&c.tfull[a], 1);
      ptx::mbar_init(&c.tempty[a], PAIR ? 8 : 4);  // one arrive per epilogue warp (of both CTAs for PAIR)
    }
    ptx::mbar_init(&c.drain, 1);
    ptx::mbar_init(&c.stall, 1);
    ptx::mbar_init(&c.exit_bar, CL - 1);  // the other CTAs' "done" arrivals
    ptx::fence_barrier_init();
  }
  // Barriers must be initialised in both CTAs before either signals the other.
  ptx::cluster_sync_all();
  constexpr int kStage = MODE == MODE_GATE_UP ? ST_GATE_UP : ST_DOWN;
  stamp_begin(args.stamps, kStage);
  // Everything up to grid_dependency_wait overlaps the previous kernel's tail
  // (programmatic dependent launch).  The routing arrays read here (segment
  // offsets) are older: this grid is launched only once every CTA of the
  // previous kernel has passed its own wait, so the kernel that wrote them
  // has completed.
  if (threadIdx.x == 0) {
    // Unit table from the padded segment offsets written by the grouping kernel.
    int acc = 0;
    bool bad = false;
    for (int e = 0; e < args.E; ++e) {
      const int p0 = args.poffsets[e], p1 = args.poffsets[e + 1];
      if (p1 < p0 || (p1 - p0) % BM != 0 || p1 > args.rows_bound) bad = true;
      c.wslot[e] = args.use_slots ? args.wslot[e] : e;
      if (p1 > p0 && c.wslot[e] < 0) bad = true;  // rows routed to an expert that is not resident
      const int mt = bad ? 0 : (p1 - p0) / BM;
      c.poff[e] = p0;
      c.uoff[e] = args.offsets[e];
      c.mtiles[e] = mt;
      c.ustart[e] = acc;
      acc += units_of<FORM>(mt, NT, S);
    }
    if (bad) {
      atomicCAS(args.status, 0, MOE_ERR_DEVICE_BOUNDS);
      for (int e = 0; e < args.E; ++e) { c.mtiles[e] = 0; c.ustart[e] = 0; }
      acc = 0;
    }
    c.poff[args.E] = args.poffsets[args.E];
    c.uoff[args.E] = args.offsets[args.E];
    c.ustart[args.E] = acc;
    c.total_units = acc;
    // Tail split: when the last of several waves of long units (a
    // contraction of 8192 or more elements, the down projection's) leaves
    // most clusters idle, its r units run as 2r halves of their contraction.
    // (Units of 4096 elements, the gate/up projection's, gain nothing: the
    // owner's wait for the partial costs about what the halving saves.)
    int items = acc, tail_base = -1;
    if (FORM == FORM_MC2 && S == 1 && args.tail_part != nullptr && args.num_kb * KB_ELEMS >= 8192) {
      const int waves = (acc + nclusters - 1) / nclusters;
      const int r = acc - (waves - 1) * nclusters;
      if (waves >= 3 && r > 0 && 2 * r <= nclusters && r <= args.tail_slots && args.num_kb >= 2) {
        tail_base = (waves - 1) * nclusters;
        items = tail_base + 2 * r;
      }
    }
    c.total_items = items;
    c.tail_base = tail_base;
    c.abort = 0;
  }
  __syncthreads();
  const int total = c.total_items;
  // Both CTAs of a cluster read the same table, so they leave together.
  if (cluster >= total) return;

  // Producer bookkeeping: stages ever filled, the phase parity of each one's
  // latest fill, and the ring position after the last fill.
  uint32_t issued = 0, last_par = 0;
  int p_stage = 0;
  uint32_t p_phase = 0;
  uint64_t pol_a = 0, pol_b = 0;
  // Stage `st` of k-block k0 of tile t: arm its barrier for all the bytes
  // that complete it, and issue this CTA's weight (B) and activation (A) copies.
  auto stage_bar = [&](int st) -> uint64_t * { return &c.full[st]; };
  // e4m3: first row of the 128 x 128 weight tile holding columns nb.. and
  // k-elements k0.. of bank slot wz, in the tiles' 128-byte-row view
  auto fp8_tile_row = [&](int wz, int nb, int k0) {
    return ((wz * args.b_nt + nb / kFp8Tile) * args.b_kt + k0 / kFp8Tile) * kFp8Tile;
  };
  auto arm = [&](int st) {
    // pair MMA: both CTAs' copies complete on the first CTA's barrier, which
    // expects the bytes of both
    if (!PAIR || leader) ptx::mbar_arrive_expect_tx(stage_bar(st), RG::STAGE_TX);
  };
  auto load_b = [&](int st, const Tile &t, int k0) {
    uint8_t *b_dst = sB + st * RG::B_BYTES;
    const int wz = c.wslot[t.e];  // the bank slot holding expert e's weights
    if (PAIR) {
      // CTA r holds half r of the 256 B columns (gate/up: W1 for CTA 0, W3 for CTA 1)
      const uint32_t bar = ptx::mapa_shared(ptx::smem_u32(&c.full[st]), 0);
      const CUtensorMap *mb = (MODE == MODE_GATE_UP && rank == 1) ? &tmB1 : &tmB0;
      const int nb = MODE == MODE_GATE_UP ? t.nt * (BN / 2) : t.nt * BN + rank * (BN / 2);
      if (FP8) {
        // e4m3 banks are stored in 128 x 128 tiles: one contiguous 16 KiB box
        ptx::tma_load_2d_pair(b_dst, mb, bar, 0, fp8_tile_row(wz, nb, k0), pol_b);
      } else if (args.b4d) {
        ptx::tma_load_4d_pair(b_dst, mb, bar, 0, k0, nb / 64, wz, pol_b);
      } else {
        ptx::tma_load_3d_pair(b_dst, mb, bar, nb, k0, wz, pol_b);
        ptx::tma_load_3d_pair(b_dst + B_CHUNK, mb, bar, nb + 64, k0, wz, pol_b);
      }
      return;
    }
    uint64_t *bar = stage_bar(st);
    // B: half h (128 of the 256 columns) of the tile; gate/up half 0 is W1,
    // half 1 is W3; delivered to the CTAs of the cluster that compute with it
    auto load_b_half = [&](int h, uint16_t mask) {
      const CUtensorMap *mb = (MODE == MODE_GATE_UP && h == 1) ? &tmB1 : &tmB0;
      const int nb = MODE == MODE_GATE_UP ? t.nt * (BN / 2) : t.nt * BN + h * (BN / 2);
      uint8_t *dst = b_dst + h * (2 * B_CHUNK);
      if (FP8) {
        const int row = fp8_tile_row(wz, nb, k0);
        if (mask) ptx::tma_load_2d_mc(dst, mb, bar, 0, row, mask, pol_b);
        else ptx::tma_load_2d(dst, mb, bar, 0, row, pol_b);
      } else if (args.b4d) {
        if (mask) ptx::tma_load_4d_mc(dst, mb, bar, 0, k0, nb / 64, wz, mask, pol_b);
        else ptx::tma_load_4d(dst, mb, bar, 0, k0, nb / 64, wz, pol_b);
      } else {
        if (mask) {
          ptx::tma_load_3d_mc(dst, mb, bar, nb, k0, wz, mask, pol_b);
          ptx::tma_load_3d_mc(dst + B_CHUNK, mb, bar, nb + 64, k0, wz, mask, pol_b);
        } else {
          ptx::tma_load_3d(dst, mb, bar, nb, k0, wz, pol_b);
          ptx::tma_load_3d(dst + B_CHUNK, mb, bar, nb + 64, k0, wz, pol_b);
        }
      }
    };
    if (t.npair) {
      load_b_half(0, 0);  // own n-tile, whole
      load_b_half(1, 0);
    } else if (QUAD) {
      // row i of the 2x2 tiles loads half i of its column's B tile, for both CTAs of that column
      load_b_half(rank >> 1, uint16_t((1u << (rank & 1)) | (1u << (2 + (rank & 1)))));
    } else {
      load_b_half(rank, kBothCtas);  // M-pair: half r, for both CTAs
    }
  };
  auto load_a = [&](int st, const Tile &t, int k0) {
    uint8_t *a_dst = sA + st * A_BYTES;
    const int row0 = c.poff[t.e] + t.mt * BM;
    if (PAIR) {
      const uint32_t bar = ptx::mapa_shared(ptx::smem_u32(&c.full[st]), 0);
      ptx::tma_load_2d_pair(a_dst, &tmA, bar, k0, row0, pol_a);
    } else if (!t.npair && !QUAD) {
      ptx::tma_load_2d(a_dst, &tmA, stage_bar(st), k0, row0, pol_a);  // M-pair: own A tile
    } else {
      // shared A tile: halves (N-pair; 2x2 tiles: the two CTAs of a row)
      // or quarters (the odd m-tile of the 2x2 form: all four CTAs)
      const bool quarter = QUAD && t.npair;
      const int part = quarter ? rank : (QUAD ? (rank & 1) : rank);
      const int prow = quarter ? 32 : 64;
      const uint16_t amask = quarter ? uint16_t(0xF) : (QUAD ? uint16_t(0x3 << (rank & 2)) : kBothCtas);
      ptx::tma_load_2d_mc(a_dst + part * prow * 128, quarter ? &tmA_quarter : &tmA_half, stage_bar(st), k0,
                          row0 + part * prow, amask, pol_a);
    }
  };
  // The weights do not depend on the previous kernel: the first stages of
  // this CTA's first unit get their weight copies before the wait, so the
  // weight stream starts while the previous kernel finishes; their
  // activation copies follow the wait.
  int pre_kb = 0;
  Tile t_first{};
  int kb_first = 0;
  if (warp == 0 && lane == 0) {
    pol_a = ptx::policy_evict_last();
    pol_b = ptx::policy_evict_normal();
    ptx::prefetch_tmap(&tmB0);
    if (MODE == MODE_GATE_UP) ptx::prefetch_tmap(&tmB1);
    const Work w0 = work_item<FORM>(cluster, c, NT, S, rank, args.kb_per_split, args.num_kb);
    t_first = w0.t;
    kb_first = w0.kb0;
    pre_kb = min(STAGES, w0.kb1 - w0.kb0);
    for (int i = 0; i < pre_kb; ++i) {
      arm(i);
      load_b(i, t_first, (kb_first + i) * KB_ELEMS);
    }
    issued = (1u << pre_kb) - 1u;
    p_stage = pre_kb % STAGES;
    p_phase = pre_kb == STAGES ? 1u : 0u;
  }
  ptx::grid_dependency_wait();
  ptx::allow_dependent_launch();

  if (warp == 1) {
    if (PAIR) {
      ptx::tmem_alloc_pair(&c.tmem_base, TMEM_COLS);  // with the peer CTA's warp 1
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&c.tmem_base, TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    if (!PAIR) ptx::prefetch_tmap(&tmA_half);
    if (QUAD) ptx::prefetch_tmap(&tmA_quarter);
    // the activations of the stages whose weights went out before the wait
    for (int i = 0; i < pre_kb; ++i) load_a(i, t_first, (kb_first + i) * KB_ELEMS);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = c.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      for (int u = cluster; ok && u < total; u += nclusters) {
        const Work w = work_item<FORM>(u, c, NT, S, rank, args.kb_per_split, args.num_kb);
        const Tile &t = w.t;
        for (int kb = u == cluster ? w.kb0 + pre_kb : w.kb0; kb < w.kb1; ++kb) {
          if (!wait_bounded(&c.empty[p_stage], p_phase ^ 1u, c, args.status, true)) { ok = false; break; }
          const int k0 = kb * KB_ELEMS;
          arm(p_stage);
          load_b(p_stage, t, k0);
          load_a(p_stage, t, k0);
          issued |= 1u << p_stage;
          last_par = (last_par & ~(1u << p_stage)) | (p_phase << p_stage);
          if (++p_stage == STAGES) { p_stage = 0; p_phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      // pair MMA: M = 256 over both CTAs' rows
      constexpr uint32_t idesc = FP8 ? ptx::idesc_e4m3_f32(PAIR ? 2 * BM : BM, BN)
                                     : ptx::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN, /*A MN-major*/ false,
                                                           /*B MN-major*/ true);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      // failure-path test: this wait expires, raising the CTA's abort flag
      if (args.force_timeout) ok = wait_bounded(&c.stall, 0, c, args.status, true);
      for (int u = cluster; ok && u < total; u += nclusters) {
        const Work w = work_item<FORM>(u, c, NT, S, rank, args.kb_per_split, args.num_kb);
        const int kb0 = w.kb0, kb1 = w.kb1;
        const int acc = local & 1;
        const uint32_t apar = (local >> 1) & 1;
        if (!wait_bounded(&c.tempty[acc], apar ^ 1u, c, args.status, true)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * ACC_COLS;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded(&c.full[stage], phase, c, args.status, true)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(sA + stage * A_BYTES);
          const uint32_t b_addr = ptx::smem_u32(sB + stage * RG::B_BYTES);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            // A: K-major, 128 B rows, 8-row groups 1024 B apart; K step = 32 B
            // (16 bf16 or 32 e4m3 elements per MMA).
            const uint64_t ad = ptx::smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            const uint32_t accum = (kb > kb0 || ks > 0) ? 1u : 0u;
            if (FP8) {
              // B: K-major like A (one 128-byte row per column).
              const uint64_t bd = ptx::smem_desc_sw128(b_addr + ks * 32, 16, 1024);
              if (PAIR) ptx::mma_f8_pair(d_tmem, ad, bd, idesc, accum);
              else ptx::mma_f8(d_tmem, ad, bd, idesc, accum);
            } else {
              // B: N-major, 64-column chunks 8 KiB apart (LBO), 8-row K groups
              // 1024 B apart (SBO); K step = 16 rows.
              const uint64_t bd = ptx::smem_desc_sw128(b_addr + ks * 2048, B_CHUNK, 1024);
              if (PAIR) ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, accum);
              else ptx::mma_bf16(d_tmem, ad, bd, idesc, accum);
            }
          }
          // frees the stage in both CTAs once these MMAs have read it
          if (PAIR) ptx::mma_commit_pair_mc(&c.empty[stage], kAll);
          else ptx::mma_commit_mc(&c.empty[stage], kAll);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        // accumulator ready for the epilogue (of both CTAs for pair MMA)
        if (PAIR) ptx::mma_commit_pair_mc(&c.tfull[acc], kBothCtas);
        else ptx::mma_commit(&c.tfull[acc]);
        ++local;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // where this warp reports a drained accumulator: the MMA-issuing CTA
    const uint32_t tempty_at0 = ptx::mapa_shared(ptx::smem_u32(&c.tempty[0]), PAIR ? 0 : rank);
    const uint32_t tempty_at1 = ptx::mapa_shared(ptx::smem_u32(&c.tempty[1]), PAIR ? 0 : rank);
    int local = 0;
    for (int u = cluster; u < total; u += nclusters) {
      const Work w = work_item<FORM>(u, c, NT, S, rank, args.kb_per_split, args.num_kb);
      const Tile &t = w.t;
      const int acc = local & 1;
      const uint32_t apar = (local >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = wait_bounded(&c.tfull[acc], apar, c, args.status, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      // Tail split: this thread's accumulator row in the (slot, CTA) scratch tile
      float *tail_row = w.role ? args.tail_part + (static_cast<size_t>(w.slot) * 2 + rank) * BM * BN +
                                     static_cast<size_t>(q * 32 + lane) * BN
                               : nullptr;
      if (w.role == 1) {
        // first k-half: store the raw fp32 sums for the owner, release the
        // accumulator, count this warp's arrival
        const uint32_t tb = tmem + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
        for (int cc = 0; cc < BN / 32; ++cc) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tb + cc * 32, v);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4)
            __stcg(reinterpret_cast<float4 *>(tail_row + cc * 32 + 4 * j4),
                   make_float4(__uint_as_float(v[4 * j4]), __uint_as_float(v[4 * j4 + 1]),
                               __uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3])));
        }
        __threadfence();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          atomicAdd(args.tail_flag + w.slot * 2 + rank, 1);
          ptx::mbar_arrive_cluster(acc ? tempty_at1 : tempty_at0);
        }
        ++local;
        continue;
      }
      const float *part = nullptr;  // owner of a split tile: the first half's sums, added below
      if (w.role == 2) {
        int okp = 1;
        if (lane == 0) okp = wait_count(args.tail_flag + w.slot * 2 + rank, 4, args.status) ? 1 : 0;
        okp = __shfl_sync(0xffffffffu, okp, 0);
        __threadfence();
        if (okp) part = tail_row;
      }
      // acc_cols[i] += part[c0 + i]: the first half's sums, in one fixed order
      auto add_part = [&](uint32_t(&r)[32], int c0) {
        if (part == nullptr) return;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 x = __ldcg(reinterpret_cast<const float4 *>(part + c0 + 4 * j4));
          r[4 * j4] = __float_as_uint(x.x + __uint_as_float(r[4 * j4]));
          r[4 * j4 + 1] = __float_as_uint(x.y + __uint_as_float(r[4 * j4 + 1]));
          r[4 * j4 + 2] = __float_as_uint(x.z + __uint_as_float(r[4 * j4 + 2]));
          r[4 * j4 + 3] = __float_as_uint(x.w + __uint_as_float(r[4 * j4 + 3]));
        }
      };
      // This thread's accumulator row: padded grouped row `row`; the first
      // count_e rows of an expert's segment are real, the rest padding, and
      // rows past the segment (the phantom tile of pair MMA) are not stored.
      const int seg_row = t.mt * BM + q * 32 + lane;
      const int row = c.poff[t.e] + seg_row;
      const bool in_seg = seg_row < c.mtiles[t.e] * BM;
      const bool real = seg_row < c.uoff[t.e + 1] - c.uoff[t.e];
      const int ru = c.uoff[t.e] + seg_row;  // unpadded grouped row (valid if real)
      // A warp whose 32 rows are all padding has nothing anyone reads (the down
      // projection drops padding rows), so it skips its quarter entirely.
      // (The training forward keeps every row: the weight gradients contract
      // over whole segments, so padding rows of H and of a, b must be zeros.)
      const bool warp_real = __ballot_sync(0xffffffffu, real) != 0 || (!FP8 && args.save_ab != nullptr);
      const uint32_t tbase = tmem + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      if (MODE == MODE_GATE_UP) {
        const int n0 = t.nt * (BN / 2);
        if (S == 1) {
          __nv_bfloat16 *H = static_cast<__nv_bfloat16 *>(args.out);
          if (n0 < args.n_out && warp_real) {
            // e4m3 operands: accumulators carry codes; scale by the A row's and
            // the B column's scales, and keep the row's max |bf16 H| over the tile
            const float rs = FP8 && in_seg ? args.row_scale[row] : 0.f;  // phantom rows lie past the buffers
            const float *cs1 = FP8 ? args.col_scale0 + static_cast<size_t>(t.e) * args.n_out : nullptr;
            const float *cs3 = FP8 ? args.col_scale1 + static_cast<size_t>(t.e) * args.n_out : nullptr;
            float hmax = 0.f;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
              uint32_t g[32], v[32];
              ptx::tmem_ld_32x32b_x32(tbase + cc * 32, g);
              ptx::tmem_ld_32x32b_x32(tbase + BN / 2 + cc * 32, v);
              ptx::tmem_wait_ld();
              add_part(g, cc * 32);
              add_part(v, BN / 2 + cc * 32);
              if (FP8) {
                const int cb = n0 + cc * 32;
                // the chunk's 32 column scales of each bank: addresses clamped
                // into range so that all sixteen loads are in flight together
                float4 a4s[8], b4s[8];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                  const int c0 = min(cb + 4 * j4, args.n_out - 4);
                  a4s[j4] = __ldg(reinterpret_cast<const float4 *>(cs1 + c0));
                  b4s[j4] = __ldg(reinterpret_cast<const float4 *>(cs3 + c0));
                }
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                  // n_out is a multiple of 16, so a group of four is all in or all out
                  const bool in = cb + 4 * j4 < args.n_out;
                  const float4 a4 = in ? a4s[j4] : make_float4(0, 0, 0, 0);
                  const float4 b4 = in ? b4s[j4] : make_float4(0, 0, 0, 0);
                  const float sa[4] = {a4.x, a4.y, a4.z, a4.w}, sb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    g[4 * j4 + i] = __float_as_uint(__uint_as_float(g[4 * j4 + i]) * rs * sa[i]);
                    v[4 * j4 + i] = __float_as_uint(__uint_as_float(v[4 * j4 + i]) * rs * sb[i]);
                  }
                }
              }
              const int col = n0 + cc * 32;
              if (!FP8 && args.save_ab != nullptr && in_seg) {
                __nv_bfloat16 *pa = args.save_ab + static_cast<size_t>(row) * 2 * args.n_out + col;
                __nv_bfloat16 *pb = pa + args.n_out;
#pragma unroll
                for (int vv = 0; vv < 4; ++vv)
                  if (col + vv * 8 < args.n_out) {
                    uint32_t wa[4], wb[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                      const int c2 = 8 * vv + 2 * j;
                      __nv_bfloat162 ha = __floats2bfloat162_rn(__uint_as_float(g[c2]), __uint_as_float(g[c2 + 1]));
                      __nv_bfloat162 hb2 = __floats2bfloat162_rn(__uint_as_float(v[c2]), __uint_as_float(v[c2 + 1]));
                      wa[j] = *reinterpret_cast<uint32_t *>(&ha);
                      wb[j] = *reinterpret_cast<uint32_t *>(&hb2);
                    }
                    *reinterpret_cast<uint4 *>(pa + vv * 8) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
                    *reinterpret_cast<uint4 *>(pb + vv * 8) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
                  }
              }
              uint32_t packed[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float h0 = silu_f(__uint_as_float(g[2 * j])) * __uint_as_float(v[2 * j]);
                const float h1 = silu_f(__uint_as_float(g[2 * j + 1])) * __uint_as_float(v[2 * j + 1]);
                __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
                if (FP8) {
                  const float2 hr = __bfloat1622float2(hb);
                  hmax = fmaxf(hmax, fmaxf(fabsf(hr.x), fabsf(hr.y)));
                }
                packed[j] = *reinterpret_cast<uint32_t *>(&hb);
              }
              __nv_bfloat16 *dst = H + static_cast<size_t>(row) * args.n_out + col;
              if (in_seg) {
#pragma unroll
                for (int vv = 0; vv < 4; ++vv)
                  if (col + vv * 8 < args.n_out)
                    *reinterpret_cast<uint4 *>(dst + vv * 8) =
                        make_uint4(packed[4 * vv], packed[4 * vv + 1], packed[4 * vv + 2], packed[4 * vv + 3]);
              }
            }
            if (FP8 && in_seg) args.habs[static_cast<size_t>(row) * NT + t.nt] = hmax;
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_cluster(acc ? tempty_at1 : tempty_at0);
        } else {
          // Split contraction: store this split's fp32 sums of the real rows,
          // release the accumulator, and let the CTA that completes the tile
          // (the last of its S splits to arrive) add the S partials in split
          // order and apply SwiGLU -- deterministic whatever the arrival order.
          const size_t pstride = 2 * static_cast<size_t>(args.n_out);
          float *P = args.part + static_cast<size_t>(t.s) * args.tk * pstride;
          if (n0 < args.n_out && warp_real) {
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
              uint32_t g[32], v[32];
              ptx::tmem_ld_32x32b_x32(tbase + cc * 32, g);
              ptx::tmem_ld_32x32b_x32(tbase + BN / 2 + cc * 32, v);
              ptx::tmem_wait_ld();
              const int col = n0 + cc * 32;
              if (real) {
                float *pg = P + static_cast<size_t>(ru) * pstride + col;
                float *pv = pg + args.n_out;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (col + 4 * j < args.n_out) {
                    __stcg(reinterpret_cast<float4 *>(pg + 4 * j),
                           make_float4(__uint_as_float(g[4 * j]), __uint_as_float(g[4 * j + 1]),
                                       __uint_as_float(g[4 * j + 2]), __uint_as_float(g[4 * j + 3])));
                    __stcg(reinterpret_cast<float4 *>(pv + 4 * j),
                           make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                       __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
                  }
              }
            }
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_cluster(acc ? tempty_at1 : tempty_at0);
          if (n0 < args.n_out && warp_real) {
            // One arrival counter per (m-tile, n-tile, lane quarter): each
            // epilogue warp completes its own 32 rows, with no cross-warp wait.
            int *cnt = args.tile_cnt + (static_cast<size_t>(row / BM) * NT + t.nt) * 4 + q;
            __syncwarp();  // the warp's partial stores precede its arrival
            int last = 0;
            if (lane == 0) {
              __threadfence();
              last = atomicAdd(cnt, 1) == S - 1 ? 1 : 0;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
              __threadfence();  // the other splits' partials are visible to every lane
              // The warp completes its real rows four at a time, lane l taking
              // columns [4l, 4l + 4) of the tile's 128, so the partial loads
              // are coalesced and those of four rows are in flight together.
              // Each sum runs over the splits in order.  e4m3 operands: the
              // sums are scaled by the A row's and the B columns' scales, and
              // the row's max |bf16 H| over the tile goes to habs.
              const int col = n0 + 4 * lane;
              const size_t sstride = static_cast<size_t>(args.tk) * pstride;
              float4 c1 = make_float4(1.f, 1.f, 1.f, 1.f), c3 = c1;
              if (FP8) {
                const float *b1 = args.col_scale0 + static_cast<size_t>(t.e) * args.n_out;
                const float *b3 = args.col_scale1 + static_cast<size_t>(t.e) * args.n_out;
                if (col < args.n_out) {
                  c1 = make_float4(b1[col], b1[col + 1], b1[col + 2], b1[col + 3]);
                  c3 = make_float4(b3[col], b3[col + 1], b3[col + 2], b3[col + 3]);
                }
              }
              unsigned m = __ballot_sync(0xffffffffu, real);
              while (m) {
                int src[4];
                float hm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  src[j] = m ? __ffs(m) - 1 : -1;
                  m &= m - 1;
                }
                if (col < args.n_out) {
                  const float *pg[4];
                  float4 a[4], b[4];
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    pg[j] = args.part + static_cast<size_t>(ru - lane + (src[j] < 0 ? lane : src[j])) * pstride + col;
                    a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    b[j] = a[j];
                  }
#pragma unroll 2
                  for (int sp = 0; sp < S; ++sp) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                      if (src[j] < 0) continue;
                      const float4 ga = __ldcg(reinterpret_cast<const float4 *>(pg[j] + sp * sstride));
                      const float4 gb = __ldcg(reinterpret_cast<const float4 *>(pg[j] + sp * sstride + args.n_out));
                      a[j].x += ga.x; a[j].y += ga.y; a[j].z += ga.z; a[j].w += ga.w;
                      b[j].x += gb.x; b[j].y += gb.y; b[j].z += gb.z; b[j].w += gb.w;
                    }
                  }
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    if (src[j] < 0) continue;
                    if (FP8) {
                      const float rsj = args.row_scale[row - lane + src[j]];
                      a[j].x *= rsj * c1.x; a[j].y *= rsj * c1.y; a[j].z *= rsj * c1.z; a[j].w *= rsj * c1.w;
                      b[j].x *= rsj * c3.x; b[j].y *= rsj * c3.y; b[j].z *= rsj * c3.z; b[j].w *= rsj * c3.w;
                    }
                    __nv_bfloat162 h01 = __floats2bfloat162_rn(silu_f(a[j].x) * b[j].x, silu_f(a[j].y) * b[j].y);
                    __nv_bfloat162 h23 = __floats2bfloat162_rn(silu_f(a[j].z) * b[j].z, silu_f(a[j].w) * b[j].w);
                    uint2 packed;
                    packed.x = *reinterpret_cast<uint32_t *>(&h01);
                    packed.y = *reinterpret_cast<uint32_t *>(&h23);
                    __nv_bfloat16 *H = static_cast<__nv_bfloat16 *>(args.out) +
                                       static_cast<size_t>(row - lane + src[j]) * args.n_out + col;
                    *reinterpret_cast<uint2 *>(H) = packed;
                    if (FP8) {
                      const float2 p = __bfloat1622float2(h01), q2 = __bfloat1622float2(h23);
                      hm[j] = fmaxf(fmaxf(fabsf(p.x), fabsf(p.y)), fmaxf(fabsf(q2.x), fabsf(q2.y)));
                    }
                  }
                }
                if (FP8) {
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    float m = hm[j];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if (lane == 0 && src[j] >= 0)
                      args.habs[static_cast<size_t>(row - lane + src[j]) * NT + t.nt] = m;
                  }
                }
              }
            }
          }
        }
      } else {
        // gate-scaled rows into the compact output; padding rows are dropped
        float *O = static_cast<float *>(args.out) + static_cast<size_t>(t.s) * args.out_split_stride;
        // e4m3 operands: the gate times the H row's scale; the W2 column scale below
        const float gsc = real ? args.perm_gate[row] * (FP8 ? args.row_scale[row] : 1.f) : 0.f;
        const int n0 = t.nt * BN;
        // A chunk of 32 accumulator columns of this thread's row: TMEM load
        // (warp-collective), the tail split's first half, the e4m3 column
        // scales.  The row's output is this times gsc.
        auto chunk = [&](int cc, uint32_t(&v)[32]) {
          ptx::tmem_ld_32x32b_x32(tbase + cc * 32, v);
          ptx::tmem_wait_ld();
          add_part(v, cc * 32);
          const int col = n0 + cc * 32;
          if (FP8) {
            const float *cs2 = args.col_scale0 + static_cast<size_t>(t.e) * args.n_out;
            // the chunk's 32 column scales, addresses clamped into range so
            // that all eight loads are in flight together
            float4 s4s[8];
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4)
              s4s[j4] = __ldg(reinterpret_cast<const float4 *>(cs2 + min(col + 4 * j4, args.n_out - 4)));
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 s4 = col + 4 * j4 < args.n_out ? s4s[j4] : make_float4(0, 0, 0, 0);
              v[4 * j4] = __float_as_uint(__uint_as_float(v[4 * j4]) * s4.x);
              v[4 * j4 + 1] = __float_as_uint(__uint_as_float(v[4 * j4 + 1]) * s4.y);
              v[4 * j4 + 2] = __float_as_uint(__uint_as_float(v[4 * j4 + 2]) * s4.z);
              v[4 * j4 + 3] = __float_as_uint(__uint_as_float(v[4 * j4 + 3]) * s4.w);
            }
          }
        };
        // Fused combine of an unsplit down GEMM: every real row counts its
        // arrival on its token's n-tile counter (low 16 bits) before storing
        // anything, so the slot row that arrives last knows it and keeps its
        // sums out of O (unless keep_o).  The other rows store theirs and then signal (high
        // 16 bits).  Once all of the warp's stores and signals are out, its
        // last rows wait (bounded) for the other slot's signal, take their own
        // sums from TMEM again, add the other slot's row and store y.  A warp
        // signals before it waits on anything, so no two warps wait on each
        // other; and two fp32 addends sum the same in either order, so y is
        // the combine kernel's bit for bit.
        const bool fused1 = args.y != nullptr && S == 1 && n0 < args.n_out;
        int tok = -1, other = -1;
        bool last = false;
        int *cnt = nullptr;
        if (fused1 && real) {
          tok = args.perm_tok[row];
          if (tok < 0 || tok >= args.T) {
            atomicCAS(args.status, 0, MOE_ERR_DEVICE_BOUNDS);
            tok = -1;
          } else {
            cnt = args.tok_cnt + static_cast<size_t>(tok) * NT + t.nt;
            last = (atomicAdd(cnt, 1) & 0xffff) == args.K - 1;
            if (last && args.K > 1) {
              const int p0 = args.pos[tok * args.K], p1 = args.pos[tok * args.K + 1];
              if (p0 < 0 || p0 >= args.tk || p1 < 0 || p1 >= args.tk || (p0 != ru && p1 != ru))
                atomicCAS(args.status, 0, MOE_ERR_DEVICE_BOUNDS);
              else
                other = p0 == ru ? p1 : p0;
            }
          }
        }
        if (n0 < args.n_out && warp_real) {
#pragma unroll 1
          for (int cc = 0; cc < BN / 32; ++cc) {
            uint32_t v[32];
            chunk(cc, v);
            const int col = n0 + cc * 32;
            if (real && (!last || args.keep_o)) {
              float *dst = O + static_cast<size_t>(ru) * args.n_out + col;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (col + 4 * j < args.n_out)
                  *reinterpret_cast<float4 *>(dst + 4 * j) =
                      make_float4(__uint_as_float(v[4 * j]) * gsc, __uint_as_float(v[4 * j + 1]) * gsc,
                                  __uint_as_float(v[4 * j + 2]) * gsc, __uint_as_float(v[4 * j + 3]) * gsc);
            }
          }
        }
        if (cnt != nullptr && !last) {
          __threadfence();  // this row's O stores precede its signal
          atomicAdd(cnt, 0x10000);
        }
        if (fused1 && __ballot_sync(0xffffffffu, last) != 0) {
          bool ok = last && (args.K == 1 || (other >= 0 && wait_signals(cnt, args.K - 1, args.status)));
          __threadfence();  // the other slot's O row is visible once its signal is
          const float *orow = ok && other >= 0 ? O + static_cast<size_t>(other) * args.n_out : nullptr;
#pragma unroll 1
          for (int cc = 0; cc < BN / 32; ++cc) {
            uint32_t v[32];
            chunk(cc, v);
            const int col = n0 + cc * 32;
            if (!ok) continue;
            float4 o4[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              o4[j] = orow != nullptr && col + 4 * j < args.n_out
                          ? __ldcg(reinterpret_cast<const float4 *>(orow + col + 4 * j))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
            __nv_bfloat16 *yrow = args.y + static_cast<size_t>(tok) * args.n_out + col;
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8) {
              if (col + 8 * j8 >= args.n_out) continue;  // n_out is a multiple of 8
              float f[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float own = __uint_as_float(v[8 * j8 + i]) * gsc;
                const float4 &o = o4[2 * j8 + (i >> 2)];
                const float oth = (i & 3) == 0 ? o.x : (i & 3) == 1 ? o.y : (i & 3) == 2 ? o.z : o.w;
                f[i] = orow != nullptr ? own + oth : own;
              }
              uint4 *yp = reinterpret_cast<uint4 *>(yrow + 8 * j8);
              if (args.y_accumulate) {
                const uint4 old = *yp;
                const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ow[i]));
                  f[2 * i] = f2.x + f[2 * i];
                  f[2 * i + 1] = f2.y + f[2 * i + 1];
                }
              }
              uint32_t yw[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
                yw[i] = *reinterpret_cast<const uint32_t *>(&h);
              }
              *yp = make_uint4(yw[0], yw[1], yw[2], yw[3]);
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(acc ? tempty_at1 : tempty_at0);
        if (args.y != nullptr && S > 1 && n0 < args.n_out) {
          // Fused combine of a split down GEMM: the writer that completes this
          // token's 256 columns last (of its K slot rows times S splits) adds them -- per slot the
          // splits in order, then the slots in order: the combine kernel's
          // order, so y is the same bit for bit -- and stores y.  The warp
          // finishes its rows that arrived last together, four at a time,
          // lane l taking columns [8l, 8l + 8) of each.
          int tok = -1, last = 0;
          if (real) {
            __threadfence();  // this row's O stores precede the arrival
            tok = args.perm_tok[row];
            if (tok < 0 || tok >= args.T) {
              atomicCAS(args.status, 0, MOE_ERR_DEVICE_BOUNDS);
            } else {
              last = atomicAdd(args.tok_cnt + static_cast<size_t>(tok) * NT + t.nt, 1) == args.K * S - 1;
            }
          }
          unsigned m = __ballot_sync(0xffffffffu, last);
          if (m) __threadfence();  // the other slots' stores are visible to every lane
          const int c8 = 8 * lane;
          const bool col_in = c8 < args.n_out - n0;  // n_out is a multiple of 8
          static_assert(kMaxK == 2, "the fused combine adds at most two slot rows");
          while (m) {
            int tk[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int src = m ? __ffs(m) - 1 : -1;
              m &= m ? m - 1 : 0u;
              tk[q] = __shfl_sync(0xffffffffu, tok, src < 0 ? 0 : src);
              if (src < 0) tk[q] = -1;
            }
            float4 a[4][2], b[4][2];
            bool ok[4];
            // split 0 of the slot outputs (this unit wrote split t.s)
            const float *O0 = static_cast<const float *>(args.out);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              ok[q] = false;
              if (tk[q] < 0) continue;
              const int p0 = args.pos[tk[q] * args.K];
              const int p1 = args.K > 1 ? args.pos[tk[q] * args.K + 1] : 0;
              ok[q] = p0 >= 0 && p0 < args.tk && p1 >= 0 && p1 < args.tk;
              if (!ok[q] || !col_in) continue;
              const float *s0 = O0 + static_cast<size_t>(p0) * args.n_out + n0 + c8;
              const float *s1 = O0 + static_cast<size_t>(p1) * args.n_out + n0 + c8;
              a[q][0] = __ldcg(reinterpret_cast<const float4 *>(s0));
              a[q][1] = __ldcg(reinterpret_cast<const float4 *>(s0 + 4));
              if (args.K > 1) {
                b[q][0] = __ldcg(reinterpret_cast<const float4 *>(s1));
                b[q][1] = __ldcg(reinterpret_cast<const float4 *>(s1 + 4));
              }
              // the other splits of each slot, added in split order
              for (int sp = 1; sp < S; ++sp) {
                const float *r0 = s0 + static_cast<size_t>(sp) * args.out_split_stride;
                const float4 x0 = __ldcg(reinterpret_cast<const float4 *>(r0));
                const float4 x1 = __ldcg(reinterpret_cast<const float4 *>(r0 + 4));
                a[q][0].x += x0.x; a[q][0].y += x0.y; a[q][0].z += x0.z; a[q][0].w += x0.w;
                a[q][1].x += x1.x; a[q][1].y += x1.y; a[q][1].z += x1.z; a[q][1].w += x1.w;
                if (args.K > 1) {
                  const float *r1 = s1 + static_cast<size_t>(sp) * args.out_split_stride;
                  const float4 z0 = __ldcg(reinterpret_cast<const float4 *>(r1));
                  const float4 z1 = __ldcg(reinterpret_cast<const float4 *>(r1 + 4));
                  b[q][0].x += z0.x; b[q][0].y += z0.y; b[q][0].z += z0.z; b[q][0].w += z0.w;
                  b[q][1].x += z1.x; b[q][1].y += z1.y; b[q][1].z += z1.z; b[q][1].w += z1.w;
                }
              }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (tk[q] < 0) continue;
              if (!ok[q]) {
                if (lane == 0) atomicCAS(args.status, 0, MOE_ERR_DEVICE_BOUNDS);
                continue;
              }
              if (!col_in) continue;
              float v[8] = {a[q][0].x, a[q][0].y, a[q][0].z, a[q][0].w, a[q][1].x, a[q][1].y, a[q][1].z, a[q][1].w};
              if (args.K > 1) {
                const float w[8] = {b[q][0].x, b[q][0].y, b[q][0].z, b[q][0].w,
                                    b[q][1].x, b[q][1].y, b[q][1].z, b[q][1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] += w[i];
              }
              uint4 *yp = reinterpret_cast<uint4 *>(args.y + static_cast<size_t>(tk[q]) * args.n_out + n0 + c8);
              if (args.y_accumulate) {
                const uint4 o = *yp;
                const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ow[i]));
                  v[2 * i] = f2.x + v[2 * i];
                  v[2 * i + 1] = f2.y + v[2 * i + 1];
                }
              }
              uint32_t yw[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                yw[i] = *reinterpret_cast<const uint32_t *>(&h);
              }
              *yp = make_uint4(yw[0], yw[1], yw[2], yw[3]);
            }
          }
        }
      }
      ++local;
    }
  }

  // Producer tail: every stage's last release has arrived, so no commit can
  // still land in this CTA's barriers.  (After an abort some releases never
  // come; the drain below covers that case.)
  if (warp == 0 && lane == 0 && !*reinterpret_cast<volatile int *>(&c.abort)) {
    for (int i = 0; i < STAGES; ++i) {
      wait_bounded(&c.empty[p_stage], p_phase ^ 1u, c, args.status, false);
      if (++p_stage == STAGES) { p_stage = 0; p_phase ^= 1u; }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (*reinterpret_cast<volatile int *>(&c.abort)) {
    // Some role gave up: before TMEM and shared memory are released, wait
    // (bounded) for the MMAs this CTA issued and for every copy completing on
    // its barriers.
    if (warp == 1 && lane == 0 && leader) {
      if (PAIR) ptx::mma_commit_pair(&c.drain);
      else ptx::mma_commit(&c.drain);
      wait_bounded(&c.drain, 0, c, args.status, false);
    }
    if (warp == 0 && lane == 0 && leader) {
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) wait_bounded(&c.full[s], (last_par >> s) & 1u, c, args.status, false);
    }
    if (PAIR && warp == 0 && lane == 0) {
      // Pair MMA: a CTA's copies complete on its partner's barriers, which
      // cannot tell this CTA when they have landed; copies take microseconds,
      // so give any still in flight 50 us before shared memory is released.
      const uint64_t t0 = ptx::globaltimer_ns();
      while (ptx::globaltimer_ns() - t0 < 50000ull) {
      }
    }
    ptx::tc_fence_before();
    __syncthreads();
  }
  // No CTA leaves while another CTA of the cluster may still send it copies
  // or arrivals.
  if (threadIdx.x == 0) {
    for (int r2 = 0; r2 < CL; ++r2)
      if (r2 != rank) ptx::mbar_arrive_remote(&c.exit_bar, static_cast<uint32_t>(r2));
    wait_bounded(&c.exit_bar, 0, c, args.status, false);
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (PAIR) ptx::tmem_dealloc_pair(tmem, TMEM_COLS);  // with the peer CTA's warp 1
    else ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
  if (args.stamps != nullptr && threadIdx.x == 0) atomicMax(args.stamps + kNumStages + kStage, stamp_now());
}

// ---------------------------------------------------------------- host side
// Per device: shared-memory attribute set, and how many 2-CTA clusters of
// this kernel can be resident at once (the persistent grid size).
struct DevState {
  bool ready = false;
  int clusters = 0;
};

template <int MODE, int FORM, bool FP8>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(expert_gemm_kernel<MODE, FORM, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Ring<FormInfo<FORM>::PAIR>::SMEM);
}

template <int FORM>
cudaError_t max_clusters(int num_sms, int *n) {
  constexpr int CL = FormInfo<FORM>::CL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((num_sms / CL) * CL);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = Ring<FormInfo<FORM>::PAIR>::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, expert_gemm_kernel<MODE_GATE_UP, FORM, false>, &cfg);
}

template <int MODE>
cudaError_t set_attrs_mode() {
  cudaError_t err = set_smem_attr<MODE, FORM_MC2, false>();
  if (err == cudaSuccess) err = set_smem_attr<MODE, FORM_PAIR, false>();
  if (err == cudaSuccess) err = set_smem_attr<MODE, FORM_MC4, false>();
  if (err == cudaSuccess) err = set_smem_attr<MODE, FORM_MC2, true>();
  if (err == cudaSuccess) err = set_smem_attr<MODE, FORM_PAIR, true>();
  if (err == cudaSuccess) err = set_smem_attr<MODE, FORM_MC4, true>();
  return err;
}

// Persistent grid sizes: co-resident 2-CTA clusters (pair forms) and 4-CTA
// clusters (2x2 form).
struct Grids {
  int clusters2 = 0, clusters4 = 0;
};

cudaError_t device_state(int num_sms, Grids *g) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static std::mutex mu;
  static DevState st[64];
  static Grids grids[64];
  std::lock_guard<std::mutex> lock(mu);
  if (!st[dev].ready) {
    err = set_attrs_mode<MODE_GATE_UP>();
    if (err == cudaSuccess) err = set_attrs_mode<MODE_DOWN>();
    if (err != cudaSuccess) return err;
    int n0 = 0, n1 = 0, n4 = 0;
    err = max_clusters<FORM_MC2>(num_sms, &n0);
    if (err == cudaSuccess) err = max_clusters<FORM_PAIR>(num_sms, &n1);
    if (err == cudaSuccess) err = max_clusters<FORM_MC4>(num_sms, &n4);
    if (err != cudaSuccess) return err;
    const int n = n0 < n1 ? n0 : n1;  // one persistent grid size for both 2-CTA forms
    if (n < 1) return cudaErrorInvalidConfiguration;
    grids[dev].clusters2 = n;
    grids[dev].clusters4 = n4;  // 0 if 4-CTA clusters cannot be resident: that form is not used
    st[dev].clusters = n;
    st[dev].ready = true;
  }
  *g = grids[dev];
  return cudaSuccess;
}

template <int MODE, int FORM, bool FP8>
cudaError_t launch_gemm(const Grids &g, cudaStream_t s, bool pdl, const CUtensorMap &a, const CUtensorMap &ah,
                        const CUtensorMap &aq, const CUtensorMap &b0, const CUtensorMap &b1, const GemmArgs &args) {
  constexpr int CL = FormInfo<FORM>::CL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((FORM == FORM_MC4 ? g.clusters4 : g.clusters2) * CL);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = Ring<FormInfo<FORM>::PAIR>::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, expert_gemm_kernel<MODE, FORM, FP8>, a, ah, aq, b0, b1, args);
}

// The form a call's grouping calls for (see ws_layout), and whether the 2x2
// form can run on this device.
int pick_form(const WsLayout &L, const Grids &g) {
  if (L.form == FORM_MC4 && g.clusters4 < 1) return FORM_MC2;
  return L.form;
}

template <int MODE, bool FP8>
cudaError_t launch_form(int form, const Grids &g, cudaStream_t s, bool pdl, const CUtensorMap &a,
                        const CUtensorMap &ah, const CUtensorMap &aq, const CUtensorMap &b0, const CUtensorMap &b1,
                        const GemmArgs &args) {
  if (form == FORM_PAIR) return launch_gemm<MODE, FORM_PAIR, FP8>(g, s, pdl, a, ah, aq, b0, b1, args);
  if (form == FORM_MC4) return launch_gemm<MODE, FORM_MC4, FP8>(g, s, pdl, a, ah, aq, b0, b1, args);
  return launch_gemm<MODE, FORM_MC2, FP8>(g, s, pdl, a, ah, aq, b0, b1, args);
}

// Tail split of an unsplit GEMM in the multicast-pair form (the kernel decides
// from the routing whether the last wave is worth splitting); `which` selects
// the GEMM's own arrival counters (0 gate/up, 1 down).
void set_tail_split(GemmArgs &g, const WsLayout &L, const Ptrs &P, int form, int splits, int which) {
  g.tail_part = nullptr;
  g.tail_flag = nullptr;
  g.tail_slots = 0;
  if (form != FORM_MC2 || splits != 1 || L.tail_slots < 1) return;
  g.tail_part = P.tail_part;
  g.tail_flag = P.tail_flag + which * L.tail_slots * 2;
  g.tail_slots = L.tail_slots;
}

// The down GEMM's fused-combine arguments (y formed in its epilogue).
void set_fused_combine(GemmArgs &g, const WsLayout &L, const Ptrs &P, void *y, unsigned flags) {
  if (!L.fuse_combine) return;
  g.y = static_cast<__nv_bfloat16 *>(y);
  g.y_accumulate = (flags & MOE_ACCUMULATE) ? 1 : 0;
  g.pos = P.pos;
  g.perm_tok = P.perm_tok;
  g.tok_cnt = P.tok_cnt;
  g.T = L.T;
  g.K = L.K;
  g.keep_o = L.train ? 1 : 0;
}

}  // namespace

cudaError_t launch_expert_gemms_bf16(const void *W1, const void *W3, const void *W2, int d, int f, int E,
                                     const WsLayout &L, const Ptrs &P, void *y, unsigned flags, int num_sms,
                                     cudaStream_t s, const int *slot_of, int n_slots) {
  Grids grids;
  cudaError_t err = device_state(num_sms, &grids);
  if (err != cudaSuccess) return err;
  const int form = pick_form(L, grids);
  const int banks = slot_of ? n_slots : E;  // matrices held by each weight bank
  CUtensorMap tm_x, tm_xh, tm_xq, tm_w1, tm_w3, tm_h, tm_hh, tm_hq, tm_w2;
  // weights whose column count is a multiple of 128 go through the 4-D view:
  // one copy per 128-column half tile instead of two (2.3% per prefill layer)
  const bool w13_4d = f % 128 == 0, w2_4d = d % 128 == 0;
  if (!tmap_2d(&tm_x, P.xperm, d, L.R, BM) || !tmap_2d(&tm_xh, P.xperm, d, L.R, BM / 2) ||
      !tmap_2d(&tm_xq, P.xperm, d, L.R, BM / 4) ||
      !(w13_4d ? tmap_4d_w(&tm_w1, W1, f, d, banks) : tmap_3d(&tm_w1, W1, f, d, banks)) ||
      !(w13_4d ? tmap_4d_w(&tm_w3, W3, f, d, banks) : tmap_3d(&tm_w3, W3, f, d, banks)) ||
      !tmap_2d(&tm_h, P.hbuf, f, L.R, BM) ||
      !tmap_2d(&tm_hh, P.hbuf, f, L.R, BM / 2) || !tmap_2d(&tm_hq, P.hbuf, f, L.R, BM / 4) ||
      !(w2_4d ? tmap_4d_w(&tm_w2, W2, d, f, banks) : tmap_3d(&tm_w2, W2, d, f, banks)))
    return cudaErrorInvalidValue;

  GemmArgs g1{};
  g1.poffsets = P.poffsets;
  g1.offsets = P.offsets;
  g1.perm_gate = P.perm_gate;
  g1.out = P.hbuf;
  g1.out_split_stride = 0;
  g1.part = P.gu_part;
  g1.tile_cnt = P.tile_cnt;
  g1.E = E;
  g1.rows_bound = L.R;
  g1.tk = L.TK;
  g1.n_out = f;
  g1.num_n_tiles = (f + BN / 2 - 1) / (BN / 2);
  g1.num_kb = (d + BK - 1) / BK;
  g1.b4d = w13_4d ? 1 : 0;
  g1.splits = L.S_gu;
  g1.kb_per_split = L.kb_per_split_gu;
  g1.force_timeout = (flags & MOE_DEBUG_FORCE_TIMEOUT) ? 1 : 0;
  g1.save_ab = static_cast<__nv_bfloat16 *>(P.ab);  // training forward only (then splits == 1)
  g1.status = P.status;
  g1.use_slots = slot_of ? 1 : 0;
  for (int e = 0; e < E && slot_of; ++e) g1.wslot[e] = slot_of[e];
  g1.stamps = P.stamps;
  set_tail_split(g1, L, P, form, L.S_gu, 0);
  err = launch_form<MODE_GATE_UP, false>(form, grids, s, true, tm_x, tm_xh, tm_xq, tm_w1, tm_w3, g1);
  if (err != cudaSuccess) return err;

  GemmArgs g2 = g1;
  g2.out = P.obuf;
  g2.out_split_stride = static_cast<long long>(g1.tk) * d;
  g2.part = nullptr;
  g2.tile_cnt = nullptr;
  g2.force_timeout = 0;
  g2.save_ab = nullptr;
  set_fused_combine(g2, L, P, y, flags);
  g2.n_out = d;
  g2.num_n_tiles = (d + BN - 1) / BN;
  g2.num_kb = (f + BK - 1) / BK;
  g2.b4d = w2_4d ? 1 : 0;
  g2.splits = L.S;
  g2.kb_per_split = L.kb_per_split;
  set_tail_split(g2, L, P, form, L.S, 1);
  return launch_form<MODE_DOWN, false>(form, grids, s, true, tm_h, tm_hh, tm_hq, tm_w2, tm_w2, g2);
}

cudaError_t launch_expert_gemms_fp8(const void *W1q, const float *s1, const void *W3q, const float *s3,
                                    const void *W2q, const float *s2, int d, int f, int E, const WsLayout &L,
                                    const Ptrs &P, void *y, unsigned flags, int num_sms, cudaStream_t s) {
  Grids grids;
  cudaError_t err = device_state(num_sms, &grids);
  if (err != cudaSuccess) return err;
  const int form = pick_form(L, grids);
  // e4m3 operands: X_perm [R, d] and H [R, f] K-contiguous; the banks in
  // 128 x 128 tiles, addressed as rows of 128 codes (tile t = rows 128 t ..)
  const int nt13 = (f + kFp8Tile - 1) / kFp8Tile, kt13 = (d + kFp8Tile - 1) / kFp8Tile;
  const int nt2 = (d + kFp8Tile - 1) / kFp8Tile, kt2 = (f + kFp8Tile - 1) / kFp8Tile;
  const uint64_t rows13 = static_cast<uint64_t>(E) * nt13 * kt13 * kFp8Tile;
  const uint64_t rows2 = static_cast<uint64_t>(E) * nt2 * kt2 * kFp8Tile;
  CUtensorMap tm_x, tm_xh, tm_xq, tm_w1, tm_w3, tm_h, tm_hh, tm_hq, tm_w2;
  if (!tmap_2d_u8(&tm_x, P.xperm, d, L.R, BM) || !tmap_2d_u8(&tm_xh, P.xperm, d, L.R, BM / 2) ||
      !tmap_2d_u8(&tm_xq, P.xperm, d, L.R, BM / 4) || !tmap_2d_u8(&tm_w1, W1q, kFp8Tile, rows13, kFp8Tile) ||
      !tmap_2d_u8(&tm_w3, W3q, kFp8Tile, rows13, kFp8Tile) || !tmap_2d_u8(&tm_h, P.hq, f, L.R, BM) ||
      !tmap_2d_u8(&tm_hh, P.hq, f, L.R, BM / 2) || !tmap_2d_u8(&tm_hq, P.hq, f, L.R, BM / 4) ||
      !tmap_2d_u8(&tm_w2, W2q, kFp8Tile, rows2, kFp8Tile))
    return cudaErrorInvalidValue;

  GemmArgs g1{};
  g1.poffsets = P.poffsets;
  g1.offsets = P.offsets;
  g1.perm_gate = P.perm_gate;
  g1.out = P.hbuf;
  g1.E = E;
  g1.rows_bound = L.R;
  g1.tk = L.TK;
  g1.n_out = f;
  g1.num_n_tiles = (f + BN / 2 - 1) / (BN / 2);
  g1.num_kb = (d + 127) / 128;
  g1.splits = L.S_gu;
  g1.kb_per_split = L.kb_per_split_gu;
  g1.part = P.gu_part;
  g1.tile_cnt = P.tile_cnt;
  g1.force_timeout = (flags & MOE_DEBUG_FORCE_TIMEOUT) ? 1 : 0;
  g1.row_scale = P.xscale;
  g1.col_scale0 = s1;
  g1.col_scale1 = s3;
  g1.habs = P.habs;
  g1.b_nt = nt13;
  g1.b_kt = kt13;
  g1.status = P.status;
  g1.stamps = P.stamps;
  set_tail_split(g1, L, P, form, L.S_gu, 0);
  err = launch_form<MODE_GATE_UP, true>(form, grids, s, true, tm_x, tm_xh, tm_xq, tm_w1, tm_w3, g1);
  // H rows to e4m3 with their own scales
  if (err == cudaSuccess) err = launch_quant_h(f, E, L.T * L.K, g1.num_n_tiles, P, num_sms, s);
  if (err != cudaSuccess) return err;

  GemmArgs g2 = g1;
  g2.out = P.obuf;
  g2.out_split_stride = static_cast<long long>(L.TK) * d;
  g2.part = nullptr;
  g2.tile_cnt = nullptr;
  set_fused_combine(g2, L, P, y, flags);
  g2.n_out = d;
  g2.num_n_tiles = (d + BN - 1) / BN;
  g2.num_kb = (f + 127) / 128;
  g2.splits = L.S;
  g2.kb_per_split = L.kb_per_split;
  g2.force_timeout = 0;
  g2.row_scale = P.hscale;
  g2.col_scale0 = s2;
  g2.col_scale1 = nullptr;
  g2.habs = nullptr;
  g2.b_nt = nt2;
  g2.b_kt = kt2;
  set_tail_split(g2, L, P, form, L.S, 1);
  return launch_form<MODE_DOWN, true>(form, grids, s, true, tm_h, tm_hh, tm_hq, tm_w2, tm_w2, g2);
}

}  // namespace moe
