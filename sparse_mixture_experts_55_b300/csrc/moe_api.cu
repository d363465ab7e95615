// moe_api.cu -- the C ABI declared in include/moe.h: argument validation,
// workspace layout, and the enqueue sequence of one MoE forward pass
//   router -> grouping -> row gather -> gate/up GEMM (+SwiGLU)
//   -> down GEMM (x gate) -> two-slot combine
// (section 3.4 "MoE Layer Formulation" of the Mixtral of Experts summary:
// y = sum_i G(x)_i E_i(x), with only the selected experts computing).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace moe {

namespace {

struct DevInfo {
  bool ready = false;
  int sms = 0, major = 0, minor = 0;
};

// Cached per-device attributes: the library's only global state.
bool device_info(DevInfo &out) {
  static std::mutex mu;
  static DevInfo table[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  DevInfo &di = table[dev];
  if (!di.ready) {
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return false;
    di.ready = true;
  }
  out = di;
  return true;
}

constexpr int kDefaultSms = 148;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

constexpr unsigned kFormFlags = MOE_GEMM_PAIR_MMA | MOE_GEMM_QUAD | MOE_GEMM_MULTICAST_PAIRS;

// At most one form flag; returns false for a combination.
bool form_flags_ok(unsigned flags) {
  const unsigned f = flags & kFormFlags;
  return (f & (f - 1)) == 0;
}

// The layout's GEMM form, overridden by a form flag unless the gate/up
// contraction is split.
void apply_form_flags(WsLayout &L, unsigned flags) {
  if (L.S_gu != 1) return;
  if (flags & MOE_GEMM_PAIR_MMA) L.form = 1;
  if (flags & MOE_GEMM_QUAD) L.form = 2;
  if (flags & MOE_GEMM_MULTICAST_PAIRS) L.form = 0;
}

// bytes per element of the tokens x, y (the e4m3 variant keeps them bf16)
int elem_bytes(int dtype) { return dtype == MOE_F32 ? 4 : 2; }

// Shape checks shared by every entry point.  Returns MOE_OK or an error code.
int check_shape(int T, int d, int f, int E, int K, int dtype) {
  if (dtype != MOE_BF16 && dtype != MOE_F32 && dtype != MOE_FP8_E4M3) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || d < 1 || f < 1 || E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (K > E) return MOE_ERR_INVALID_ARG;
  if (K > kMaxK || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  // 16-byte rows for vector loads and TMA strides (one-byte codes for e4m3)
  const int mult = dtype == MOE_BF16 ? 8 : dtype == MOE_F32 ? 4 : 16;
  if (d % mult != 0 || f % mult != 0) return MOE_ERR_INVALID_ARG;
  // index arithmetic of the grouped buffers stays in 32-bit rows
  const long long rows = static_cast<long long>(T) * K + static_cast<long long>(E) * kSegPad;
  if (rows >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}


bool stamps_ok(const unsigned long long *stamps) {
  return stamps != nullptr && (reinterpret_cast<uintptr_t>(stamps) & 7u) == 0;
}

}  // namespace

int sm_count_or_default() {
  DevInfo di;
  return device_info(di) ? di.sms : kDefaultSms;
}

int check_device() {
  DevInfo di;
  if (!device_info(di)) return MOE_ERR_CUDA;
  // The kernels are built for sm_103a only.
  if (di.major != 10 || di.minor != 3) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

SplitPlan plan_splits(long long TK, int E, int n_tiles, int kb, int clusters, double part_ratio) {
  SplitPlan best{1, kb};
  if (TK <= 0 || kb <= 1 || clusters <= 0) return best;
  const long long touched = TK < E ? TK : E;
  const long long rows_per = (TK + touched - 1) / touched;
  const long long mt = (rows_per + kSegPad - 1) / kSegPad;  // m-tiles per touched expert
  // cluster units per split: pairs of m-tiles sharing the weight tile, and
  // for an odd m-tile count, pairs of n-tiles sharing the activation tile
  const long long per_split = touched * ((mt >> 1) * n_tiles + (mt & 1) * ((n_tiles + 1) / 2));
  constexpr double kUnitOverheadKb = 0.5;
  auto cost = [&](int S, int kps) {
    const long long waves = (per_split * S + clusters - 1) / clusters;
    return static_cast<double>(waves) * (kps + kUnitOverheadKb) * (1.0 + part_ratio * (S > 1 ? S : 0));
  };
  const double base = cost(1, kb);
  double best_cost = base;
  for (int s = 2; s <= 32 && s <= kb; ++s) {
    const int kps = (kb + s - 1) / s;
    const int S = (kb + kps - 1) / kps;  // every split owns >= 1 k-block
    const double c = cost(S, kps);
    if (c < best_cost) {
      best_cost = c;
      best = SplitPlan{S, kps};
    }
  }
  if (best_cost > 0.97 * base) best = SplitPlan{1, kb};
  return best;
}

WsLayout ws_layout(int T, int d, int f, int E, int K, int dtype, int num_sms, bool train, bool routing_only) {
  WsLayout L{};
  L.train = train;
  const size_t eb = elem_bytes(dtype);
  L.R = static_cast<int>(align_up(static_cast<size_t>(T) * K + static_cast<size_t>(E) * (kSegPad - 1), kSegPad));
  {
    // about one wave of router blocks: ceil(T / SMs) tokens each, in groups of kRouteGroup
    const int per = (T + num_sms - 1) / (num_sms > 0 ? num_sms : 1);
    L.route_tpb = ((per > 0 ? per : 1) + kRouteGroup - 1) / kRouteGroup * kRouteGroup;
    L.route_single = T <= kSingleRouteT;
    if (L.route_single) L.route_tpb = T > 0 ? (T + kRouteGroup - 1) / kRouteGroup * kRouteGroup : kRouteGroup;
    L.n_route_blocks = (T + L.route_tpb - 1) / L.route_tpb;
  }
  const long long TKl = static_cast<long long>(T) * K;
  L.T = T;
  L.K = K;
  L.TK = static_cast<int>(TKl);
  const long long touched = TKl < E ? TKl : E;
  const bool fp8 = dtype == MOE_FP8_E4M3;
  const int kbw = fp8 ? 128 : 64;  // contraction elements per 128-byte k-block
  SplitPlan down{1, (f + kbw - 1) / kbw}, gu{1, (d + kbw - 1) / kbw};
  if (dtype != MOE_F32 && touched > 0) {
    const int clusters = num_sms / 2;
    const double wb = fp8 ? 1.0 : 2.0;  // weight bytes per element
    // partial-sum bytes (written once, read once, fp32) per split over the
    // weight bytes each projection streams
    down = plan_splits(TKl, E, (d + 255) / 256, (f + kbw - 1) / kbw, clusters,
                       8.0 / wb * static_cast<double>(TKl) / (static_cast<double>(touched) * f));
    // The split gate/up tile is completed inside the GEMM by the last split's
    // epilogue warp, whose latency grows with the real rows it owns; beyond
    // about four rows per expert it stalls the MMA pipeline more than the
    // balanced split saves, so larger batches keep one split.
    if (TKl <= 4 * touched && !train)  // the training forward saves a, b from the unsplit epilogue
      gu = plan_splits(TKl, E, (f + 127) / 128, (d + kbw - 1) / kbw, clusters,
                       8.0 / wb * static_cast<double>(TKl) / (static_cast<double>(touched) * d));
  }
  L.S = down.S;
  L.kb_per_split = down.kb_per_split;
  L.S_gu = gu.S;
  L.kb_per_split_gu = gu.kb_per_split;
  // Expert GEMM form (gemm_tc.cu): CTA-pair MMAs once experts average 16 or
  // more 128-row tiles (the phantom half-tile of an odd count then costs at
  // most ~3%), multicast pairs otherwise.  Measured on B300 under the power
  // cap: pairs are ~1% faster at 16+ tiles per expert and ~1% slower at 8;
  // the 2x2 form is 3% slower at both.  With e4m3 weights a k-block carries
  // twice the MMA work per byte, so the pair form's deeper ring (6 stages of
  // 32 KiB fetched per SM against 4) pays from 8 tiles per expert: at the
  // Mixtral prefill shape it measured 3.3% faster per layer at full clocks
  // (1.281 against 1.324 ms), while bf16 tied.
  const long long pair_tiles = dtype == MOE_FP8_E4M3 ? 8 : 16;
  L.form = (dtype != MOE_F32 && touched > 0 && TKl >= pair_tiles * kSegPad * touched && L.S_gu == 1) ? 1 : 0;
  const size_t TK = static_cast<size_t>(T) * K;
  const size_t R = static_cast<size_t>(L.R);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.status = take(kStatusInts * sizeof(int));
  // one arrival counter per (128-row m-tile, n-tile, 32-row quarter) of the split gate/up GEMM
  const size_t n_cnt = L.S_gu > 1 ? (R / kSegPad) * static_cast<size_t>((f + 127) / 128) * 4 : 0;
  L.tile_cnt = take(n_cnt * sizeof(int));
  // fused combine: one slot-arrival counter per (token, 256-column tile of y)
  // (a split down projection for the smallest batches too: the last of a
  // token's K*S writers reads at most 2 * kFuseSplitT * S rows per tile, and
  // a separate combine launch would cost more)
  L.fuse_combine = dtype != MOE_F32 && (L.S == 1 || T <= kFuseSplitT) && !routing_only;
  L.tok_cnt = take(L.fuse_combine ? static_cast<size_t>(T) * ((d + 255) / 256) * sizeof(int) : 0);
  // tail split of an unsplit expert GEMM (gemm_tc.cu): at most one split
  // tile per two 2-CTA clusters, i.e. num_sms / 4, each for both CTAs
  const bool tail = dtype != MOE_F32 && !routing_only && (L.S == 1 || L.S_gu == 1) && touched > 0;
  L.tail_slots = tail ? (num_sms > 0 ? num_sms : 1) / 4 + 1 : 0;
  L.tail_flag = take(static_cast<size_t>(L.tail_slots) * 2 * 2 * sizeof(int));
  L.zero_bytes = o - L.status;
  L.idx = take(TK * 4);
  L.gate = take(TK * 4);
  L.blockcounts = take(static_cast<size_t>(L.n_route_blocks > 0 ? L.n_route_blocks : 1) * E * 4);
  L.offsets = take((E + 1) * 4);
  L.poffsets = take((E + 1) * 4);
  L.pos = take(TK * 4);
  L.perm_tok = take(R * 4);
  L.perm_gate = take(R * 4);
  L.xperm = take(R * d * (fp8 ? 1 : eb));
  L.hbuf = take(R * f * eb);
  L.obuf = take(static_cast<size_t>(L.S) * TK * d * 4);
  L.gu_part = take(L.S_gu > 1 ? static_cast<size_t>(L.S_gu) * TK * 2 * f * 4 : 0);
  L.xnorm = take(static_cast<size_t>(T) * d * eb);
  const size_t nt_gu = (f + 127) / 128;
  L.xscale = take(fp8 ? R * 4 : 0);
  L.habs = take(fp8 ? R * nt_gu * 4 : 0);
  L.hq = take(fp8 ? R * f : 0);
  L.hscale = take(fp8 ? R * 4 : 0);
  // training: saved pre-activations, then the backward's buffers; the router
  // weight gradient is summed over token chunks (about four blocks per SM)
  const size_t tr = train ? 1 : 0;
  L.dwg_chunks = 1;
  if (train) {
    const int col_blocks = (d / 2 + 127) / 128;
    int ch = (4 * num_sms + col_blocks - 1) / col_blocks;
    const int max_ch = (T + 63) / 64;
    if (ch > max_ch) ch = max_ch;
    L.dwg_chunks = ch > 0 ? ch : 1;
  }
  L.ab = take(tr * R * 2 * f * 2);
  L.dye = take(tr * R * d * 2);
  L.dab = take(tr * R * 2 * f * 2);
  L.dxc = take(tr * TK * d * 4);
  L.dl = take(tr * static_cast<size_t>(T) * E * 4);
  L.dwg_part = take(tr * static_cast<size_t>(L.dwg_chunks) * d * E * 4);
  L.tail_part = take(static_cast<size_t>(L.tail_slots) * 2 * 128 * 256 * sizeof(float));
  L.total = o;
  return L;
}

Ptrs carve(void *ws, const WsLayout &L) {
  char *b = static_cast<char *>(ws);
  Ptrs P;
  P.status = reinterpret_cast<int *>(b + L.status);
  P.tile_cnt = reinterpret_cast<int *>(b + L.tile_cnt);
  P.tok_cnt = reinterpret_cast<int *>(b + L.tok_cnt);
  P.tail_flag = reinterpret_cast<int *>(b + L.tail_flag);
  P.tail_part = reinterpret_cast<float *>(b + L.tail_part);
  P.idx = reinterpret_cast<int32_t *>(b + L.idx);
  P.gate = reinterpret_cast<float *>(b + L.gate);
  P.blockcounts = reinterpret_cast<int32_t *>(b + L.blockcounts);
  P.offsets = reinterpret_cast<int32_t *>(b + L.offsets);
  P.poffsets = reinterpret_cast<int32_t *>(b + L.poffsets);
  P.pos = reinterpret_cast<int32_t *>(b + L.pos);
  P.perm_tok = reinterpret_cast<int32_t *>(b + L.perm_tok);
  P.perm_gate = reinterpret_cast<float *>(b + L.perm_gate);
  P.xperm = b + L.xperm;
  P.hbuf = b + L.hbuf;
  P.obuf = reinterpret_cast<float *>(b + L.obuf);
  P.gu_part = reinterpret_cast<float *>(b + L.gu_part);
  P.xnorm = b + L.xnorm;
  P.xscale = reinterpret_cast<float *>(b + L.xscale);
  P.habs = reinterpret_cast<float *>(b + L.habs);
  P.hq = b + L.hq;
  P.hscale = reinterpret_cast<float *>(b + L.hscale);
  P.ab = L.train ? b + L.ab : nullptr;  // non-null switches the gate/up epilogue to saving
  P.dye = L.train ? b + L.dye : nullptr;
  P.dab = L.train ? b + L.dab : nullptr;
  P.dxc = L.train ? reinterpret_cast<float *>(b + L.dxc) : nullptr;
  P.dl = L.train ? reinterpret_cast<float *>(b + L.dl) : nullptr;
  P.dwg_part = L.train ? reinterpret_cast<float *>(b + L.dwg_part) : nullptr;
  P.stamps = nullptr;
  return P;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(int T, int d, int f, int E, int K, int dtype) {
  if (check_shape(T, d, f, E, K, dtype) != MOE_OK) return 0;
  return ws_layout(T, d, f, E, K, dtype, sm_count_or_default()).total;
}

// The training path (moe_forward_train / moe_backward) covers the bf16 layer
// with d and f multiples of 64 (whole k-blocks in every backward product).
static int check_train_shape(int T, int d, int f, int E, int K, int dtype) {
  const int st = check_shape(T, d, f, E, K, dtype);
  if (st != MOE_OK) return st;
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (d % 64 != 0 || f % 64 != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static int forward_impl(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2, void *y,
                        int T, int d, int f, int E, int K, int dtype, void *workspace, size_t ws_bytes,
                        unsigned flags, moe_stream_t stream, unsigned long long *stamps, bool train = false) {
  if (dtype == MOE_FP8_E4M3) return MOE_ERR_UNSUPPORTED;  // e4m3 weights go through moe_forward_fp8
  int st = train ? check_train_shape(T, d, f, E, K, dtype) : check_shape(T, d, f, E, K, dtype);
  if (st != MOE_OK) return st;
  if (flags & ~(MOE_ACCUMULATE | MOE_DEBUG_CHECKS | MOE_DEBUG_FORCE_TIMEOUT | kFormFlags)) return MOE_ERR_INVALID_ARG;
  if (!form_flags_ok(flags)) return MOE_ERR_INVALID_ARG;
  if ((flags & MOE_DEBUG_FORCE_TIMEOUT) && dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;  // empty input: nothing to compute, x and y may be NULL
  if (!x || !Wg || !W1 || !W3 || !W2 || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const size_t act_bytes = static_cast<size_t>(T) * d * elem_bytes(dtype);
  if (T > 0 && overlaps(x, act_bytes, y, act_bytes)) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  const int sms = sm_count_or_default();
  WsLayout L = ws_layout(T, d, f, E, K, dtype, sms, train);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  apply_form_flags(L, flags);
  st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Ptrs P = carve(workspace, L);
  P.stamps = stamps;
  // status word and split-tile counters start at zero (small batches: the
  // routing kernel clears them)
  if (!L.route_single && cudaMemsetAsync(P.status, 0, L.zero_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;

  cudaError_t err = launch_route_group(x, Wg, T, d, E, K, dtype, flags, L, P, s);
  if (err == cudaSuccess) err = launch_gather(x, T, d, E, dtype, L.R, P, sms, s, /*zero_pads=*/L.train);
  if (err == cudaSuccess) {
    if (dtype == MOE_BF16)
      err = launch_expert_gemms_bf16(W1, W3, W2, d, f, E, L, P, y, flags, sms, s);
    else
      err = launch_expert_ffn_f32(W1, W3, W2, d, f, E, L, P, s);
  }
  if (err == cudaSuccess && !L.fuse_combine) err = launch_combine(y, T, d, K, L.S, dtype, flags, P, sms, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_forward(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2, void *y, int T,
                int d, int f, int E, int K, int dtype, void *workspace, size_t ws_bytes, unsigned flags,
                moe_stream_t stream) {
  return forward_impl(x, Wg, W1, W3, W2, y, T, d, f, E, K, dtype, workspace, ws_bytes, flags, stream, nullptr);
}

static int block_forward_impl(void *h, const void *Wg, const void *W1, const void *W3, const void *W2, int T, int d,
                              int f, int E, int K, int dtype, float eps, void *workspace, size_t ws_bytes,
                              unsigned flags, moe_stream_t stream, unsigned long long *stamps) {
  if (dtype == MOE_FP8_E4M3) return MOE_ERR_UNSUPPORTED;
  int st = check_shape(T, d, f, E, K, dtype);
  if (st != MOE_OK) return st;
  if (flags & ~(MOE_DEBUG_CHECKS | MOE_DEBUG_FORCE_TIMEOUT | kFormFlags)) return MOE_ERR_INVALID_ARG;
  if (!(eps > 0.f)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!h || !aligned16(h)) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  const WsLayout L = ws_layout(T, d, f, E, K, dtype, sm_count_or_default());
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (overlaps(h, static_cast<size_t>(T) * d * elem_bytes(dtype), workspace, L.total)) return MOE_ERR_INVALID_ARG;
  st = check_device();
  if (st != MOE_OK) return st;
  const Ptrs P = carve(workspace, L);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // x_n = RMSNorm(h) into the workspace, then h += MoE(x_n)
  if (launch_rmsnorm(h, P.xnorm, T, d, eps, dtype, s, stamps) != cudaSuccess) return MOE_ERR_CUDA;
  return forward_impl(P.xnorm, Wg, W1, W3, W2, h, T, d, f, E, K, dtype, workspace, ws_bytes, flags | MOE_ACCUMULATE,
                      stream, stamps);
}

int moe_block_forward(void *h, const void *Wg, const void *W1, const void *W3, const void *W2, int T, int d, int f,
                      int E, int K, int dtype, float eps, void *workspace, size_t ws_bytes, unsigned flags,
                      moe_stream_t stream) {
  return block_forward_impl(h, Wg, W1, W3, W2, T, d, f, E, K, dtype, eps, workspace, ws_bytes, flags, stream,
                            nullptr);
}

int moe_block_forward_stamped(void *h, const void *Wg, const void *W1, const void *W3, const void *W2, int T, int d,
                              int f, int E, int K, int dtype, float eps, void *workspace, size_t ws_bytes,
                              unsigned flags, moe_stream_t stream, unsigned long long *stamps) {
  if (!stamps_ok(stamps)) return MOE_ERR_INVALID_ARG;
  return block_forward_impl(h, Wg, W1, W3, W2, T, d, f, E, K, dtype, eps, workspace, ws_bytes, flags, stream,
                            stamps);
}

int moe_forward_stamped(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2, void *y,
                        int T, int d, int f, int E, int K, int dtype, void *workspace, size_t ws_bytes,
                        unsigned flags, moe_stream_t stream, unsigned long long *stamps) {
  if (!stamps_ok(stamps)) return MOE_ERR_INVALID_ARG;
  return forward_impl(x, Wg, W1, W3, W2, y, T, d, f, E, K, dtype, workspace, ws_bytes, flags, stream, stamps);
}

int moe_forward_cached(const void *x, const void *Wg, const void *W1_host, const void *W3_host, const void *W2_host,
                       void *W1_dev, void *W3_dev, void *W2_dev, moe_expert_cache *cache, void *y, int T, int d,
                       int f, int E, int K, int dtype, void *workspace, size_t ws_bytes, unsigned flags,
                       moe_stream_t stream) {
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  int st = check_shape(T, d, f, E, K, dtype);
  if (st != MOE_OK) return st;
  if (flags & ~(MOE_ACCUMULATE | MOE_DEBUG_CHECKS)) return MOE_ERR_INVALID_ARG;
  if (!cache || cache->E != E || cache->C < 1 || cache->C > E) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const void *ptrs[] = {x, Wg, W1_host, W3_host, W2_host, W1_dev, W3_dev, W2_dev, y};
  for (const void *p : ptrs)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  const size_t act_bytes = static_cast<size_t>(T) * d * 2;
  if (overlaps(x, act_bytes, y, act_bytes)) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  const int sms = sm_count_or_default();
  WsLayout L = ws_layout(T, d, f, E, K, dtype, sms);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Ptrs P = carve(workspace, L);
  if (cudaMemsetAsync(P.status, 0, L.zero_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_route_group(x, Wg, T, d, E, K, dtype, flags, L, P, s) != cudaSuccess) return MOE_ERR_CUDA;
  // the experts this batch needs: wait for the grouping's segment offsets
  int32_t offs[kMaxE + 1];
  if (cudaMemcpyAsync(offs, P.offsets, (E + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  int needed[kMaxE], load_e[kMaxE], load_s[kMaxE], n_loads = 0;
  for (int e = 0; e < E; ++e) needed[e] = offs[e + 1] > offs[e] ? 1 : 0;
  st = moe_expert_cache_plan(cache, needed, load_e, load_s, &n_loads);
  if (st != MOE_OK) return st;
  // one copy per missed expert and bank, into its slot (ordered before the GEMMs)
  const size_t mat = static_cast<size_t>(d) * f * 2;
  const char *hosts[3] = {static_cast<const char *>(W1_host), static_cast<const char *>(W3_host),
                          static_cast<const char *>(W2_host)};
  char *devs[3] = {static_cast<char *>(W1_dev), static_cast<char *>(W3_dev), static_cast<char *>(W2_dev)};
  for (int i = 0; i < n_loads; ++i)
    for (int b = 0; b < 3; ++b)
      if (cudaMemcpyAsync(devs[b] + load_s[i] * mat, hosts[b] + load_e[i] * mat, mat, cudaMemcpyHostToDevice, s) !=
          cudaSuccess)
        return MOE_ERR_CUDA;
  cache->bytes_loaded += static_cast<long long>(n_loads) * 3 * static_cast<long long>(mat);
  cudaError_t err = launch_gather(x, T, d, E, dtype, L.R, P, sms, s, /*zero_pads=*/false);
  if (err == cudaSuccess)
    err = launch_expert_gemms_bf16(W1_dev, W3_dev, W2_dev, d, f, E, L, P, y, flags, sms, s, cache->slot_of, cache->C);
  if (err == cudaSuccess && !L.fuse_combine) err = launch_combine(y, T, d, K, L.S, dtype, flags, P, sms, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_forward_launches(int T, int d, int f, int E, int K, int dtype) {
  if (check_shape(T, d, f, E, K, dtype) != MOE_OK) return 0;
  if (T == 0) return 0;
  const WsLayout L = ws_layout(T, d, f, E, K, dtype, sm_count_or_default());
  // route and group (one fused launch up to kGroupTokens tokens), gather
  // (e4m3: gather + quantise), the two expert GEMMs (e4m3: plus the H
  // quantiser), and the combine unless the down GEMM forms y
  return (T <= kGroupTokens ? 1 : 2) + 3 + (dtype == MOE_FP8_E4M3 ? 1 : 0) + (L.fuse_combine ? 0 : 1);
}

size_t moe_train_workspace_bytes(int T, int d, int f, int E, int K, int dtype) {
  if (check_train_shape(T, d, f, E, K, dtype) != MOE_OK) return 0;
  return ws_layout(T, d, f, E, K, dtype, sm_count_or_default(), true).total;
}

int moe_forward_train(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2, void *y, int T,
                      int d, int f, int E, int K, int dtype, void *workspace, size_t ws_bytes, unsigned flags,
                      moe_stream_t stream) {
  return forward_impl(x, Wg, W1, W3, W2, y, T, d, f, E, K, dtype, workspace, ws_bytes, flags, stream, nullptr, true);
}

static int backward_impl(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2,
                         const void *dy, float *dx, float *dWg, float *dW1, float *dW3, float *dW2, int T, int d,
                         int f, int E, int K, int dtype, void *workspace, size_t ws_bytes, unsigned flags,
                         moe_stream_t stream, void *const *events) {
  int st = check_train_shape(T, d, f, E, K, dtype);
  if (st != MOE_OK) return st;
  if (flags & ~(MOE_ACCUMULATE | MOE_DEBUG_CHECKS | MOE_DEBUG_FORCE_TIMEOUT)) return MOE_ERR_INVALID_ARG;
  const bool acc = (flags & MOE_ACCUMULATE) != 0;
  if (!Wg || !W1 || !W3 || !W2 || !dWg || !dW1 || !dW3 || !dW2) return MOE_ERR_INVALID_ARG;
  if (!aligned16(Wg) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(dWg) || !aligned16(dW1) ||
      !aligned16(dW3) || !aligned16(dW2))
    return MOE_ERR_INVALID_ARG;
  const size_t wbytes = static_cast<size_t>(E) * d * f * 4;
  const float *outs[4] = {dWg, dW1, dW3, dW2};
  const size_t out_bytes[4] = {static_cast<size_t>(d) * E * 4, wbytes, wbytes, wbytes};
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    // no tokens: the weight gradients are zero
    st = check_device();
    if (st != MOE_OK || acc) return st;
    for (int i = 0; i < 4; ++i)
      if (cudaMemsetAsync(const_cast<float *>(outs[i]), 0, out_bytes[i], s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (!x || !dy || !dx) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dx)) return MOE_ERR_INVALID_ARG;
  const size_t dx_bytes = static_cast<size_t>(T) * d * 4;
  for (int i = 0; i < 4; ++i)
    if (overlaps(dx, dx_bytes, outs[i], out_bytes[i])) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  const int sms = sm_count_or_default();
  const WsLayout L = ws_layout(T, d, f, E, K, dtype, sms, true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  st = check_device();
  if (st != MOE_OK) return st;
  const Ptrs P = carve(workspace, L);
  cudaError_t err = events ? cudaEventRecord(static_cast<cudaEvent_t>(events[0]), s) : cudaSuccess;
  if (err == cudaSuccess) err = launch_bwd_prep(dy, T, d, E, K, L.S, L, P, sms, s);
  if (err == cudaSuccess && events) err = cudaEventRecord(static_cast<cudaEvent_t>(events[1]), s);
  if (err == cudaSuccess)
    err = launch_bwd_gemms(W1, W3, W2, dW1, dW3, dW2, d, f, E, acc, (flags & MOE_DEBUG_FORCE_TIMEOUT) != 0, L, P,
                           sms, s, events ? events + 2 : nullptr);
  if (err == cudaSuccess)
    err = launch_bwd_input(x, Wg, dx, dWg, T, d, E, K, acc, L, P, sms, s, events ? events + 6 : nullptr);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_backward(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2, const void *dy,
                 float *dx, float *dWg, float *dW1, float *dW3, float *dW2, int T, int d, int f, int E, int K,
                 int dtype, void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream) {
  return backward_impl(x, Wg, W1, W3, W2, dy, dx, dWg, dW1, dW3, dW2, T, d, f, E, K, dtype, workspace, ws_bytes,
                       flags, stream, nullptr);
}

int moe_backward_timed(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2, const void *dy,
                       float *dx, float *dWg, float *dW1, float *dW3, float *dW2, int T, int d, int f, int E, int K,
                       int dtype, void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream,
                       void *const *events) {
  if (!events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < MOE_NUM_BWD_STAGE_EVENTS; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return backward_impl(x, Wg, W1, W3, W2, dy, dx, dWg, dW1, dW3, dW2, T, d, f, E, K, dtype, workspace, ws_bytes,
                       flags, stream, events);
}

size_t moe_fp8_weight_bytes(int E, int K, int N) {
  if (E < 1 || K < 1 || N < 1) return 0;
  const size_t nt = (static_cast<size_t>(N) + 127) / 128, kt = (static_cast<size_t>(K) + 127) / 128;
  return static_cast<size_t>(E) * nt * kt * 128 * 128;
}

int moe_quantize_weights_fp8(const void *W, int E, int K, int N, void *Wq, float *scales, moe_stream_t stream) {
  if (E < 1 || K < 1 || N < 1) return MOE_ERR_INVALID_ARG;
  if (!W || !Wq || !scales) return MOE_ERR_INVALID_ARG;
  if (overlaps(W, static_cast<size_t>(E) * K * N * 2, Wq, moe_fp8_weight_bytes(E, K, N))) return MOE_ERR_INVALID_ARG;
  const int st = check_device();
  if (st != MOE_OK) return st;
  return launch_quantize_weights_fp8(W, E, K, N, Wq, scales, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

static int forward_fp8_impl(const void *x, const void *Wg, const void *W1q, const float *s1, const void *W3q,
                            const float *s3, const void *W2q, const float *s2, void *y, int T, int d, int f, int E,
                            int K, void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream,
                            unsigned long long *stamps) {
  constexpr int dtype = MOE_FP8_E4M3;
  int st = check_shape(T, d, f, E, K, dtype);
  if (st != MOE_OK) return st;
  if (flags & ~(MOE_ACCUMULATE | MOE_DEBUG_CHECKS | MOE_DEBUG_FORCE_TIMEOUT | kFormFlags)) return MOE_ERR_INVALID_ARG;
  if (!form_flags_ok(flags)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !Wg || !W1q || !W3q || !W2q || !s1 || !s3 || !s2 || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(W1q) || !aligned16(W3q) || !aligned16(W2q) || !aligned16(y) ||
      !aligned16(s1) || !aligned16(s3) || !aligned16(s2))
    return MOE_ERR_INVALID_ARG;
  const size_t act_bytes = static_cast<size_t>(T) * d * 2;
  if (overlaps(x, act_bytes, y, act_bytes)) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  const int sms = sm_count_or_default();
  WsLayout L = ws_layout(T, d, f, E, K, dtype, sms);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  apply_form_flags(L, flags);
  st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Ptrs P = carve(workspace, L);
  P.stamps = stamps;
  if (!L.route_single && cudaMemsetAsync(P.status, 0, L.zero_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
  // routing on the bf16 tokens, as moe_forward; the gather quantises rows
  cudaError_t err = launch_route_group(x, Wg, T, d, E, K, MOE_BF16, flags, L, P, s);
  if (err == cudaSuccess) err = launch_gather_quant(x, T, d, E, L.R, P, sms, s);
  if (err == cudaSuccess) err = launch_expert_gemms_fp8(W1q, s1, W3q, s3, W2q, s2, d, f, E, L, P, y, flags, sms, s);
  if (err == cudaSuccess && !L.fuse_combine) err = launch_combine(y, T, d, K, L.S, MOE_BF16, flags, P, sms, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_forward_fp8(const void *x, const void *Wg, const void *W1q, const float *s1, const void *W3q, const float *s3,
                    const void *W2q, const float *s2, void *y, int T, int d, int f, int E, int K, void *workspace,
                    size_t ws_bytes, unsigned flags, moe_stream_t stream) {
  return forward_fp8_impl(x, Wg, W1q, s1, W3q, s3, W2q, s2, y, T, d, f, E, K, workspace, ws_bytes, flags, stream,
                          nullptr);
}

int moe_forward_fp8_stamped(const void *x, const void *Wg, const void *W1q, const float *s1, const void *W3q,
                            const float *s3, const void *W2q, const float *s2, void *y, int T, int d, int f, int E,
                            int K, void *workspace, size_t ws_bytes, unsigned flags, moe_stream_t stream,
                            unsigned long long *stamps) {
  if (!stamps_ok(stamps)) return MOE_ERR_INVALID_ARG;
  return forward_fp8_impl(x, Wg, W1q, s1, W3q, s3, W2q, s2, y, T, d, f, E, K, workspace, ws_bytes, flags, stream,
                          stamps);
}

int moe_route(const void *x, const void *Wg, int T, int d, int E, int K, int dtype, int32_t *idx, float *gate,
              int32_t *perm_tok, int32_t *offsets, int32_t *pos, void *workspace, size_t ws_bytes,
              moe_stream_t stream) {
  // f only sizes the expert buffers; routing needs none of them.
  int st = check_shape(T, d, dtype == MOE_BF16 ? 8 : 4, E, K, dtype);
  if (st != MOE_OK) return st;
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (T == 0) {
    // Empty input: every expert segment is empty; the other outputs have no elements.
    if (check_device() != MOE_OK) return MOE_ERR_CUDA;
    return cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  }
  if (!x || !Wg || !idx || !gate || !perm_tok) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg)) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  const WsLayout L = ws_layout(T, d, dtype == MOE_BF16 ? 8 : 4, E, K, dtype, sm_count_or_default());
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Ptrs P = carve(workspace, L);
  if (cudaMemsetAsync(P.status, 0, kStatusInts * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t err = launch_route_group(x, Wg, T, d, E, K, dtype, 0, L, P, s);
  if (err == cudaSuccess) err = launch_route_export(T, E, K, P, idx, gate, perm_tok, offsets, pos, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_rmsnorm(const void *x, void *out, int T, int d, float eps, int dtype, moe_stream_t stream) {
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || d < 1 || !(eps > 0.f)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out) return MOE_ERR_INVALID_ARG;
  const int st = check_device();
  if (st != MOE_OK) return st;
  cudaError_t err = launch_rmsnorm(x, out, T, d, eps, dtype, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_read_status(const void *workspace, moe_stream_t stream) {
  if (!workspace) return MOE_ERR_WORKSPACE;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  return v;
}

const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA runtime or launch error";
    case MOE_ERR_DEVICE_TIMEOUT: return "bounded device-side wait expired";
    case MOE_ERR_NONFINITE: return "non-finite router logit";
    case MOE_ERR_DEVICE_BOUNDS: return "device-side index out of range";
    default: return "unknown status";
  }
}

int moe_version(void) { return 100; }

}  // extern "C"
