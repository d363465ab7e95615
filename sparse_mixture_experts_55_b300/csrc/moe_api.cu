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

int elem_bytes(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }

// Shape checks shared by every entry point.  Returns MOE_OK or an error code.
int check_shape(int T, int d, int f, int E, int K, int dtype) {
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || d < 1 || f < 1 || E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (K > E) return MOE_ERR_INVALID_ARG;
  if (K > kMaxK || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  const int mult = dtype == MOE_BF16 ? 8 : 4;  // 16-byte rows for vector loads and TMA strides
  if (d % mult != 0 || f % mult != 0) return MOE_ERR_INVALID_ARG;
  // index arithmetic of the grouped buffers stays in 32-bit rows
  const long long rows = static_cast<long long>(T) * K + static_cast<long long>(E) * kSegPad;
  if (rows >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

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

}  // namespace

int down_splits(int T, int d, int f, int E, int K, int num_sms) {
  const int n_tiles = (d + 255) / 256;
  const long long rows = static_cast<long long>(T) * K;
  const long long touched = rows < E ? rows : E;
  // upper bound on the number of 128-row tiles over all experts
  const long long m_tiles = (rows + kSegPad - 1) / kSegPad + (touched > 0 ? touched - 1 : 0);
  const long long units = m_tiles * n_tiles;
  if (units <= 0 || units >= num_sms) return 1;
  int S = static_cast<int>(num_sms / units);
  const int kb = (f + 63) / 64;
  if (S > 16) S = 16;
  if (S > kb) S = kb;
  return S < 1 ? 1 : S;
}

WsLayout ws_layout(int T, int d, int f, int E, int K, int dtype, int num_sms) {
  WsLayout L{};
  const size_t eb = elem_bytes(dtype);
  L.R = static_cast<int>(align_up(static_cast<size_t>(T) * K + static_cast<size_t>(E) * (kSegPad - 1), kSegPad));
  L.n_route_blocks = (T + kRouteTokens - 1) / kRouteTokens;
  const int kb = (f + 63) / 64;
  int S = dtype == MOE_BF16 ? down_splits(T, d, f, E, K, num_sms) : 1;
  L.kb_per_split = (kb + S - 1) / S;
  L.S = (kb + L.kb_per_split - 1) / L.kb_per_split;  // every split owns >= 1 k-block
  const size_t TK = static_cast<size_t>(T) * K;
  const size_t R = static_cast<size_t>(L.R);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.status = take(kStatusInts * sizeof(int));
  L.idx = take(TK * 4);
  L.gate = take(TK * 4);
  L.blockcounts = take(static_cast<size_t>(L.n_route_blocks > 0 ? L.n_route_blocks : 1) * E * 4);
  L.offsets = take((E + 1) * 4);
  L.poffsets = take((E + 1) * 4);
  L.pos = take(TK * 4);
  L.perm_tok = take(R * 4);
  L.perm_gate = take(R * 4);
  L.xperm = take(R * d * eb);
  L.hbuf = take(R * f * eb);
  L.obuf = take(static_cast<size_t>(L.S) * R * d * 4);
  L.total = o;
  return L;
}

Ptrs carve(void *ws, const WsLayout &L) {
  char *b = static_cast<char *>(ws);
  Ptrs P;
  P.status = reinterpret_cast<int *>(b + L.status);
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
  return P;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(int T, int d, int f, int E, int K, int dtype) {
  if (check_shape(T, d, f, E, K, dtype) != MOE_OK) return 0;
  return ws_layout(T, d, f, E, K, dtype, sm_count_or_default()).total;
}

static int forward_impl(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2, void *y,
                        int T, int d, int f, int E, int K, int dtype, void *workspace, size_t ws_bytes,
                        unsigned flags, moe_stream_t stream, void *const *events) {
  int st = check_shape(T, d, f, E, K, dtype);
  if (st != MOE_OK) return st;
  if (flags & ~(MOE_ACCUMULATE | MOE_DEBUG_CHECKS)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;  // empty input: nothing to compute, x and y may be NULL
  if (!x || !Wg || !W1 || !W3 || !W2 || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  const size_t act_bytes = static_cast<size_t>(T) * d * elem_bytes(dtype);
  if (T > 0 && overlaps(x, act_bytes, y, act_bytes)) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
  const int sms = sm_count_or_default();
  const WsLayout L = ws_layout(T, d, f, E, K, dtype, sms);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Ptrs P = carve(workspace, L);
  if (cudaMemsetAsync(P.status, 0, kStatusInts * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;

  // events (optional): one before the router and one after each of the six stages
  auto mark = [&](int i) -> cudaError_t {
    return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) : cudaSuccess;
  };
  cudaError_t err = mark(0);
  if (err == cudaSuccess) err = launch_route(x, Wg, T, d, E, K, dtype, flags, P, s);
  if (err == cudaSuccess) err = mark(1);
  if (err == cudaSuccess) err = launch_group(T, E, K, L.n_route_blocks, flags, P, s);
  if (err == cudaSuccess) err = mark(2);
  if (err == cudaSuccess) err = launch_gather(x, T, d, E, dtype, L.R, P, sms, s);
  if (err == cudaSuccess) err = mark(3);
  if (err == cudaSuccess) {
    if (dtype == MOE_BF16)
      err = launch_expert_gemms_bf16(W1, W3, W2, d, f, E, L, P, flags, sms, s, events ? events + 4 : nullptr);
    else
      err = launch_expert_ffn_f32(W1, W3, W2, d, f, E, L, P, s, events ? events + 4 : nullptr);
  }
  if (err == cudaSuccess) err = mark(5);
  if (err == cudaSuccess) err = launch_combine(y, T, d, K, L.S, L.R, dtype, flags, P, sms, s);
  if (err == cudaSuccess) err = mark(6);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_forward(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2, void *y, int T,
                int d, int f, int E, int K, int dtype, void *workspace, size_t ws_bytes, unsigned flags,
                moe_stream_t stream) {
  return forward_impl(x, Wg, W1, W3, W2, y, T, d, f, E, K, dtype, workspace, ws_bytes, flags, stream, nullptr);
}

int moe_forward_timed(const void *x, const void *Wg, const void *W1, const void *W3, const void *W2, void *y,
                      int T, int d, int f, int E, int K, int dtype, void *workspace, size_t ws_bytes,
                      unsigned flags, moe_stream_t stream, void *const *events) {
  if (!events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < MOE_NUM_STAGE_EVENTS; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return forward_impl(x, Wg, W1, W3, W2, y, T, d, f, E, K, dtype, workspace, ws_bytes, flags, stream, events);
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
  cudaError_t err = launch_route(x, Wg, T, d, E, K, dtype, 0, P, s);
  if (err == cudaSuccess) err = launch_group(T, E, K, L.n_route_blocks, 0, P, s);
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
