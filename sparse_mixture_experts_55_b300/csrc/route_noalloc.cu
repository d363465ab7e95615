// route_noalloc.cu -- moe_route_noalloc: the routing entry point for callers
// that cannot allocate device memory, and moe_route_noalloc_status, which
// reads its device status word.
//
// Some callers have no way to hand the library a workspace: a plugin host
// that gives its kernels no scratch buffer, code that runs while another
// thread captures a CUDA graph in global mode (cudaMalloc is illegal then), or
// a serving loop that must never risk an allocation (and the device
// synchronisation it can bring) on its hot path.  For them this entry point
// runs the same router and grouping kernels as moe_route with their scratch in
// a fixed array compiled into the library instead of a caller buffer.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library reserves it until the process exits, and every call on that GPU
// shares it.  Host code cannot use the array's name as a device address, so
// the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it, keyed by the
// device's current context so that a new context (after cudaDeviceReset, for
// instance) looks it up again; make that first call before any stream
// capture.  Calls that overlap on the GPU (two streams, or two host threads)
// race on the array.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace moe {
namespace {

// Routing scratch for T <= MOE_ROUTE_NOALLOC_MAX_T tokens, K <= 2, E <= 32:
// status word, idx, gate, block histograms, offsets, pos and the padded
// grouped token/gate arrays (under 0.7 MiB at the limit).
constexpr size_t kNoAllocBytes = 1024 * 1024;
static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocBytes];

// The current context, through the runtime's driver entry-point query (the
// library does not link libcuda); null if the query is unavailable.
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  CUcontext ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

struct ScratchSlot {
  bool ready = false;
  CUcontext ctx = nullptr;
  void *ptr = nullptr;
};

// Device address of g_route_scratch on the current device, looked up on the
// first call in each context of the device.
cudaError_t scratch_address(void **out) {
  static std::mutex mu;
  static ScratchSlot slots[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(mu);
  ScratchSlot &s = slots[dev];
  if (!s.ready || s.ctx != ctx) {
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess) return err;
    s.ptr = p;
    s.ctx = ctx;
    s.ready = true;
  }
  *out = s.ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_route_noalloc(const void *x, const void *Wg, int T, int d, int E, int K, int dtype,
                                 int32_t *idx, float *gate, int32_t *perm_tok, int32_t *offsets, int32_t *pos,
                                 unsigned flags, moe_stream_t stream) {
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || d < 1 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
  if (K > kMaxK || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if (d % (dtype == MOE_BF16 ? 8 : 4) != 0) return MOE_ERR_INVALID_ARG;
  if (flags & ~MOE_DEBUG_CHECKS) return MOE_ERR_INVALID_ARG;
  if (T > MOE_ROUTE_NOALLOC_MAX_T) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch array
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0) {
    if (!x || !Wg || !idx || !gate || !perm_tok) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(Wg) & 15u))
      return MOE_ERR_INVALID_ARG;
  }
  const int st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) {
    // no tokens: every expert segment is empty, and no device error
    if (cudaMemsetAsync(scratch, 0, kStatusInts * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
    return cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }

  // Only the routing part of the workspace layout is used: everything before
  // the grouped activation buffers.
  const WsLayout L = ws_layout(T, d, dtype == MOE_BF16 ? 8 : 4, E, K, dtype, sm_count_or_default(), false,
                               /*routing_only=*/true);
  if (L.xperm > kNoAllocBytes) return MOE_ERR_UNSUPPORTED;
  const Ptrs P = carve(scratch, L);
  // The status words (the status and the fused router's ticket) must start
  // at zero; every other scratch word the kernels read is written earlier in
  // the same call.
  if (cudaMemsetAsync(P.status, 0, kStatusInts * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t err = launch_route_group(x, Wg, T, d, E, K, dtype, flags, L, P, s);
  if (err == cudaSuccess) err = launch_route_export(T, E, K, P, idx, gate, perm_tok, offsets, pos, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_route_noalloc_status(moe_stream_t stream) {
  const int st = check_device();
  if (st != MOE_OK) return st;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  return v;
}
