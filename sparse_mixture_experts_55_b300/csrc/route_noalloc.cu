// route_noalloc.cu -- moe_route_noalloc: the routing entry point for callers
// that cannot allocate device memory.
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
// cudaGetSymbolAddress (with that device current) and caches it; make that
// first call before any stream capture.  Calls that overlap on the GPU (two
// streams, or two host threads) race on the array.
#include <cuda_runtime.h>

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

struct ScratchSlot {
  bool ready = false;
  void *ptr = nullptr;
};

// Device address of g_route_scratch on the current device, looked up once per device.
cudaError_t scratch_address(void **out) {
  static std::mutex mu;
  static ScratchSlot slots[64];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  ScratchSlot &s = slots[dev];
  if (!s.ready) {
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess) return err;
    s.ptr = p;
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
                                 moe_stream_t stream) {
  if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || d < 1 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
  if (K > kMaxK || E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if (d % (dtype == MOE_BF16 ? 8 : 4) != 0) return MOE_ERR_INVALID_ARG;
  if (T > MOE_ROUTE_NOALLOC_MAX_T) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch array
  if (!offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0) {
    if (!x || !Wg || !idx || !gate || !perm_tok) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(Wg) & 15u))
      return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0)
    return cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;

  // Only the routing part of the workspace layout is used: everything before
  // the grouped activation buffers.
  const WsLayout L = ws_layout(T, d, dtype == MOE_BF16 ? 8 : 4, E, K, dtype, 148, false, /*routing_only=*/true);
  if (L.xperm > kNoAllocBytes) return MOE_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  const Ptrs P = carve(scratch, L);
  // The status word must start at zero; every other scratch word the kernels
  // read is written earlier in the same call.
  if (cudaMemsetAsync(P.status, 0, kStatusInts * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t err = launch_route(x, Wg, T, d, E, K, dtype, 0, L, P, s);
  if (err == cudaSuccess) err = launch_group(T, E, K, L, 0, P, s);
  if (err == cudaSuccess) err = launch_route_export(T, E, K, P, idx, gate, perm_tok, offsets, pos, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
