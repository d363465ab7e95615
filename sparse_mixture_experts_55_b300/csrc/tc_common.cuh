// tc_common.cuh -- pieces shared by the tensor-core GEMM kernels: the bounded
// mbarrier wait and the TMA tensor-map encoders (defined in tmap.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr uint64_t kTimeoutNs = 1000000000ull;  // about one second per wait

// Bounded mbarrier wait for a CTA whose control block C has an `abort` flag.
// Returns false if the CTA is aborting (when honor_abort) or the wait
// expired; expiry records MOE_ERR_DEVICE_TIMEOUT in *status and raises the
// CTA's abort flag.
template <class C>
__device__ __noinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, C &c, int *status, bool honor_abort) {
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

// Tensor maps with 128-byte swizzle (all return false if the driver entry
// point is missing or rejects the map):
//   tmap_2d      bf16 [rows, cols] (cols contiguous), box 64 cols x box_rows rows
//   tmap_3d      bf16 bank [E, rows, cols], box 64 cols x box_rows rows x 1
//   tmap_2d_u8   e4m3 [rows, cols], box 128 cols x box_rows rows
//   tmap_4d_w    bf16 bank viewed in 64-column blocks, box 128 cols x 64 rows
//   tmap_blocks_2d  bf16 [rows, cols] viewed in 64-column blocks, box nblk blocks x 64 rows
bool tmap_2d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_rows);
bool tmap_3d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t E, uint32_t box_rows = 64);
bool tmap_2d_u8(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_rows);
// bf16 bank [E, rows, cols] with cols a multiple of 128, viewed as [E, cols/64, rows, 64]:
// one box is 64 x 64 x 2 blocks, i.e. 128 columns x 64 rows in two 8 KiB swizzled blocks.
bool tmap_4d_w(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint64_t E);
// bf16 matrix [rows, cols] with cols a multiple of 64, viewed as [cols/64, rows, 64]:
// one box is 64 columns x 64 rows x nblk column blocks (nblk 8 KiB swizzled blocks).
bool tmap_blocks_2d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t nblk);

}  // namespace moe
