// stamps.cuh -- per-stage device timestamps for the profiling entry points
// (moe_forward_stamped and friends).  A stamps array holds kNumStages begin
// times followed by kNumStages end times, in nanoseconds of the GPU's global
// timer; each CTA of a stage's kernel lowers the begin time to the moment it
// starts its work (after waiting for its inputs) and raises the end time to
// the moment it finishes, so end - begin is the kernel's span as the
// surrounding run sees it.  A null array costs one predicated branch.
#pragma once

#include <cstdint>

#include "internal.h"

namespace moe {

__device__ __forceinline__ unsigned long long stamp_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Called by every thread of the CTA once its inputs are ready.
__device__ __forceinline__ void stamp_begin(unsigned long long *st, int stage) {
  if (st != nullptr && threadIdx.x == 0) atomicMin(st + stage, stamp_now());
}

// Called by every thread of the CTA after its last store (a CTA barrier).
__device__ __forceinline__ void stamp_end(unsigned long long *st, int stage) {
  if (st != nullptr) {
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(st + kNumStages + stage, stamp_now());
  }
}

}  // namespace moe
