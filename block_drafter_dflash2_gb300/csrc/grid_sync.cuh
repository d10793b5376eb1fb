// Grid-wide and group barriers between the CTAs of one cooperative launch: an arrival
// counter in global memory per barrier, counted up by one per member and round (the host
// zeroes it before the launch), and a bounded acquire spin by one thread per CTA.
#pragma once

#include "../../include/dflash2.h"
#include "ptx.cuh"

namespace df {

DF_DEV uint32_t ld_acquire(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Barrier number `round` (1, 2, ...) of `members` CTAs sharing `count`. The arrival is a
// release (it orders every write the CTA made before the __syncthreads) and the wait is an
// acquire spin by one thread, so the CTA's reads after the closing __syncthreads see every
// member's writes. The time limit is checked every 256 polls. A CTA that has already
// stopped (an earlier wait timed out) still arrives, so the others are not held up, but
// does not wait.
DF_DEV bool group_barrier(unsigned* count, unsigned round, unsigned members, int32_t* err, volatile int* stop) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(count) : "memory");
    const unsigned target = round * members;
    uint64_t t0 = 0;
    for (unsigned it = 0; *stop == 0 && ld_acquire(count) < target; ++it) {
      if ((it & 255u) == 0) {
        const uint64_t now = globaltimer_ns();
        if (it == 0) {
          t0 = now;
        } else if (now - t0 > kWaitLimitNs) {
          flag_error(err, DFLASH2_DEVERR_WAIT_TIMEOUT);
          *stop = 1;
          break;
        }
      }
    }
  }
  __syncthreads();
  return *stop == 0;
}

}  // namespace df
