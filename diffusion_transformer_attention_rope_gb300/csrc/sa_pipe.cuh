// sa_pipe.cuh -- bounded pipeline waits shared by the attention kernels.
#pragma once

#include <cstdint>

#include "sa_ptx.cuh"

namespace sa {

// Pipeline wait: bounded by the wall clock and by the CTA abort flag.  The first probe is a
// non-blocking test (several times cheaper than a suspending probe when the phase has already
// completed, the common case); the clock is read only after it fails.  A suspending probe
// returns only once the phase completes or after a limit of about a microsecond or more, so
// with bounds that short (failure tests) the wait keeps polling and reads the clock each time.
__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      int* err, int err_bit, uint64_t timeout_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const bool poll = timeout_ns < 4000u;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      atomicOr(err, err_bit);
      return false;
    }
  }
}

// Warp-uniform pipeline wait: every lane waits, and the warp agrees on the outcome.
__device__ __forceinline__ bool pwait_w(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        int* err, int err_bit, uint64_t timeout_ns) {
  return __all_sync(0xffffffffu, pwait(bar, parity, abort_flag, err, err_bit, timeout_ns));
}

}  // namespace sa
