// wait.cuh -- the bounded mbarrier wait every pipelined kernel of the library uses.
#pragma once

#include <cstdint>

#include "ptx_sm103.cuh"
#include "rec_attn_internal.cuh"

namespace recattn {

// Wait for the phase of `bar` with the given parity.  Gives up (returns false) when
// another role of the CTA has aborted (*abort_flag set), or after limit_ns of global
// time, in which case it records REC_ATTN_ERR_TIMEOUT in the status word and raises
// the CTA's abort flag, so the other roles stop at their next wait instead of hanging.
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status,
                                             uint64_t limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > limit_ns) {
      *abort_flag = 1;
      set_status(status, REC_ATTN_ERR_TIMEOUT);
      return false;
    }
  }
}

}  // namespace recattn
