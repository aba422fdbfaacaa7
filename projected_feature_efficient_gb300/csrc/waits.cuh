// waits.cuh -- bounded waits and the static work order shared by the
// persistent tcgen05 kernels (forward and backward).
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace spa {

// What a bounded wait needs: the CTA's abort flag, the device error word and
// the time limit of one wait.
struct WaitCtl {
  volatile int* abort;
  int* err;
  uint64_t limit_ns;
};

// Bounded wait that also gives up once another role of the CTA has aborted.
// The common case (phase already complete) costs one try_wait.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  if (*ctl.abort) return false;
  if (ptx::mbar_wait(bar, parity, ctl.limit_ns)) return true;
  *ctl.abort = 1;
  atomicExch(ctl.err, 1);
  return false;
}

// The k-th work item of this CTA: rounds of gridDim.x items, every other round
// in reverse, so that a CTA that drew a longer item in one round draws a
// shorter one in the next.  Returns -1 past the end.
__device__ __forceinline__ int item_index(int k, int items) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int w = k * G + ((k & 1) ? G - 1 - c : c);
  return w < items ? w : -1;
}

}  // namespace spa
