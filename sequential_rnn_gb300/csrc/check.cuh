// Index checks of the bounds-check build (-DRNN_BOUNDS_CHECK, libsrnn_bc.so).
//
// No sanitizer runs on the GPUs this library targets, so the kernels check the
// indices they compute themselves: every global-memory element index against
// its buffer's extent (derived from the call's T, B, NH, Dh) and the main
// shared-memory offsets (R fragments, the Wx ring, the h buffers, remote
// st.async destinations) against the CTA's layout.  A failed check records
// kStatusBounds in the call's status word (rnn_read_status: RNN_ERR_BOUNDS) and
// the access is skipped.  In the normal build bc_ok() is a constant true and
// the checks compile away.
#pragma once
#include "kernels.h"

namespace srnn {

#ifdef RNN_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif

__device__ __forceinline__ bool bc_ok(long long i, long long n, int* status) {
  if constexpr (!kBoundsCheck) {
    return true;
  } else {
    if (i >= 0 && i < n) return true;
    if (status != nullptr) atomicOr(status, kStatusBounds);
    return false;
  }
}

}  // namespace srnn
