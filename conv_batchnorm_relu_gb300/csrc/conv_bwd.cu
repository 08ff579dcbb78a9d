// B2 (dgrad) and B3 (wgrad) -- placeholders until the tensor-core kernels land.
#include "cbr_internal.h"
#include "common.cuh"

namespace cbr {

size_t wgrad_partial_floats(int num_sms, int c_in, int c_out, int taps) {
  const int cin_pad = ((c_in + 63) / 64) * 64;
  const int groups = (taps + 1) / 2;
  return (size_t)num_sms * groups * 2 * cin_pad * c_out;
}

int launch_dgrad(const DgradArgs&, int, int, bool, const void*, int, cudaStream_t) { return 3; }
int launch_wgrad(const WgradArgs&, int, int, bool, const void*, int, cudaStream_t) { return 3; }

}  // namespace cbr
