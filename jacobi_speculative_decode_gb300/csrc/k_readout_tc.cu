// tcgen05 readout (placeholder until the tensor-core kernel lands).
#include "xp_internal.h"

bool xp_readout_tc_call_ok(const xp_head*, const void*, const void*, int64_t, int64_t, int) {
  return false;
}
cudaError_t xp_launch_readout_tc(const xp_head*, const void*, const void*, int64_t, int64_t, int,
                                 int64_t*, float*, unsigned long long*, unsigned*, cudaStream_t) {
  return cudaErrorNotSupported;
}
