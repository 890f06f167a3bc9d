// Cluster tensor-core latent (placeholder until the kernel lands).
#include "xp_internal.h"

cudaError_t xp_launch_latent_mma(const xp_head*, const int64_t*, const int64_t*, const float*,
                                 int, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
