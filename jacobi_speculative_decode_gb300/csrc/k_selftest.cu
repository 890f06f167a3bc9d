// Self-test of the kernels' failure path: every mbarrier wait in the library is
// bounded in time (ptx::mbar_wait gives up after about half a second, sets
// XP_ERR_TIMEOUT in the head's error word and raises the CTA's abort flag), so a
// wait that can never be satisfied ends the kernel with an error the host reads,
// instead of a hung GPU.  This file launches one wait that nothing will ever
// complete, so that callers and tests can check that path without any fault.
#include "sm100_ptx.cuh"
#include "xp_internal.h"

namespace {

__global__ void wait_timeout_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  // nothing arrives on the barrier: phase 0 never completes, the wait runs out
  if (threadIdx.x == 0) ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_flag, err);
  __syncthreads();
}

}  // namespace

extern "C" xp_status xp_selftest_wait_timeout(const xp_head* h, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!xp_on_head_device(h)) return XP_EINVAL;
  wait_timeout_kernel<<<1, 32, 0, stream>>>(h->err);
  return cudaGetLastError() == cudaSuccess ? XP_OK : XP_ECUDA;
}
