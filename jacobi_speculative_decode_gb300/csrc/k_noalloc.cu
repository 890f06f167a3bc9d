// Readout + argmax for callers that cannot hand the library device memory.
//
// xp_readout_argmax needs a caller-allocated workspace for its cross-CTA argmax
// partials and tickets.  Some callers cannot allocate device memory at the point
// where they refine a block: code running inside another framework's memory
// pool that it does not own, or a latency-critical path where a cudaMalloc (and
// the device synchronisation it can bring) is not acceptable.  For them this
// file keeps that scratch in a fixed array in the library's own device memory,
// present on every GPU that loads the library until the process exits; the
// entry point below allocates nothing.
#include <mutex>

#include "xp_internal.h"

namespace {

// Largest number of draft rows (N * (B - 1)) one call may refine.
constexpr int kMaxRows = 4096;
// argmax partials (one u64 per row), then tickets (at most one per row)
constexpr size_t kPackedBytes = (size_t)kMaxRows * 8;
constexpr size_t kScratchBytes = kPackedBytes + (size_t)kMaxRows * 4;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" xp_status xp_readout_argmax_noalloc(const xp_head* h, const void* lat, const void* base,
                                               int64_t stride_n, int64_t stride_b, int N,
                                               int64_t* blk, float* win_val,
                                               cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!lat || !base || stride_n < 0 || stride_b < 0 || !blk || N < 0) return XP_EINVAL;
  // the scratch address looked up below is the current device's: it must be the head's
  if (!xp_on_head_device(h)) return XP_EINVAL;
  if (N > h->max_N) return XP_ECAPACITY;
  if ((int64_t)N * (h->B - 1) > kMaxRows) return XP_ECAPACITY;
  if (N == 0) return XP_OK;
  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return XP_ECUDA;
  // the partials and tickets must start at zero; the array keeps the last call's state
  if (cudaMemsetAsync(scratch, 0, kScratchBytes, stream) != cudaSuccess) return XP_ECUDA;
  auto* packed = static_cast<unsigned long long*>(scratch);
  auto* ticket = reinterpret_cast<unsigned*>(static_cast<unsigned char*>(scratch) + kPackedBytes);
  if (h->readout_tc && xp_readout_tc_call_ok(h, lat, base, stride_n, stride_b, N)) {
    const cudaError_t e = xp_launch_readout_tc(h, lat, base, stride_n, stride_b, N, blk, win_val,
                                               packed, ticket, stream);
    if (e != cudaErrorNotSupported) return e == cudaSuccess ? XP_OK : XP_ECUDA;
  }
  return xp_launch_readout_simt(h, lat, base, stride_n, stride_b, N, blk, win_val, packed, ticket,
                                stream) == cudaSuccess
             ? XP_OK
             : XP_ECUDA;
}
