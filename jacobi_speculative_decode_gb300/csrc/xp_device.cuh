// Device-side helpers shared by the kernels: loads, argmax keys, token checks.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "xp_internal.h"

namespace xpd {

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Monotone map float -> uint32 for finite values; -0 and +0 share one key.
__device__ __forceinline__ uint32_t f2key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}
// (value, index) packed so that a larger u64 is the better candidate: larger
// value first, then the lower index.  0 is below every finite candidate.
__device__ __forceinline__ unsigned long long pack_best(float v, uint32_t idx) {
  return ((unsigned long long)f2key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t packed_idx(unsigned long long p) {
  return 0xFFFFFFFFu - (uint32_t)(p & 0xFFFFFFFFull);
}
__device__ __forceinline__ float packed_val(unsigned long long p) { return key2f((uint32_t)(p >> 32)); }

// better(v, i) than (bv, bi): higher value, or equal value and lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// warp-wide (value, index) argmax with the same ordering
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// Token id read from the block buffer: out-of-range ids are clamped and flagged.
__device__ __forceinline__ int64_t checked_token(int64_t t, int V, uint32_t* err) {
  if (t < 0 || t >= (int64_t)V) {
    atomicOr(err, XP_ERR_BADTOKEN);
    t = t < 0 ? 0 : (int64_t)V - 1;
  }
  return t;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

// After this CTA merged its per-row candidates into `packed` with atomicMax,
// take a ticket on `ticket`; the CTA that arrives last (ticket == expected-1)
// returns true and must publish + reset.  No CTA waits for another.  One thread
// takes the ticket with an acquire-release atomic after the CTA barrier: the
// release covers every thread's earlier atomics (the barrier orders them before
// it), and in the last CTA the acquire orders the other CTAs' atomics before the
// publish that follows the second barrier.
__device__ __forceinline__ bool arrive_last(unsigned* ticket, unsigned expected, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned t;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(t) : "l"(ticket) : "memory");
    *s_flag = (t == expected - 1u);
  }
  __syncthreads();
  return *s_flag != 0;
}

}  // namespace xpd
