// Latent stage of one pass on tensor cores, persistent 8-CTA clusters
// (xpress kernels page, _xpress_latent_kernel; qwen3_xpress page, _refine_latent):
//   prev[0] = am1[n], prev[b] = blk[n, b-1]
//   x[b]    = xh[n, b] + w_lat w1[prev[b]]
//   u[b, c] = sum_j mix[c, b, j] x[j, c]            (stored mixer is lower-triangular)
//   lat[b]  = u[b] + w_down (silu(w_gate u[b]) * (w_up u[b]))      for b = 1..B-1
//
// w_lat w1[t] is read from a table E = w1 w_lat^T (fp32, [V, r]) that the head
// prepares once from its weights, so the per-pass work starts from a row gather.
//
// The cluster splits the work so each CTA holds only 1/8 of the weights: CTA q
// owns channels [q*r/8, (q+1)*r/8) (mixer, residual, output) and hidden units
// [q*H/8, (q+1)*H/8) (SwiGLU).  Per group of MT rows (whole blocks):
//   1. gather E rows and xh for the own channels (cp.async), x = xh + E[prev]
//   2. u = per-channel causal mix of x (fp32); push the own u slice to every CTA
//      of the cluster as a bf16 hi + lo pair (u = hi + lo to ~2^-17) with
//      st.async, which completes bytes on the receiver's mbarrier
//   3. a = silu(u w_gate[own]^T) * (u w_up[own]^T) from hi and lo: tcgen05.mma
//      (M = 128 rows, of which the group's MT are real) into TMEM, kept as hi + lo
//   4. partial = a w_down[:, own]^T for ALL channels, tcgen05.mma again (w_down's
//      column slice arrives by TMA into the u buffer, dead by then); each
//      32-channel piece is pushed to the CTA owning those channels
//   5. lat = u + the 8 partials of the own channels, added in a fixed order
// The only cluster-wide barrier per group is a split arrive/wait that keeps a
// CTA from pushing into buffers a peer is still reading.
//
// bf16 matrices in shared memory use the TMA 128-byte-swizzle layout in
// 64-column chunks: element (row, k) of an R-row matrix lives at
//   (k / 64) * R * 128 + row * 128 + ((((k % 64) / 8) ^ (row % 8)) * 16) + (k % 8) * 2.
#include <cooperative_groups.h>

#include <algorithm>

#include "sm100_ptx.cuh"
#include "xp_device.cuh"

namespace cg = cooperative_groups;
using namespace xpd;
typedef __nv_bfloat16 bf16;

namespace {

constexpr int CL = 8;          // CTAs per cluster
constexpr int THREADS = 256;   // 8 warps

struct Plan {                  // byte offsets into dynamic shared memory
  int MT, CS, HS;
  int wg, wu, mix, ubuf, ahi, alo, rcv, ex, xh, us, prev, bars;
  int mix_rows;
  int total;
};

__host__ __device__ inline Plan make_plan(int MT, int r, int H, int B) {
  Plan p;
  p.MT = MT;
  p.CS = r / CL;
  p.HS = H / CL;
  p.mix_rows = B * B;
  const int mparts = (p.mix_rows + 255) / 256, mbox = std::min(p.mix_rows, 256);
  int o = 0;
  // TMA / swizzled regions 1024-byte aligned, the rest 16-byte aligned
  auto take = [&](int bytes, int align) {
    o = (o + align - 1) / align * align;
    const int at = o;
    o += bytes;
    return at;
  };
  p.wg = take(p.HS * r * 2, 1024);
  p.wu = take(p.HS * r * 2, 1024);
  p.mix = take(mparts * mbox * p.CS * 2, 1024);
  // u hi + lo ([MT, r] each), later w_down[:, own units] ([r, HS])
  p.ubuf = take(std::max(2 * MT * r * 2, r * p.HS * 2), 1024);
  p.ahi = take(MT * p.HS * 2, 1024);
  p.alo = take(MT * p.HS * 2, 1024);
  p.rcv = take(CL * MT * p.CS * 4, 16);    // partial sums received, one slot per CTA
  p.ex = take(MT * p.CS * 4, 16);          // E[prev] rows, own channels
  p.xh = take(MT * p.CS * 4, 16);
  p.us = take(MT * (p.CS + 1) * 4, 16);
  p.prev = take(MT * 8, 16);
  p.bars = take(64, 16);
  p.total = o;
  return p;
}

// byte offset of element (row, k) of an R-row swizzled matrix
__device__ __forceinline__ int swz(int row, int k, int R) {
  return ((k >> 6) * R + row) * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + ((k & 7) << 1);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---- cluster (distributed shared memory) helpers ----
__device__ __forceinline__ uint32_t mapa(uint32_t local, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// 16 bytes into a peer's shared memory; the bytes complete on the peer's mbarrier
__device__ __forceinline__ void st_async16(uint32_t raddr, uint4 v, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          raddr),
      "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait with cluster-scope acquire (the data came from peers)
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint32_t* err) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      const uint64_t now = ptx::globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > 500000000ull) {
        atomicOr(err, XP_ERR_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

struct Maps {
  CUtensorMap wg, wu, wdk, mix;
};

constexpr uint32_t TMEM_COLS = 512;    // gate 64 | up 64 | partial sums 256 (r <= 256)
constexpr uint32_t COL_G = 0, COL_U = 64, COL_P = 128;

template <int MTILES>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS, 1) latent_mma_kernel(
    const __grid_constant__ Maps maps, const int64_t* __restrict__ blk,
    const int64_t* __restrict__ am1, const float* __restrict__ xh, const float* __restrict__ E,
    bf16* __restrict__ lat, int N, int B, int r, int H, int V, uint32_t* err) {
  constexpr int MT = MTILES * 16;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (ptx::smem_u32(sm_raw) & 1023u)) & 1023u);
  const int q = (int)cg::this_cluster().block_rank();
  const int cid = blockIdx.x / CL, nclusters = gridDim.x / CL;
  const Plan P = make_plan(MT, r, H, B);
  const int CS = P.CS, HS = P.HS;
  const uint32_t s0 = ptx::smem_u32(sm);
  const uint32_t aWg = s0 + P.wg, aWu = s0 + P.wu, aU = s0 + P.ubuf;
  const uint32_t aUhi = aU, aUlo = aU + MT * r * 2;
  const uint32_t aAhi = s0 + P.ahi, aAlo = s0 + P.alo;
  const bf16* sMix = (const bf16*)(sm + P.mix);
  const float* sEx = (const float*)(sm + P.ex);
  const float* sXh = (const float*)(sm + P.xh);
  const float* sRcv = (const float*)(sm + P.rcv);
  float* sUs = (float*)(sm + P.us);
  int64_t* sPrev = (int64_t*)(sm + P.prev);
  const uint32_t bar_w = s0 + P.bars, bar_wd = bar_w + 8, bar_u = bar_w + 16, bar_p = bar_w + 24;
  const uint32_t bar_mma = bar_w + 32;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + P.bars + 40);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int nb = MT / B;                   // blocks per group
  const int groups = (N + nb - 1) / nb;
  const int ldp = CS + 1;
  const uint32_t u_bytes_in = (uint32_t)((CL - 1) * 2 * MT * CS * 2);
  const uint32_t p_bytes_in = (uint32_t)((CL - 1) * MT * CS * 4);
  const uint64_t pol = ptx::policy_evict_last();

  // ---- set-up: barriers, then the resident weight and mixer slices by TMA ----
  if (tid == 0) {
    ptx::mbar_init(bar_w, 1);
    ptx::mbar_init(bar_wd, 1);
    ptx::mbar_init(bar_u, 1);
    ptx::mbar_init(bar_p, 1);
    ptx::mbar_init(bar_mma, 1);
    ptx::fence_barrier_init();
    const int mparts = (P.mix_rows + 255) / 256, mbox = std::min(P.mix_rows, 256);
    ptx::mbar_arrive_expect_tx(bar_w, 2 * HS * r * 2 + mparts * mbox * CS * 2);
    for (int kc = 0; kc < r / 64; ++kc) {
      ptx::tma_load_2d(aWg + kc * HS * 128, &maps.wg, bar_w, kc * 64, q * HS, pol);
      ptx::tma_load_2d(aWu + kc * HS * 128, &maps.wu, bar_w, kc * 64, q * HS, pol);
    }
    for (int pt = 0; pt < mparts; ++pt)
      ptx::tma_load_2d(s0 + P.mix + pt * mbox * CS * 2, &maps.mix, bar_w, q * CS, pt * mbox, pol);
    // the first group's incoming u halves and partial sums
    ptx::mbar_arrive_expect_tx(bar_u, u_bytes_in);
    ptx::mbar_arrive_expect_tx(bar_p, p_bytes_in);
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(s_tmem), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  // peers push into this CTA only after its barriers exist
  ptx::tc_fence_before();
  cluster_arrive();
  ptx::pdl_wait();                         // blk (and xh) come from earlier kernels
  ptx::pdl_trigger();
  cluster_wait();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  {
    volatile int no_abort = 0;
    ptx::mbar_wait(bar_w, 0, &no_abort, err);
  }
  uint32_t mma_phase = 0;
  // TMEM readers: warps whose lane quadrant holds real rows (MT <= 64), two column halves
  const bool reader = (warp & 3) * 32 < MT;
  const int quad = warp & 3, half = warp >> 2;
  const int trow = quad * 32 + lane;        // this thread's row when it is a reader

  int it = 0;
  for (int grp = cid; grp < groups; grp += nclusters, ++it) {
    const uint32_t ph = it & 1;
    const int n0 = grp * nb;
    const int rows = std::min(nb, N - n0) * B;   // valid rows of this group

    // ---- 1. token ids, then E[prev] and xh for the own channels ----
    for (int m = tid; m < MT; m += THREADS) {
      int64_t t = 0;
      if (m < rows) {
        const int n = n0 + m / B, b = m % B;
        t = checked_token(b == 0 ? am1[n] : blk[(int64_t)n * B + b - 1], V, err);
      }
      sPrev[m] = t;
    }
    __syncthreads();
    {
      const int xc = CS / 4;                   // 16-byte chunks per row and table
      for (int i = tid; i < MT * 2 * xc; i += THREADS) {
        const int m = i / (2 * xc), c = i % (2 * xc);
        const int cc = c % xc;
        const bool is_e = c < xc;
        const uint32_t dst = s0 + (is_e ? P.ex : P.xh) + (m * CS + cc * 4) * 4;
        if (m < rows) {
          const float* src = is_e ? E + sPrev[m] * r + q * CS + cc * 4
                                  : xh + ((int64_t)(n0 * B + m)) * r + q * CS + cc * 4;
          cp_async16(dst, src);
        } else {
          *reinterpret_cast<uint4*>(sm + (dst - s0)) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- 2. x = xh + E[prev]; u = per-channel causal mix (fp32); push u hi/lo ----
    for (int i = tid; i < MT * CS; i += THREADS) {
      const int m = i / CS, c = i % CS;
      sUs[m * ldp + c] = sXh[m * CS + c] + sEx[m * CS + c];
    }
    __syncthreads();
    // the previous group's peers are done reading this CTA's buffers, and it theirs
    if (it > 0) cluster_wait();
    float uown[8];
    int own_m = -1, own_c0 = 0;
    for (int w = tid; w < MT * CS / 8; w += THREADS) {
      const int m = w / (CS / 8), c0 = (w % (CS / 8)) * 8;
      float u[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) u[e] = 0.f;
      if (m < rows) {
        const int bl = m / B, b = m % B;
        for (int j = 0; j < B; ++j) {
          const uint4 mv = *reinterpret_cast<const uint4*>(sMix + (b * B + j) * CS + c0);
          const bf16* mj = reinterpret_cast<const bf16*>(&mv);
          const float* xj = sUs + (bl * B + j) * ldp + c0;
#pragma unroll
          for (int e = 0; e < 8; ++e) u[e] = fmaf(__bfloat162float(mj[e]), xj[e], u[e]);
        }
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(u[e], u[e + 1]);
        const float2 hf = __bfloat1622float2(h2);
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(u[e] - hf.x, u[e + 1] - hf.y);
        hi[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
        lo[e / 2] = *reinterpret_cast<const uint32_t*>(&l2);
      }
      const uint4 vh = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      const uint4 vl = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      const int off = swz(m, q * CS + c0, MT);
      *reinterpret_cast<uint4*>(sm + P.ubuf + off) = vh;
      *reinterpret_cast<uint4*>(sm + P.ubuf + MT * r * 2 + off) = vl;
#pragma unroll 1
      for (int dp = 1; dp < CL; ++dp) {
        const int p = (q + dp) % CL;
        const uint32_t rb = mapa(bar_u, p);
        st_async16(mapa(aUhi + off, p), vh, rb);
        st_async16(mapa(aUlo + off, p), vl, rb);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) uown[e] = u[e];
      own_m = m;
      own_c0 = c0;
    }
    __syncthreads();                         // every x read before u (fp32) replaces it
    if (own_m >= 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sUs[own_m * ldp + own_c0 + e] = uown[e];
    }
    __syncthreads();
    mbar_wait_cluster(bar_u, ph, err);

    // ---- 3. SwiGLU on own hidden units from u = hi + lo (tcgen05, fp32 in TMEM) ----
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // u seen by the MMA
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
      constexpr uint32_t ID64 = ptx::idesc_bf16_f32(128, 64);
      int first = 1;
      for (int kc = 0; kc < r / 64; ++kc)
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t ko = kc * MT * 128 + kk * 32;
          const uint64_t bg = ptx::sw128_desc(aWg + kc * HS * 128 + kk * 32);
          const uint64_t bu = ptx::sw128_desc(aWu + kc * HS * 128 + kk * 32);
          const uint64_t ah = ptx::sw128_desc(aUhi + ko), al = ptx::sw128_desc(aUlo + ko);
          ptx::mma_bf16(tmem + COL_G, ah, bg, ID64, !first);
          ptx::mma_bf16(tmem + COL_U, ah, bu, ID64, !first);
          ptx::mma_bf16(tmem + COL_G, al, bg, ID64, 1);
          ptx::mma_bf16(tmem + COL_U, al, bu, ID64, 1);
          first = 0;
        }
      ptx::mma_commit(bar_mma);
    }
    {
      volatile int no_abort = 0;
      ptx::mbar_wait(bar_mma, mma_phase, &no_abort, err);
      mma_phase ^= 1;
    }
    ptx::tc_fence_after();
    if (reader) {
      // each reader thread: its row, 32 of the 64 own hidden units (gate and up)
      uint32_t g[32], v[32];
      const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + half * 32;
      ptx::tmem_ld32(ta + COL_G, g);
      ptx::tmem_ld32(ta + COL_U, v);
      ptx::tmem_wait_ld();
      if (trow < MT) {
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int k = c8 * 8 + e;
            const float a0 = silu(__uint_as_float(g[k])) * __uint_as_float(v[k]);
            const float a1 = silu(__uint_as_float(g[k + 1])) * __uint_as_float(v[k + 1]);
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(a0, a1);
            const float2 hf = __bfloat1622float2(h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(a0 - hf.x, a1 - hf.y);
            hw[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
            lw[e / 2] = *reinterpret_cast<const uint32_t*>(&l2);
          }
          const int off = swz(trow, half * 32 + c8 * 8, MT);
          *reinterpret_cast<uint4*>(sm + P.ahi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(sm + P.alo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    }
    ptx::tc_fence_before();
    __syncthreads();                         // u is dead: w_down's slice may overwrite it
    if (tid == 0) {
      ptx::mbar_arrive_expect_tx(bar_wd, r * HS * 2);
      const int rbox = std::min(r, 256);
      for (int kc = 0; kc < HS / 64; ++kc)
        for (int rp = 0; rp < r / rbox; ++rp)
          ptx::tma_load_2d(aU + (kc * r + rp * rbox) * 128, &maps.wdk, bar_wd, q * HS + kc * 64,
                           rp * rbox, pol);
    }
    {
      volatile int no_abort = 0;
      ptx::mbar_wait(bar_wd, ph, &no_abort, err);
    }

    // ---- 4. partial down projection over own units (tcgen05), pushed to each owner ----
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // activations seen by the MMA
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint32_t idn = ptx::idesc_bf16_f32(128, r);
      for (int kc = 0; kc < HS / 64; ++kc)
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bw = ptx::sw128_desc(aU + kc * r * 128 + kk * 32);
          const uint32_t ko = kc * MT * 128 + kk * 32;
          ptx::mma_bf16(tmem + COL_P, ptx::sw128_desc(aAhi + ko), bw, idn, (kc | kk) != 0);
          ptx::mma_bf16(tmem + COL_P, ptx::sw128_desc(aAlo + ko), bw, idn, 1);
        }
      ptx::mma_commit(bar_mma);
    }
    {
      volatile int no_abort = 0;
      ptx::mbar_wait(bar_mma, mma_phase, &no_abort, err);
      mma_phase ^= 1;
    }
    ptx::tc_fence_after();
    if (reader) {
      // each reader thread: its row, channels [half*r/2, (half+1)*r/2), 32 at a time
      const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + COL_P;
      for (int c32 = half * (r / 64); c32 < (half + 1) * (r / 64); ++c32) {
        uint32_t pv[32];
        ptx::tmem_ld32(ta + c32 * 32, pv);
        ptx::tmem_wait_ld();
        if (trow < MT) {
          // channels [c32*32, c32*32+32) belong to owner c32*32 / CS
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const int c = c32 * 32 + c4 * 4;
            const int owner = c / CS, cl = c - owner * CS;
            const uint32_t o = s0 + P.rcv + (uint32_t)(((q * MT + trow) * CS + cl) * 4);
            const uint4 v4 = make_uint4(pv[c4 * 4], pv[c4 * 4 + 1], pv[c4 * 4 + 2], pv[c4 * 4 + 3]);
            if (owner == q)
              *reinterpret_cast<uint4*>(sm + (o - s0)) = v4;
            else
              st_async16(mapa(o, owner), v4, mapa(bar_p, owner));
          }
        }
      }
    }
    ptx::tc_fence_before();
    __syncthreads();
    mbar_wait_cluster(bar_p, ph, err);

    // ---- 5. lat (own channels) = u + sum_p partial_p, p = 0..7 in order ----
    for (int i = tid; i < MT * CS; i += THREADS) {
      const int m = i / CS, c = i % CS;
      if (m < rows && (m % B) != 0) {
        float v = sUs[m * ldp + c];
#pragma unroll
        for (int p = 0; p < CL; ++p) v += sRcv[(p * MT + m) * CS + c];
        const int n = n0 + m / B, b = m % B;
        lat[((int64_t)n * (B - 1) + b - 1) * r + q * CS + c] = __float2bfloat16_rn(v);
      }
    }
    __syncthreads();
    // arm the next group's receive barriers, then tell the peers this CTA's
    // buffers (u, w_down slice, partial slots) are free again
    if (tid == 0 && grp + nclusters < groups) {
      ptx::mbar_arrive_expect_tx(bar_u, u_bytes_in);
      ptx::mbar_arrive_expect_tx(bar_p, p_bytes_in);
    }
    cluster_arrive();
  }
  cluster_wait();   // no CTA leaves while a peer may still push into it
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

int g_max_clusters[2] = {0, 0};   // co-resident clusters per variant (queried once)

size_t smem_bytes(int MT, int r, int H, int B) {
  return (size_t)make_plan(MT, r, H, B).total + 1024;
}

template <int MTILES>
int max_clusters(int smem) {
  int& cached = g_max_clusters[MTILES - 2];
  if (cached > 0) return cached;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaFuncSetAttribute(latent_mma_kernel<MTILES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, latent_mma_kernel<MTILES>, &cfg) != cudaSuccess || n <= 0)
    n = 1;
  cached = n;
  return n;
}

template <int MTILES>
cudaError_t launch(const xp_head* h, const int64_t* blk, const int64_t* am1, const float* xh,
                   int N, void* lat, cudaStream_t s) {
  const int MT = MTILES * 16;
  const int smem = (int)smem_bytes(MT, h->r, h->H, h->B);
  cudaError_t e = cudaFuncSetAttribute(latent_mma_kernel<MTILES>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nb = MT / h->B;
  const int groups = (N + nb - 1) / nb;
  const int clusters = std::min(groups, max_clusters<MTILES>(smem));
  const Maps maps = {h->tm_wg, h->tm_wu, h->tm_wd, h->tm_mixT};
  e = xp_launch_pdl(latent_mma_kernel<MTILES>, dim3(clusters * CL), dim3(THREADS), (size_t)smem,
                    s, maps, blk, am1, xh, (const float*)h->E, (bf16*)lat, N, h->B, h->r, h->H,
                    h->V, h->err);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool xp_latent_mma_ok(int r, int H, int B, xp_dtype dt) {
  if (dt != XP_BF16 || B < 2 || B > 32) return false;
  if (r != 64 && r != 128 && r != 256) return false;      // r/8 channels: 8, 16 or 32
  if (H != 8 * 64) return false;                          // 64 own units: one MMA N-tile
  return smem_bytes(48, r, H, B) <= 227 * 1024;
}

// Tensor maps of the weight and mixer slices (2-D, bf16; weights 128B-swizzled).
bool xp_latent_mma_maps(xp_head* h) {
  xp_encode_tiled_fn fn = xp_get_encode_tiled();
  if (!fn) return false;
  const int r = h->r, H = h->H, B = h->B, CS = r / CL, HS = H / CL;
  auto enc = [&](CUtensorMap* m, const void* ptr, int rows, int cols, int box_c, int box_r,
                 bool swz128) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_c, (cuuint32_t)box_r};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swz128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
  };
  return enc(&h->tm_wg, h->w_gate, H, r, 64, HS, true) &&
         enc(&h->tm_wu, h->w_up, H, r, 64, HS, true) &&
         enc(&h->tm_wd, h->w_down, r, H, 64, std::min(r, 256), true) &&
         enc(&h->tm_mixT, h->mixT, B * B, r, CS, std::min(B * B, 256), false);
}

cudaError_t xp_launch_latent_mma(const xp_head* h, const int64_t* blk, const int64_t* am1,
                                 const float* xh, int N, void* lat, cudaStream_t s) {
  // 32-row groups while they fit in one wave of co-resident clusters, else 48-row groups
  const int groups32 = (N + 32 / h->B - 1) / (32 / h->B);
  if (groups32 <= max_clusters<2>((int)smem_bytes(32, h->r, h->H, h->B)))
    return launch<2>(h, blk, am1, xh, N, lat, s);
  return launch<3>(h, blk, am1, xh, N, lat, s);
}
