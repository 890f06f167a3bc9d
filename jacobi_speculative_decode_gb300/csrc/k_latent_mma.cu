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
// owns channels [q*CS, (q+1)*CS), CS = r/8 (mixer, residual, output) and hidden
// units [q*64, (q+1)*64) (SwiGLU).  Per group of MT rows (whole blocks):
//   1. gather E rows and xh for the own channels (cp.async), x = xh + E[prev]
//   2. u = per-channel causal mix of x (fp32), split into bf16 hi + lo
//      (u = hi + lo to ~2^-17) and sent to every CTA of the cluster (itself
//      included) with one bulk shared-to-shared copy per half and CTA; in the
//      receivers the slice of CTA p is K-chunk p of a 64B-swizzled operand
//   3. [gate | up] = u [w_gate ; w_up][own units]^T from hi and lo: tcgen05.mma
//      (M = 128 rows, of which the group's MT are real, N = 128) into TMEM;
//      a = silu(gate) * up, kept as bf16 hi + lo
//   4. partial = a w_down[:, own units]^T for ALL r channels, tcgen05.mma again
//      (w_down's column slice arrives by TMA into the u buffer, dead by then);
//      each CS-channel piece goes to the CTA owning it by bulk copy
//   5. lat = u + the 8 partials of the own channels, added in a fixed order
// The only cluster-wide barrier per group is a split arrive/wait that keeps a
// CTA from sending into buffers a peer is still reading.
//
// Shared-memory operand layouts (what the TMA writes and tcgen05 reads):
//   128B swizzle: element (row, k) of an R-row matrix, 64-column chunks, at
//     (k/64)*R*128 + row*128 + ((((k%64)/8) ^ (row%8))*16) + (k%8)*2
//   64B swizzle (the exchanged u): chunk p holds columns [32p, 32p+32) of MT rows,
//     (row, c) at p*MT*64 + row*64 + (((c/8) ^ ((row/2)%4))*16) + (c%8)*2
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
constexpr int HS = 64;         // own hidden units (H = 512)
constexpr int CS = 32;         // own channels (r = 256)
constexpr int R = CL * CS;     // latent rank handled by this kernel

struct Plan {                  // byte offsets into dynamic shared memory
  int MT;
  int wgu, mix, ubuf, uout, ahi, alo, rcv, ex, xh, us, prev, bars;
  int mix_rows;
  int total;
};

__host__ __device__ inline Plan make_plan(int MT, int B) {
  Plan p;
  p.MT = MT;
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
  p.wgu = take((R / 64) * 128 * 128, 1024);     // [w_gate; w_up] own rows, 128B swizzle
  p.mix = take(mparts * mbox * CS * 2, 1024);
  // u hi + lo (64B swizzle, 8 chunks each), later w_down[:, own] (R rows x 64, 128B
  // swizzle), later the outgoing partial sums ([owner][MT][CS] fp32)
  p.ubuf = take(std::max(std::max(2 * MT * R * 2, R * HS * 2), CL * MT * CS * 4), 1024);
  p.uout = take(2 * MT * 64, 1024);             // own u slice, hi then lo
  p.ahi = take(MT * 128, 1024);
  p.alo = take(MT * 128, 1024);
  p.rcv = take(CL * MT * CS * 4, 16);           // partial sums received, one slot per CTA
  p.ex = take(MT * CS * 4, 16);                 // E[prev] rows, own channels
  p.xh = take(MT * CS * 4, 16);
  p.us = take(MT * (CS + 1) * 4, 16);
  p.prev = take(MT * 8, 16);
  p.bars = take(64, 16);
  p.total = o;
  return p;
}

__device__ __forceinline__ int swz128(int row, int k, int Rr) {
  return ((k >> 6) * Rr + row) * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + ((k & 7) << 1);
}
__device__ __forceinline__ int swz64(int row, int c) {      // within one 32-column chunk
  return row * 64 + ((((c >> 3) ^ ((row >> 1) & 3))) << 4) + ((c & 7) << 1);
}
// 16-byte chunk k of row m of a [rows][32] fp32 tile, rotated so that eight
// consecutive rows writing the same logical chunk hit eight different banks
__device__ __forceinline__ int rot32(int m, int k) { return m * 128 + (((k + m) & 7) << 4); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint32_t mapa(uint32_t local, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
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
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

struct Maps {
  CUtensorMap wg, wu, wdk, mix;
};

constexpr uint32_t TMEM_COLS = 512;    // [gate | up] 128 | partial sums 256
constexpr uint32_t COL_GU = 0, COL_P = 128;

template <int MTILES>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS, 1) latent_mma_kernel(
    const __grid_constant__ Maps maps, const int64_t* __restrict__ blk,
    const int64_t* __restrict__ am1, const float* __restrict__ xh, const float* __restrict__ E,
    bf16* __restrict__ lat, int N, int B, int V, uint32_t* err) {
  constexpr int MT = MTILES * 16;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (ptx::smem_u32(sm_raw) & 1023u)) & 1023u);
  const int q = (int)cg::this_cluster().block_rank();
  const int cid = blockIdx.x / CL, nclusters = gridDim.x / CL;
  const Plan P = make_plan(MT, B);
  const uint32_t s0 = ptx::smem_u32(sm);
  const uint32_t aW = s0 + P.wgu, aU = s0 + P.ubuf, aUo = s0 + P.uout;
  const uint32_t aUhi = aU, aUlo = aU + MT * R * 2;
  const uint32_t aAhi = s0 + P.ahi, aAlo = s0 + P.alo;
  const bf16* sMix = (const bf16*)(sm + P.mix);
  const float* sEx = (const float*)(sm + P.ex);
  const float* sXh = (const float*)(sm + P.xh);
  const uint8_t* sRcv = sm + P.rcv;
  const uint8_t* sStage = sm + P.ubuf;     // outgoing partial sums, [owner][MT rows][CS]
  float* sUs = (float*)(sm + P.us);
  int64_t* sPrev = (int64_t*)(sm + P.prev);
  const uint32_t bar_w = s0 + P.bars, bar_wd = bar_w + 8, bar_u = bar_w + 16, bar_p = bar_w + 24;
  const uint32_t bar_mma = bar_w + 32;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + P.bars + 40);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int nb = MT / B;                   // blocks per group
  const int groups = (N + nb - 1) / nb;
  const int ldp = CS + 1;
  const uint32_t slice = MT * 64;          // bytes of one u half of one CTA
  const uint32_t u_bytes_in = (uint32_t)(CL * 2 * slice);
  const uint32_t p_bytes_in = (uint32_t)((CL - 1) * MT * CS * 4);
  const uint64_t pol = ptx::policy_evict_last();

  // ---- set-up: barriers, TMEM, then the resident weight and mixer slices by TMA ----
  if (tid == 0) {
    ptx::mbar_init(bar_w, 1);
    ptx::mbar_init(bar_wd, 1);
    ptx::mbar_init(bar_u, 1);
    ptx::mbar_init(bar_p, 1);
    ptx::mbar_init(bar_mma, 1);
    ptx::fence_barrier_init();
    const int mparts = (P.mix_rows + 255) / 256, mbox = std::min(P.mix_rows, 256);
    ptx::mbar_arrive_expect_tx(bar_w, 2 * HS * R * 2 + mparts * mbox * CS * 2);
    for (int kc = 0; kc < R / 64; ++kc) {
      ptx::tma_load_2d(aW + kc * 16384, &maps.wg, bar_w, kc * 64, q * HS, pol);
      ptx::tma_load_2d(aW + kc * 16384 + 8192, &maps.wu, bar_w, kc * 64, q * HS, pol);
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
  // peers send into this CTA only after its barriers exist
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
    for (int i = tid; i < MT * 2 * (CS / 4); i += THREADS) {
      const int m = i / (2 * (CS / 4)), c = i % (2 * (CS / 4));
      const int cc = c % (CS / 4);
      const bool is_e = c < CS / 4;
      const uint32_t dst = s0 + (is_e ? P.ex : P.xh) + (m * CS + cc * 4) * 4;
      if (m < rows) {
        const float* src = is_e ? E + sPrev[m] * R + q * CS + cc * 4
                                : xh + ((int64_t)(n0 * B + m)) * R + q * CS + cc * 4;
        cp_async16(dst, src);
      } else {
        *reinterpret_cast<uint4*>(sm + (dst - s0)) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- 2. x = xh + E[prev]; u = per-channel causal mix (fp32); send u hi/lo ----
    for (int i = tid; i < MT * CS; i += THREADS) {
      const int m = i / CS, c = i % CS;
      sUs[m * ldp + c] = sXh[m * CS + c] + sEx[m * CS + c];
    }
    __syncthreads();
    // the previous group's peers are done reading this CTA's buffers, and it theirs
    if (it > 0) cluster_wait();
    float uown[8];
    const int wm = tid / (CS / 8), wc0 = (tid % (CS / 8)) * 8;   // one 8-channel run each
    const bool mixer = tid < MT * CS / 8;
    if (mixer) {
#pragma unroll
      for (int e = 0; e < 8; ++e) uown[e] = 0.f;
      if (wm < rows) {
        const int bl = wm / B, b = wm % B;
#pragma unroll 4
        for (int j = 0; j < B; ++j) {
          const uint4 mv = *reinterpret_cast<const uint4*>(sMix + (b * B + j) * CS + wc0);
          const bf16* mj = reinterpret_cast<const bf16*>(&mv);
          const float* xj = sUs + (bl * B + j) * ldp + wc0;
#pragma unroll
          for (int e = 0; e < 8; ++e) uown[e] = fmaf(__bfloat162float(mj[e]), xj[e], uown[e]);
        }
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(uown[e], uown[e + 1]);
        const float2 hf = __bfloat1622float2(h2);
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(uown[e] - hf.x, uown[e + 1] - hf.y);
        hi[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
        lo[e / 2] = *reinterpret_cast<const uint32_t*>(&l2);
      }
      const int off = swz64(wm, wc0);
      *reinterpret_cast<uint4*>(sm + P.uout + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sm + P.uout + slice + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    fence_async_smem();                    // the bulk copies read u_out
    __syncthreads();                       // every x read before u (fp32) replaces it
    if (tid == 0) {
      for (int dp = 0; dp < CL; ++dp) {
        const int p = (q + dp) % CL;       // itself first
        const uint32_t rb = mapa(bar_u, p);
        ptx::bulk_copy_to_peer(mapa(aUhi + q * slice, p), aUo, slice, rb);
        ptx::bulk_copy_to_peer(mapa(aUlo + q * slice, p), aUo + slice, slice, rb);
      }
    }
    if (mixer) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sUs[wm * ldp + wc0 + e] = uown[e];
    }
    mbar_wait_cluster(bar_u, ph, err);

    // ---- 3. [gate | up] from u = hi + lo (tcgen05, fp32 in TMEM); a = silu(g) * up ----
    if (tid == 0) {
      ptx::tc_fence_after();
      constexpr uint32_t ID = ptx::idesc_bf16_f32(128, 128);
      for (int s = 0; s < R / 16; ++s) {
        const uint64_t bw = ptx::sw128_desc(aW + (s / 4) * 16384 + (s % 4) * 32);
        const uint32_t ao = (s / 2) * slice + (s % 2) * 32;
        ptx::mma_bf16(tmem + COL_GU, ptx::sw64_desc(aUhi + ao), bw, ID, s != 0);
        ptx::mma_bf16(tmem + COL_GU, ptx::sw64_desc(aUlo + ao), bw, ID, 1);
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
      const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + COL_GU + half * 32;
      ptx::tmem_ld32(ta, g);
      ptx::tmem_ld32(ta + HS, v);
      ptx::tmem_wait_ld();
      if (trow < MT) {
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int k = c8 * 8 + e;
            const float a0 = silu_fast(__uint_as_float(g[k])) * __uint_as_float(v[k]);
            const float a1 = silu_fast(__uint_as_float(g[k + 1])) * __uint_as_float(v[k + 1]);
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(a0, a1);
            const float2 hf = __bfloat1622float2(h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(a0 - hf.x, a1 - hf.y);
            hw[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
            lw[e / 2] = *reinterpret_cast<const uint32_t*>(&l2);
          }
          const int off = swz128(trow, half * 32 + c8 * 8, MT);
          *reinterpret_cast<uint4*>(sm + P.ahi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(sm + P.alo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    }
    ptx::tc_fence_before();
    fence_async_smem();                    // activations seen by the next MMA
    __syncthreads();                       // u is dead: w_down's slice may overwrite it
    if (tid == 0) {
      ptx::mbar_arrive_expect_tx(bar_wd, R * HS * 2);
      ptx::tma_load_2d(aU, &maps.wdk, bar_wd, q * HS, 0, pol);
    }
    {
      volatile int no_abort = 0;
      ptx::mbar_wait(bar_wd, ph, &no_abort, err);
    }

    // ---- 4. partial down projection over own units (tcgen05), sent to each owner ----
    if (tid == 0) {
      ptx::tc_fence_after();
      constexpr uint32_t ID = ptx::idesc_bf16_f32(128, R);
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bw = ptx::sw128_desc(aU + kk * 32);
        ptx::mma_bf16(tmem + COL_P, ptx::sw128_desc(aAhi + kk * 32), bw, ID, kk != 0);
        ptx::mma_bf16(tmem + COL_P, ptx::sw128_desc(aAlo + kk * 32), bw, ID, 1);
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
      // each reader thread: its row, owners [4*half, 4*half+4) (CS = 32 channels each)
      const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + COL_P;
#pragma unroll 1
      for (int p = half * 4; p < half * 4 + 4; ++p) {
        uint32_t pv[32];
        ptx::tmem_ld32(ta + p * CS, pv);
        ptx::tmem_wait_ld();
        if (trow < MT) {
          uint8_t* dst = sm + P.ubuf + p * MT * CS * 4;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4*>(dst + rot32(trow, k)) =
                make_uint4(pv[4 * k], pv[4 * k + 1], pv[4 * k + 2], pv[4 * k + 3]);
        }
      }
    }
    ptx::tc_fence_before();
    fence_async_smem();                    // the bulk copies read the staged partial sums
    __syncthreads();
    if (tid == 0) {
      for (int dp = 1; dp < CL; ++dp) {
        const int p = (q + dp) % CL;
        ptx::bulk_copy_to_peer(mapa(s0 + P.rcv + q * MT * CS * 4, p), aU + p * MT * CS * 4,
                               MT * CS * 4, mapa(bar_p, p));
      }
    }
    mbar_wait_cluster(bar_p, ph, err);

    // ---- 5. lat (own channels) = u + sum_p partial_p, p = 0..7 in order ----
    for (int i = tid; i < MT * CS; i += THREADS) {
      const int m = i / CS, c = i % CS;
      if (m < rows && (m % B) != 0) {
        float v = sUs[m * ldp + c];
        const int o = rot32(m, c >> 2) + (c & 3) * 4;
#pragma unroll
        for (int p = 0; p < CL; ++p) {
          const uint8_t* src = (p == q) ? sStage + q * MT * CS * 4 : sRcv + p * MT * CS * 4;
          v += *reinterpret_cast<const float*>(src + o);
        }
        const int n = n0 + m / B, b = m % B;
        lat[((int64_t)n * (B - 1) + b - 1) * R + q * CS + c] = __float2bfloat16_rn(v);
      }
    }
    __syncthreads();
    // arm the next group's receive barriers, then tell the peers this CTA's
    // buffers (u, w_down slice, staged and received partial sums) are free again
    if (tid == 0 && grp + nclusters < groups) {
      ptx::mbar_arrive_expect_tx(bar_u, u_bytes_in);
      ptx::mbar_arrive_expect_tx(bar_p, p_bytes_in);
    }
    cluster_arrive();
  }
  cluster_wait();   // no CTA leaves while a peer may still send into it
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

int g_max_clusters[2] = {0, 0};   // co-resident clusters per variant (queried once)

size_t smem_bytes(int MT, int B) { return (size_t)make_plan(MT, B).total + 1024; }

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
  const int smem = (int)smem_bytes(MT, h->B);
  cudaError_t e = cudaFuncSetAttribute(latent_mma_kernel<MTILES>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nb = MT / h->B;
  const int groups = (N + nb - 1) / nb;
  const int clusters = std::min(groups, max_clusters<MTILES>(smem));
  const Maps maps = {h->tm_wg, h->tm_wu, h->tm_wd, h->tm_mixT};
  e = xp_launch_pdl(latent_mma_kernel<MTILES>, dim3(clusters * CL), dim3(THREADS), (size_t)smem,
                    s, maps, blk, am1, xh, (const float*)h->E, (bf16*)lat, N, h->B, h->V, h->err);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool xp_latent_mma_ok(int r, int H, int B, xp_dtype dt) {
  // the production shape of the head: r = 256 (32 channels per CTA), H = 512 (64 units)
  if (dt != XP_BF16 || B < 2 || B > 32 || r != R || H != CL * HS) return false;
  return smem_bytes(48, B) <= 227 * 1024;
}

// Tensor maps of the weight and mixer slices (2-D, bf16).
bool xp_latent_mma_maps(xp_head* h) {
  xp_encode_tiled_fn fn = xp_get_encode_tiled();
  if (!fn) return false;
  const int B = h->B;
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
  return enc(&h->tm_wg, h->w_gate, CL * HS, R, 64, HS, true) &&
         enc(&h->tm_wu, h->w_up, CL * HS, R, 64, HS, true) &&
         enc(&h->tm_wd, h->w_down, R, CL * HS, 64, R, true) &&
         enc(&h->tm_mixT, h->mixT, B * B, R, CS, std::min(B * B, 256), false);
}

cudaError_t xp_launch_latent_mma(const xp_head* h, const int64_t* blk, const int64_t* am1,
                                 const float* xh, int N, void* lat, cudaStream_t s) {
  // 32-row groups while they fit in one wave of co-resident clusters, else 48-row groups
  const int groups32 = (N + 32 / h->B - 1) / (32 / h->B);
  if (groups32 <= max_clusters<2>((int)smem_bytes(32, h->B)))
    return launch<2>(h, blk, am1, xh, N, lat, s);
  return launch<3>(h, blk, am1, xh, N, lat, s);
}
