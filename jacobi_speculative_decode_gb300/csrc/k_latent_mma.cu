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
//   3. a = silu(u w_gate[own]^T) * (u w_up[own]^T) from hi and lo (mma.sync)
//   4. partial = a w_down[:, own]^T for ALL channels (w_down's column slice
//      arrives by TMA into the u buffer, dead by then); each 8-channel piece is
//      pushed to the CTA owning those channels
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
constexpr int NW = THREADS / 32;

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
__device__ __forceinline__ void ldm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldm_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

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
__device__ __forceinline__ void st_async8(uint32_t raddr, float a, float b, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(raddr),
      "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(rbar)
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
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g8 = lane / 4, t4 = lane % 4;
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
  // peers push into this CTA only after its barriers exist
  cluster_arrive();
  ptx::pdl_wait();                         // blk (and xh) come from earlier kernels
  ptx::pdl_trigger();
  cluster_wait();
  {
    volatile int no_abort = 0;
    ptx::mbar_wait(bar_w, 0, &no_abort, err);
  }

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

    // ---- 3. SwiGLU on own hidden units from u = hi + lo ----
    for (int nt = warp; nt < HS / 8; nt += NW) {
      float g0[MTILES][4] = {}, g1[MTILES][4] = {}, v0[MTILES][4] = {}, v1[MTILES][4] = {};
      const int ar = lane % 16, ak = (lane / 16) * 8;
      const int br = nt * 8 + (lane % 8), bk = ((lane / 8) % 2) * 8;
      for (int k = 0; k < r; k += 16) {
        uint32_t bg[2], bu[2];
        const int bo = swz(br, k + bk, HS);
        ldm_x2(bg, aWg + bo);
        ldm_x2(bu, aWu + bo);
#pragma unroll
        for (int i = 0; i < MTILES; ++i) {
          uint32_t ah[4], al[4];
          const int ao = swz(i * 16 + ar, k + ak, MT);
          ldm_x4(ah, aUhi + ao);
          ldm_x4(al, aUlo + ao);
          mma16816(g0[i], ah, bg);
          mma16816(v0[i], ah, bu);
          mma16816(g1[i], al, bg);
          mma16816(v1[i], al, bu);
        }
      }
#pragma unroll
      for (int i = 0; i < MTILES; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = i * 16 + g8 + (e >= 2 ? 8 : 0);
          const int hh = nt * 8 + 2 * t4 + (e & 1);
          const float a = silu(g0[i][e] + g1[i][e]) * (v0[i][e] + v1[i][e]);
          const bf16 ah = __float2bfloat16_rn(a);
          const int off = swz(m, hh, MT);
          *reinterpret_cast<bf16*>(sm + P.ahi + off) = ah;
          *reinterpret_cast<bf16*>(sm + P.alo + off) = __float2bfloat16_rn(a - __bfloat162float(ah));
        }
    }
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

    // ---- 4. partial down projection over own units, pushed to each channel's owner ----
    for (int nt = warp; nt < r / 8; nt += NW) {
      float c0[MTILES][4] = {}, c1[MTILES][4] = {};
      const int ar = lane % 16, ak = (lane / 16) * 8;
      const int br = nt * 8 + (lane % 8), bk = ((lane / 8) % 2) * 8;
      for (int k = 0; k < HS; k += 16) {
        uint32_t bw[2];
        ldm_x2(bw, aU + swz(br, k + bk, r));
#pragma unroll
        for (int i = 0; i < MTILES; ++i) {
          uint32_t ah[4], al[4];
          const int ao = swz(i * 16 + ar, k + ak, MT);
          ldm_x4(ah, aAhi + ao);
          ldm_x4(al, aAlo + ao);
          mma16816(c0[i], ah, bw);
          mma16816(c1[i], al, bw);
        }
      }
      const int owner = nt * 8 / CS, cl0 = nt * 8 - owner * CS;
      const uint32_t slot = s0 + P.rcv + (uint32_t)(q * MT * CS * 4);   // my slot at the owner
      const uint32_t rb = mapa(bar_p, owner);
#pragma unroll
      for (int i = 0; i < MTILES; ++i)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int m = i * 16 + g8 + hh * 8;
          const float a = c0[i][2 * hh] + c1[i][2 * hh];
          const float b = c0[i][2 * hh + 1] + c1[i][2 * hh + 1];
          const uint32_t o = slot + (uint32_t)((m * CS + cl0 + 2 * t4) * 4);
          if (owner == q)
            *reinterpret_cast<float2*>(sm + (o - s0)) = make_float2(a, b);
          else
            st_async8(mapa(o, owner), a, b, rb);
        }
    }
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
  if (H % (8 * 64) != 0 || H > 1024) return false;        // own units in 64-wide chunks
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
