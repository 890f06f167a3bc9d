// Latent stage of one pass on tensor cores, persistent 8-CTA clusters
// (xpress kernels page, _xpress_latent_kernel; qwen3_xpress page, _refine_latent):
//   prev[0] = am1[n], prev[b] = blk[n, b-1]
//   x[b]    = xh[n, b] + w_lat w1[prev[b]]
//   u[b, c] = sum_j mix[c, b, j] x[j, c]            (stored mixer is lower-triangular)
//   lat[b]  = u[b] + w_down (silu(w_gate u[b]) * (w_up u[b]))      for b = 1..B-1
//
// The cluster splits the work by output features so each CTA holds only 1/8 of
// the weights: CTA q owns channels [q*r/8, (q+1)*r/8) of the in_proj and
// w_down products and hidden units [q*H/8, (q+1)*H/8) of the SwiGLU.  Its
// weight and mixer slices arrive by TMA once, before the kernel waits on the
// previous pass, and stay in shared memory while the cluster walks over groups
// of 32 rows (whole blocks).  Per group the embeddings and the xh slice arrive
// by cp.async.  Products use mma.sync m16n8k16 (bf16 in, fp32 accumulate):
//   x slice   = emb . w_lat[own channels]^T
//   u         = per-channel causal mix of x (fp32); the full u is exchanged over
//               distributed shared memory as a bf16 hi + lo pair (u = hi + lo to
//               ~2^-17), so the SwiGLU sees u, not bf16(u)
//   a slice   = silu(u . w_gate[own units]^T) * (u . w_up[own units]^T), kept as hi + lo
//   partial   = a slice . w_down[:, own units]^T for ALL r channels (a K split)
//   lat       = u + sum over the 8 CTAs of their partials for the own channels,
//               added in a fixed order (deterministic), read over DSMEM.
//
// Every bf16 matrix in shared memory uses the TMA 128-byte-swizzle layout in
// 64-column chunks: element (row, k) of an R-row matrix lives at
//   (k / 64) * R * 128 + row * 128 + ((((k % 64) / 8) ^ (row % 8)) * 16) + (k % 8) * 2
// so ldmatrix row reads hit eight distinct bank groups without padding.
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

struct Plan {                  // shapes and byte offsets into dynamic shared memory
  int CS, HS;
  int nt1, ks1;                // in_proj: n-tiles of the CTA's channels, K splits
  int wlat, wg, wu, wdk, mix, ep, uhi, ulo, ahi, alo, xh, part, us, prev, bar;
  int mix_rows, pp;            // B*B; pitch (floats) of the fp32 partial sums
  int total;
};

constexpr int MTILES = 2;
constexpr int MT = MTILES * 16; // rows per group

__host__ __device__ inline Plan make_plan(int r, int H, int B) {
  Plan p;
  p.CS = r / CL;
  p.HS = H / CL;
  p.nt1 = p.CS / 8;
  // K splits: fill the warps, keep every split a whole number of 16-wide k-steps
  p.ks1 = std::min(NW / p.nt1, r / 16);
  p.mix_rows = B * B;
  p.pp = r + 4;
  const int mparts = (p.mix_rows + 255) / 256, mbox = std::min(p.mix_rows, 256);
  int o = 0;
  // TMA / swizzled regions 1024-byte aligned, the rest 16-byte aligned
  auto take = [&](int bytes, int align) {
    o = (o + align - 1) / align * align;
    const int at = o;
    o += bytes;
    return at;
  };
  p.wlat = take(p.CS * r * 2, 1024);
  p.wg = take(p.HS * r * 2, 1024);
  p.wu = take(p.HS * r * 2, 1024);
  p.wdk = take(r * p.HS * 2, 1024);          // w_down[:, own units]: r rows x HS
  p.mix = take(mparts * mbox * p.CS * 2, 1024);
  p.ep = take(std::max(MT * r * 2, MT * p.pp * 4), 1024);   // embeddings, later partials
  p.uhi = take(MT * r * 2, 1024);
  p.ulo = take(MT * r * 2, 1024);
  p.ahi = take(MT * p.HS * 2, 1024);
  p.alo = take(MT * p.HS * 2, 1024);
  p.xh = take(MT * p.CS * 4, 16);
  p.part = take(p.ks1 * MT * (p.CS + 1) * 4, 16);
  p.us = take(MT * (p.CS + 1) * 4, 16);
  p.prev = take(MT * 8, 16);
  p.bar = take(16, 16);
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

// acc[i] += A[16i.., k0:k1] . B[n0..n0+8, k0:k1]^T for every m-tile i (A: MT rows, B: RB
// rows, both swizzled).  One B fragment per k-step feeds MTILES independent MMAs.
template <int MTILES>
__device__ __forceinline__ void warp_gemm(float (&acc)[MTILES][4], uint32_t A, uint32_t Bm, int RB,
                                          int n0, int k0, int k1) {
  constexpr int MT = MTILES * 16;
  const int lane = threadIdx.x % 32;
  const int ar = lane % 16, ak = (lane / 16) * 8;
  const int br = n0 + (lane % 8), bk = ((lane / 8) % 2) * 8;
  for (int k = k0; k < k1; k += 16) {
    uint32_t b[2];
    ldm_x2(b, Bm + swz(br, k + bk, RB));
#pragma unroll
    for (int i = 0; i < MTILES; ++i) {
      uint32_t a[4];
      ldm_x4(a, A + swz(i * 16 + ar, k + ak, MT));
      mma16816(acc[i], a, b);
    }
  }
}

// Same for two B operands (gate and up) sharing every A fragment.
template <int MTILES>
__device__ __forceinline__ void warp_gemm_pair(float (&acc0)[MTILES][4], float (&acc1)[MTILES][4],
                                               uint32_t A, uint32_t B0, uint32_t B1, int RB,
                                               int n0, int K) {
  constexpr int MT = MTILES * 16;
  const int lane = threadIdx.x % 32;
  const int ar = lane % 16, ak = (lane / 16) * 8;
  const int br = n0 + (lane % 8), bk = ((lane / 8) % 2) * 8;
  for (int k = 0; k < K; k += 16) {
    uint32_t b0[2], b1[2];
    const int bo = swz(br, k + bk, RB);
    ldm_x2(b0, B0 + bo);
    ldm_x2(b1, B1 + bo);
#pragma unroll
    for (int i = 0; i < MTILES; ++i) {
      uint32_t a[4];
      ldm_x4(a, A + swz(i * 16 + ar, k + ak, MT));
      mma16816(acc0[i], a, b0);
      mma16816(acc1[i], a, b1);
    }
  }
}

// Copy the columns [p*W, (p+1)*W) of two swizzled MT-row matrices from every other CTA p
// of the cluster into this CTA's copies (same offsets everywhere); loads issued first.
template <int PER>
__device__ __forceinline__ void gather_peers2(cg::cluster_group& cluster, uint8_t* b0, uint8_t* b1,
                                              int W, int q) {
  const int chunks = W / 8;                       // 16-byte chunks per row and peer
  const int per_buf = (CL - 1) * MT * chunks;
  const int total = 2 * per_buf;
  for (int i0 = threadIdx.x; i0 < total; i0 += PER * THREADS) {
    uint4 v[PER];
    int off[PER];
    uint8_t* dst[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = i0 + u * THREADS;
      off[u] = -1;
      if (i < total) {
        const int which = i / per_buf, j = i % per_buf;
        const int pp = j / (MT * chunks), rem = j % (MT * chunks);
        const int p = pp + (pp >= q);
        const int m = rem / chunks, cc = rem % chunks;
        off[u] = swz(m, p * W + cc * 8, MT);
        dst[u] = which ? b1 : b0;
        v[u] = *reinterpret_cast<const uint4*>(cluster.map_shared_rank(dst[u], p) + off[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < PER; ++u)
      if (off[u] >= 0) *reinterpret_cast<uint4*>(dst[u] + off[u]) = v[u];
  }
}

__device__ __forceinline__ void split_store(uint8_t* hi, uint8_t* lo, int off, float v) {
  const bf16 h = __float2bfloat16_rn(v);
  *reinterpret_cast<bf16*>(hi + off) = h;
  *reinterpret_cast<bf16*>(lo + off) = __float2bfloat16_rn(v - __bfloat162float(h));
}

struct Maps {
  CUtensorMap wlat, wg, wu, wdk, mix;
};

__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS, 1) latent_mma_kernel(
    const __grid_constant__ Maps maps, const int64_t* __restrict__ blk,
    const int64_t* __restrict__ am1, const float* __restrict__ xh, const bf16* __restrict__ w1,
    bf16* __restrict__ lat, int N, int B, int r, int H, int V, uint32_t* err) {
  constexpr int MAXU = (MT * 32 + THREADS - 1) / THREADS;   // outputs per thread, CS <= 32
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (ptx::smem_u32(sm_raw) & 1023u)) & 1023u);
  cg::cluster_group cluster = cg::this_cluster();
  const int q = (int)cluster.block_rank();
  const int cid = blockIdx.x / CL, nclusters = gridDim.x / CL;
  const Plan P = make_plan(r, H, B);
  const int CS = P.CS, HS = P.HS;
  const uint32_t s0 = ptx::smem_u32(sm);
  const uint32_t aWl = s0 + P.wlat, aWg = s0 + P.wg, aWu = s0 + P.wu, aWdk = s0 + P.wdk;
  const uint32_t aE = s0 + P.ep, aUhi = s0 + P.uhi, aUlo = s0 + P.ulo;
  const uint32_t aAhi = s0 + P.ahi, aAlo = s0 + P.alo;
  const bf16* sMix = (const bf16*)(sm + P.mix);
  const float* sXh = (const float*)(sm + P.xh);
  float* sP = (float*)(sm + P.ep);          // partial sums of the down projection [MT][pp]
  float* sPart = (float*)(sm + P.part);
  float* sUs = (float*)(sm + P.us);
  int64_t* sPrev = (int64_t*)(sm + P.prev);
  const uint32_t bar = s0 + P.bar;
  int& s_abort = *reinterpret_cast<int*>(sm + P.bar + 8);   // beside the mbarrier
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g8 = lane / 4, t4 = lane % 4;
  const int nb = MT / B;                   // blocks per group
  const int groups = (N + nb - 1) / nb;
  const int ldp = CS + 1;

  // ---- weight and mixer slices by TMA, once: nothing here depends on the previous pass ----
  if (tid == 0) {
    s_abort = 0;
    ptx::mbar_init(bar, 1);
    ptx::fence_barrier_init();
    const int wbytes = (CS * r + 2 * HS * r + r * HS) * 2;
    const int mparts = (P.mix_rows + 255) / 256, mbox = std::min(P.mix_rows, 256);
    const int rparts = (r + 255) / 256, rbox = std::min(r, 256);
    ptx::mbar_arrive_expect_tx(bar, wbytes + mparts * mbox * CS * 2);
    const uint64_t pol = ptx::policy_evict_last();
    for (int kc = 0; kc < r / 64; ++kc) {
      ptx::tma_load_2d(aWl + kc * CS * 128, &maps.wlat, bar, kc * 64, q * CS, pol);
      ptx::tma_load_2d(aWg + kc * HS * 128, &maps.wg, bar, kc * 64, q * HS, pol);
      ptx::tma_load_2d(aWu + kc * HS * 128, &maps.wu, bar, kc * 64, q * HS, pol);
    }
    for (int kc = 0; kc < HS / 64; ++kc)
      for (int rp = 0; rp < rparts; ++rp)
        ptx::tma_load_2d(aWdk + (kc * r + rp * rbox) * 128, &maps.wdk, bar, q * HS + kc * 64,
                         rp * rbox, pol);
    for (int pt = 0; pt < mparts; ++pt)
      ptx::tma_load_2d(s0 + P.mix + pt * mbox * CS * 2, &maps.mix, bar, q * CS, pt * mbox, pol);
  }
  ptx::pdl_wait();                         // blk (and xh) come from earlier kernels
  ptx::pdl_trigger();
  __syncthreads();
  if (tid == 0 && !ptx::mbar_wait(bar, 0, &s_abort, err)) s_abort = 1;
  __syncthreads();

  for (int grp = cid; grp < groups; grp += nclusters) {
    const int n0 = grp * nb;
    const int rows = std::min(nb, N - n0) * B;   // valid rows of this group

    // ---- token ids, then embeddings and the xh slice by cp.async ----
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
      const int ec = r / 8, xc = CS / 4;
      for (int i = tid; i < MT * (ec + xc); i += THREADS) {
        const int m = i / (ec + xc), c = i % (ec + xc);
        if (c < ec) {
          const uint32_t dst = aE + swz(m, c * 8, MT);
          if (m < rows)
            cp_async16(dst, w1 + sPrev[m] * r + c * 8);
          else
            *reinterpret_cast<uint4*>(sm + (dst - s0)) = make_uint4(0, 0, 0, 0);
        } else {
          const int cc = c - ec;
          const uint32_t dst = s0 + P.xh + (m * CS + cc * 4) * 4;
          if (m < rows)
            cp_async16(dst, xh + ((int64_t)(n0 * B + m)) * r + q * CS + cc * 4);
          else
            *reinterpret_cast<uint4*>(sm + (dst - s0)) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- x (own channels) = xh + emb . w_lat^T, K split over warp groups ----
    if (warp < P.nt1 * P.ks1) {
      const int nt = warp % P.nt1, ks = warp / P.nt1;
      const int kl = r / P.ks1;
      float acc[MTILES][4] = {};
      warp_gemm<MTILES>(acc, aE, aWl, CS, nt * 8, ks * kl, (ks + 1) * kl);
      float* dst = sPart + ks * MT * ldp;
#pragma unroll
      for (int i = 0; i < MTILES; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dst[(i * 16 + g8 + (e >= 2 ? 8 : 0)) * ldp + nt * 8 + 2 * t4 + (e & 1)] = acc[i][e];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < MAXU; ++k) {
      const int i = tid + k * THREADS;
      if (i < MT * CS) {
        const int m = i / CS, c = i % CS;
        float x = sXh[m * CS + c];
        for (int ks = 0; ks < P.ks1; ++ks) x += sPart[ks * MT * ldp + m * ldp + c];
        sUs[m * ldp + c] = x;
      }
    }
    __syncthreads();

    // ---- causal per-channel mixer (fp32): u[b, c] = sum_j mix[c, b, j] x[j, c] ----
    float uval[MAXU];
#pragma unroll
    for (int k = 0; k < MAXU; ++k) {
      const int i = tid + k * THREADS;
      const int m = i / CS, c = i % CS;
      float u = 0.f;
      if (i < MT * CS && m < rows) {
        const int bl = m / B, b = m % B;
        const bf16* mc = sMix + (b * B) * CS + c;      // rows (b, j), columns = channels
        for (int j = 0; j < B; ++j)
          u = fmaf(__bfloat162float(mc[j * CS]), sUs[(bl * B + j) * ldp + c], u);
      }
      uval[k] = u;
    }
    __syncthreads();                       // every x read before u overwrites it
#pragma unroll
    for (int k = 0; k < MAXU; ++k) {
      const int i = tid + k * THREADS;
      if (i < MT * CS) {
        const int m = i / CS, c = i % CS;
        sUs[m * ldp + c] = uval[k];
        split_store(sm + P.uhi, sm + P.ulo, swz(m, q * CS + c, MT), uval[k]);
      }
    }
    cluster.sync();
    gather_peers2<7>(cluster, sm + P.uhi, sm + P.ulo, CS, q);
    __syncthreads();

    // ---- SwiGLU on own hidden units, from u = hi + lo: a = silu(u w_g^T) * (u w_u^T) ----
    for (int nt = warp; nt < HS / 8; nt += NW) {
      float ag[MTILES][4] = {}, au[MTILES][4] = {};
      warp_gemm_pair<MTILES>(ag, au, aUhi, aWg, aWu, HS, nt * 8, r);
      warp_gemm_pair<MTILES>(ag, au, aUlo, aWg, aWu, HS, nt * 8, r);
#pragma unroll
      for (int i = 0; i < MTILES; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = i * 16 + g8 + (e >= 2 ? 8 : 0);
          const int hh = nt * 8 + 2 * t4 + (e & 1);
          split_store(sm + P.ahi, sm + P.alo, swz(m, hh, MT), silu(ag[i][e]) * au[i][e]);
        }
    }
    __syncthreads();

    // ---- partial down projection over own units, every channel: P = a . w_down[:, own]^T ----
    for (int nt = warp; nt < r / 8; nt += NW) {
      float acc[MTILES][4] = {};
      warp_gemm<MTILES>(acc, aAhi, aWdk, r, nt * 8, 0, HS);
      warp_gemm<MTILES>(acc, aAlo, aWdk, r, nt * 8, 0, HS);
#pragma unroll
      for (int i = 0; i < MTILES; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sP[(i * 16 + g8 + (e >= 2 ? 8 : 0)) * P.pp + nt * 8 + 2 * t4 + (e & 1)] = acc[i][e];
    }
    cluster.sync();

    // ---- lat (own channels) = u + sum_p P_p, p = 0..7 in order, over DSMEM ----
#pragma unroll
    for (int k = 0; k < MAXU; ++k) {
      const int i = tid + k * THREADS;
      if (i < MT * CS) {
        const int m = i / CS, c = i % CS;
        const int off = m * P.pp + q * CS + c;
        float pv[CL];
#pragma unroll
        for (int p = 0; p < CL; ++p) pv[p] = *(cluster.map_shared_rank(sP, p) + off);
        if (m < rows && (m % B) != 0) {
          float v = sUs[m * ldp + c];
#pragma unroll
          for (int p = 0; p < CL; ++p) v += pv[p];
          const int n = n0 + m / B, b = m % B;
          lat[((int64_t)n * (B - 1) + b - 1) * r + q * CS + c] = __float2bfloat16_rn(v);
        }
      }
    }
    cluster.sync();   // peers may still read this CTA's u halves and partial sums
  }
  // nothing may land in shared memory after the CTA exits
  if (tid == 0 && s_abort) {
    volatile int no_abort = 0;
    ptx::mbar_wait(bar, 0, &no_abort, err);
  }
}

int g_max_clusters = 0;   // co-resident clusters (queried once)

size_t smem_bytes(int r, int H, int B) { return (size_t)make_plan(r, H, B).total + 1024; }

int max_clusters(int smem) {
  if (g_max_clusters > 0) return g_max_clusters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaFuncSetAttribute(latent_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, latent_mma_kernel, &cfg) != cudaSuccess || n <= 0)
    n = 1;
  g_max_clusters = n;
  return n;
}

}  // namespace

bool xp_latent_mma_ok(int r, int H, int B, xp_dtype dt) {
  if (dt != XP_BF16 || B < 2 || B > MT) return false;
  if (r != 64 && r != 128 && r != 256) return false;      // r/8 channels = 1, 2 or 4 n-tiles
  if (H % (8 * 64) != 0 || H > 1024) return false;        // own units in 64-wide chunks
  return smem_bytes(r, H, B) <= 227 * 1024;
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
  return enc(&h->tm_wlat, h->w_lat, r, r, 64, CS, true) &&
         enc(&h->tm_wg, h->w_gate, H, r, 64, HS, true) &&
         enc(&h->tm_wu, h->w_up, H, r, 64, HS, true) &&
         enc(&h->tm_wd, h->w_down, r, H, 64, std::min(r, 256), true) &&
         enc(&h->tm_mixT, h->mixT, B * B, r, CS, std::min(B * B, 256), false);
}

cudaError_t xp_launch_latent_mma(const xp_head* h, const int64_t* blk, const int64_t* am1,
                                 const float* xh, int N, void* lat, cudaStream_t s) {
  const int smem = (int)smem_bytes(h->r, h->H, h->B);
  cudaError_t e =
      cudaFuncSetAttribute(latent_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nb = MT / h->B;
  const int groups = (N + nb - 1) / nb;
  const int clusters = std::min(groups, max_clusters(smem));
  const Maps maps = {h->tm_wlat, h->tm_wg, h->tm_wu, h->tm_wd, h->tm_mixT};
  e = xp_launch_pdl(latent_mma_kernel, dim3(clusters * CL), dim3(THREADS), (size_t)smem, s, maps,
                    blk, am1, xh, (const bf16*)h->w1, (bf16*)lat, N, h->B, h->r, h->H, h->V,
                    h->err);
  return e != cudaSuccess ? e : cudaGetLastError();
}
