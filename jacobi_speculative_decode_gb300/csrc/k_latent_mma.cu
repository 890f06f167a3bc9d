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
// weight slices are copied into shared memory once, before the kernel waits
// on the previous pass, and stay there while the cluster walks over groups of
// MT rows (whole blocks).  The full u and SwiGLU activations of a group are
// exchanged through distributed shared memory.  Products use mma.sync
// m16n8k16 (bf16 in, fp32 accumulate); the mixer, the K-split partial sums
// (added in a fixed order) and the residual stay in fp32.
#include <cooperative_groups.h>

#include <algorithm>

#include "xp_device.cuh"

namespace cg = cooperative_groups;
using namespace xpd;
typedef __nv_bfloat16 bf16;

namespace {

constexpr int CL = 8;          // CTAs per cluster
constexpr int THREADS = 256;   // 8 warps
constexpr int NW = THREADS / 32;

struct Plan {                  // shapes and byte offsets into dynamic shared memory
  int MT, CS, HS, pk_r, pk_h;
  int nt1, ks1;                // in_proj / w_down: n-tiles of the CTA's channels, K splits
  int wlat, wg, wu, wd, ufull, afull, part, us, prev;
  int total;
};

__host__ __device__ inline Plan make_plan(int MT, int r, int H) {
  Plan p;
  p.MT = MT;
  p.CS = r / CL;
  p.HS = H / CL;
  p.pk_r = r + 8;              // padded pitches keep ldmatrix rows on distinct banks
  p.pk_h = H + 8;
  p.nt1 = p.CS / 8;
  // K splits: fill the warps, but keep every split a whole number of 16-wide k-steps
  p.ks1 = std::min(NW / p.nt1, std::min(r, H) / 16);
  int o = 0;
  auto take = [&](int bytes) { int at = o; o += (bytes + 127) / 128 * 128; return at; };
  p.wlat = take(p.CS * p.pk_r * 2);
  p.wg = take(p.HS * p.pk_r * 2);
  p.wu = take(p.HS * p.pk_r * 2);
  p.wd = take(p.CS * p.pk_h * 2);
  p.ufull = take(MT * p.pk_r * 2);
  // embeddings (phase 1) and gathered activations (phase 3) share one region
  p.afull = take(std::max(MT * p.pk_h * 2, MT * p.pk_r * 2));
  p.part = take(p.ks1 * MT * (p.CS + 1) * 4);   // K-split partial sums
  p.us = take(MT * (p.CS + 1) * 4);             // x, then u (fp32)
  p.prev = take(MT * 8);
  p.total = o;
  return p;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void ldm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__device__ __forceinline__ void ldm_x2(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc[i] (16x8, rows 16i..) += A[rows, k0:k1] . Bt[n0:n0+8, k0:k1]^T for every m-tile i:
// one B fragment per k-step feeds MTILES independent MMAs.
template <int MTILES>
__device__ __forceinline__ void warp_gemm(float (&acc)[MTILES][4], const bf16* A, int lda,
                                          const bf16* Bt, int ldb, int n0, int k0, int k1) {
  const int lane = threadIdx.x % 32;
  const bf16* ap = A + (lane % 16) * lda + (lane / 16) * 8;
  const bf16* bp = Bt + (n0 + (lane % 8)) * ldb + ((lane / 8) % 2) * 8;
  for (int k = k0; k < k1; k += 16) {
    uint32_t b[2];
    ldm_x2(b, bp + k);
#pragma unroll
    for (int i = 0; i < MTILES; ++i) {
      uint32_t a[4];
      ldm_x4(a, ap + i * 16 * lda + k);
      mma16816(acc[i], a, b);
    }
  }
}

// Same for two B operands (gate and up) sharing every A fragment.
template <int MTILES>
__device__ __forceinline__ void warp_gemm_pair(float (&acc0)[MTILES][4], float (&acc1)[MTILES][4],
                                               const bf16* A, int lda, const bf16* B0,
                                               const bf16* B1, int ldb, int n0, int K) {
  const int lane = threadIdx.x % 32;
  const bf16* ap = A + (lane % 16) * lda + (lane / 16) * 8;
  const int boff = (n0 + (lane % 8)) * ldb + ((lane / 8) % 2) * 8;
  for (int k = 0; k < K; k += 16) {
    uint32_t b0[2], b1[2];
    ldm_x2(b0, B0 + boff + k);
    ldm_x2(b1, B1 + boff + k);
#pragma unroll
    for (int i = 0; i < MTILES; ++i) {
      uint32_t a[4];
      ldm_x4(a, ap + i * 16 * lda + k);
      mma16816(acc0[i], a, b0);
      mma16816(acc1[i], a, b1);
    }
  }
}

// Copy columns [p*W, (p+1)*W) of buf (MT rows x pitch) from every other CTA p of the
// cluster into this CTA's buf; four 16-byte loads in flight per thread.
__device__ __forceinline__ void gather_peers(cg::cluster_group& cluster, bf16* buf, int MT,
                                             int pitch, int W, int q) {
  const int chunks = W / 8;
  const int total = (CL - 1) * MT * chunks;
  for (int i0 = threadIdx.x; i0 < total; i0 += 4 * THREADS) {
    uint4 v[4];
    int off[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * THREADS;
      off[u] = -1;
      if (i < total) {
        const int pp = i / (MT * chunks), rem = i % (MT * chunks);
        const int p = pp + (pp >= q);
        const int m = rem / chunks, cc = rem % chunks;
        off[u] = m * pitch + p * W + cc * 8;
        v[u] = *reinterpret_cast<const uint4*>(cluster.map_shared_rank(buf, p) + off[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (off[u] >= 0) *reinterpret_cast<uint4*>(buf + off[u]) = v[u];
  }
}

template <int MTILES>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS, 1) latent_mma_kernel(
    const int64_t* __restrict__ blk, const int64_t* __restrict__ am1, const float* __restrict__ xh,
    const bf16* __restrict__ w1, const bf16* __restrict__ wlat, const float* __restrict__ mixT,
    const bf16* __restrict__ wg, const bf16* __restrict__ wu, const bf16* __restrict__ wd,
    bf16* __restrict__ lat, int N, int B, int r, int H, int V, uint32_t* err) {
  constexpr int MT = MTILES * 16;
  constexpr int MAXU = (MT * 32 + THREADS - 1) / THREADS;   // outputs per thread, CS <= 32
  extern __shared__ __align__(128) uint8_t sm[];
  cg::cluster_group cluster = cg::this_cluster();
  const int q = (int)cluster.block_rank();
  const int cid = blockIdx.x / CL, nclusters = gridDim.x / CL;
  const Plan P = make_plan(MT, r, H);
  const int CS = P.CS, HS = P.HS;
  bf16* sWl = (bf16*)(sm + P.wlat);
  bf16* sWg = (bf16*)(sm + P.wg);
  bf16* sWu = (bf16*)(sm + P.wu);
  bf16* sWd = (bf16*)(sm + P.wd);
  bf16* sU = (bf16*)(sm + P.ufull);
  bf16* sA = (bf16*)(sm + P.afull);        // embeddings first, activations later
  float* sPart = (float*)(sm + P.part);
  float* sUs = (float*)(sm + P.us);
  int64_t* sPrev = (int64_t*)(sm + P.prev);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g8 = lane / 4, t4 = lane % 4;
  const int nb = MT / B;                   // blocks per group
  const int groups = (N + nb - 1) / nb;
  const int ldp = CS + 1;

  // ---- weight slices -> smem, once (nothing here depends on the previous pass) ----
  {
    auto stage = [&](bf16* dst, int pitch, const bf16* src, int nrows, int ncols) {
      const int chunks = ncols / 8;
      for (int i = tid; i < nrows * chunks; i += THREADS) {
        const int rr = i / chunks, cc = i % chunks;
        cp_async16(dst + rr * pitch + cc * 8, src + (int64_t)rr * ncols + cc * 8);
      }
    };
    stage(sWl, P.pk_r, wlat + (int64_t)q * CS * r, CS, r);
    stage(sWg, P.pk_r, wg + (int64_t)q * HS * r, HS, r);
    stage(sWu, P.pk_r, wu + (int64_t)q * HS * r, HS, r);
    stage(sWd, P.pk_h, wd + (int64_t)q * CS * H, CS, H);
  }
  pdl_wait();                              // blk (and xh) come from earlier kernels
  pdl_trigger();

  for (int grp = cid; grp < groups; grp += nclusters) {
    const int n0 = grp * nb;
    const int rows = std::min(nb, N - n0) * B;   // valid rows of this group

    // ---- token ids and embeddings ----
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
      const int chunks = r / 8;
      for (int i = tid; i < MT * chunks; i += THREADS) {
        const int m = i / chunks, cc = i % chunks;
        if (m < rows)
          cp_async16(sA + m * P.pk_r + cc * 8, w1 + sPrev[m] * r + cc * 8);
        else
          *reinterpret_cast<uint4*>(sA + m * P.pk_r + cc * 8) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- phase 1: x (own channels) = xh + emb . w_lat^T, K split over warp groups ----
    if (warp < P.nt1 * P.ks1) {
      const int nt = warp % P.nt1, ks = warp / P.nt1;
      const int kl = r / P.ks1;
      float acc[MTILES][4] = {};
      warp_gemm<MTILES>(acc, sA, P.pk_r, sWl, P.pk_r, nt * 8, ks * kl, (ks + 1) * kl);
      float* dst = sPart + ks * MT * ldp;
#pragma unroll
      for (int i = 0; i < MTILES; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dst[(i * 16 + g8 + (e >= 2 ? 8 : 0)) * ldp + nt * 8 + 2 * t4 + (e & 1)] = acc[i][e];
    }
    __syncthreads();
    for (int i = tid; i < MT * CS; i += THREADS) {
      const int m = i / CS, c = i % CS;
      float x = 0.f;
      if (m < rows) {
        x = xh[((int64_t)(n0 * B + m)) * r + q * CS + c];
        for (int ks = 0; ks < P.ks1; ++ks) x += sPart[ks * MT * ldp + m * ldp + c];
      }
      sUs[m * ldp + c] = x;
    }
    __syncthreads();

    // ---- causal per-channel mixer (fp32): u[b, c] = sum_j mix[c, b, j] x[j, c] ----
    // mixT is the folded mixer laid out [b][j][channel] (fp32): coalesced reads.
    float uval[MAXU];
#pragma unroll
    for (int k = 0; k < MAXU; ++k) {
      const int i = tid + k * THREADS;
      const int m = i / CS, c = i % CS;
      float u = 0.f;
      if (i < MT * CS && m < rows) {
        const int bl = m / B, b = m % B;
        const float* mc = mixT + (int64_t)b * B * r + q * CS + c;
        for (int j = 0; j < B; ++j)
          u = fmaf(__ldg(mc + (int64_t)j * r), sUs[(bl * B + j) * ldp + c], u);
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
        sU[m * P.pk_r + q * CS + c] = __float2bfloat16_rn(uval[k]);
      }
    }
    cluster.sync();
    gather_peers(cluster, sU, MT, P.pk_r, CS, q);
    __syncthreads();

    // ---- phase 2: SwiGLU on own hidden units: a = silu(u w_gate^T) * (u w_up^T) ----
    for (int nt = warp; nt < HS / 8; nt += NW) {
      float ag[MTILES][4] = {}, au[MTILES][4] = {};
      warp_gemm_pair<MTILES>(ag, au, sU, P.pk_r, sWg, sWu, P.pk_r, nt * 8, r);
#pragma unroll
      for (int i = 0; i < MTILES; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = i * 16 + g8 + (e >= 2 ? 8 : 0);
          const int hh = nt * 8 + 2 * t4 + (e & 1);
          sA[m * P.pk_h + q * HS + hh] = __float2bfloat16_rn(silu(ag[i][e]) * au[i][e]);
        }
    }
    cluster.sync();
    gather_peers(cluster, sA, MT, P.pk_h, HS, q);
    __syncthreads();

    // ---- phase 3: lat (own channels) = u + a . w_down^T, K split over warp groups ----
    if (warp < P.nt1 * P.ks1) {
      const int nt = warp % P.nt1, ks = warp / P.nt1;
      const int kl = H / P.ks1;
      float acc[MTILES][4] = {};
      warp_gemm<MTILES>(acc, sA, P.pk_h, sWd, P.pk_h, nt * 8, ks * kl, (ks + 1) * kl);
      float* dst = sPart + ks * MT * ldp;
#pragma unroll
      for (int i = 0; i < MTILES; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dst[(i * 16 + g8 + (e >= 2 ? 8 : 0)) * ldp + nt * 8 + 2 * t4 + (e & 1)] = acc[i][e];
    }
    __syncthreads();
    for (int i = tid; i < MT * CS; i += THREADS) {
      const int m = i / CS, c = i % CS;
      if (m < rows && (m % B) != 0) {
        float v = sUs[m * ldp + c];
        for (int ks = 0; ks < P.ks1; ++ks) v += sPart[ks * MT * ldp + m * ldp + c];
        const int n = n0 + m / B, b = m % B;
        lat[((int64_t)n * (B - 1) + b - 1) * r + q * CS + c] = __float2bfloat16_rn(v);
      }
    }
    cluster.sync();   // peers may still read this CTA's u / activation slices
  }
}

int g_max_clusters[2] = {0, 0};   // co-resident clusters per variant (queried once)

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
  const Plan P = make_plan(MTILES * 16, h->r, h->H);
  cudaError_t e = cudaFuncSetAttribute(latent_mma_kernel<MTILES>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, P.total);
  if (e != cudaSuccess) return e;
  const int nb = P.MT / h->B;
  const int groups = (N + nb - 1) / nb;
  const int clusters = std::min(groups, max_clusters<MTILES>(P.total));
  e = xp_launch_pdl(latent_mma_kernel<MTILES>, dim3(clusters * CL), dim3(THREADS),
                    (size_t)P.total, s, blk, am1, xh, (const bf16*)h->w1, (const bf16*)h->w_lat,
                    (const float*)h->mixT, (const bf16*)h->w_gate, (const bf16*)h->w_up,
                    (const bf16*)h->w_down, (bf16*)lat, N, h->B, h->r, h->H, h->V, h->err);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool xp_latent_mma_ok(int r, int H, int B, xp_dtype dt) {
  if (dt != XP_BF16 || B < 2 || B > 32) return false;
  if (r != 64 && r != 128 && r != 256) return false;      // r/8 channels = 1, 2 or 4 n-tiles
  if (H % (8 * CL) != 0 || H > 1024) return false;
  return make_plan(48, r, H).total <= 227 * 1024;
}

cudaError_t xp_launch_latent_mma(const xp_head* h, const int64_t* blk, const int64_t* am1,
                                 const float* xh, int N, void* lat, cudaStream_t s) {
  // 32-row groups while they fit in one wave of co-resident clusters, else 48-row groups
  const Plan p32 = make_plan(32, h->r, h->H);
  const int groups32 = (N + 32 / h->B - 1) / (32 / h->B);
  if (groups32 <= max_clusters<2>(p32.total)) return launch<2>(h, blk, am1, xh, N, lat, s);
  return launch<3>(h, blk, am1, xh, N, lat, s);
}
