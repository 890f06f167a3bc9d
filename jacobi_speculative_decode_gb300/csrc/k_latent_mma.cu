// Latent stage of one pass on tensor cores, one 8-CTA cluster per group of blocks
// (xpress kernels page, _xpress_latent_kernel; qwen3_xpress page, _refine_latent):
//   prev[0] = am1[n], prev[b] = blk[n, b-1]
//   x[b]    = xh[n, b] + w_lat w1[prev[b]]
//   u[b, c] = sum_j mix[c, b, j] x[j, c]            (stored mixer is lower-triangular)
//   lat[b]  = u[b] + w_down (silu(w_gate u[b]) * (w_up u[b]))      for b = 1..B-1
//
// The cluster splits the work by output features so each CTA streams only 1/8
// of the weights: CTA q owns channels [q*r/8, (q+1)*r/8) for the in_proj and
// w_down products and hidden units [q*H/8, (q+1)*H/8) for the SwiGLU.  The
// full u and SwiGLU activations are exchanged through distributed shared
// memory.  Products use mma.sync m16n8k16 (bf16 in, fp32 accumulate); the
// mixer and the residual stay in fp32.  Each cluster covers 32 rows (whole
// blocks).
#include <cooperative_groups.h>

#include <algorithm>

#include "xp_device.cuh"

namespace cg = cooperative_groups;
using namespace xpd;
typedef __nv_bfloat16 bf16;

namespace {

constexpr int CL = 8;          // CTAs per cluster
constexpr int MT = 32;         // rows per cluster (2 m16 tiles)
constexpr int THREADS = 256;

struct Smem {                  // byte offsets into dynamic shared memory
  int wlat, wg, wu, wd, mix, ufull, afull, xs, us, prev;
  int pk_r, pk_h;              // padded pitches (elements) of r- and H-wide bf16 rows
  int total;
};

__host__ __device__ inline Smem smem_plan(int r, int H, int B) {
  Smem s;
  const int CS = r / CL, HS = H / CL;
  s.pk_r = r + 8;
  s.pk_h = H + 8;
  int o = 0;
  auto take = [&](int bytes) { int at = o; o += (bytes + 127) / 128 * 128; return at; };
  s.wlat = take(CS * s.pk_r * 2);
  s.wg = take(HS * s.pk_r * 2);
  s.wu = take(HS * s.pk_r * 2);
  s.wd = take(CS * s.pk_h * 2);
  s.mix = take(B * B * (CS + 1) * 4);     // fp32, [out slot][in slot][channel]
  s.ufull = take(MT * s.pk_r * 2);
  // the embeddings (phase 1) and the gathered activations (phase 3) share one region
  s.afull = take(std::max(MT * s.pk_h * 2, MT * s.pk_r * 2));
  s.xs = take(MT * (CS + 1) * 4);
  s.us = take(MT * (CS + 1) * 4);
  s.prev = take(MT * 8);
  s.total = o;
  return s;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void pdl_wait_all() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
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
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc(16x8 tile at A rows m0.., B rows n0..) = sum_k A[m][k] * Bt[n][k]; A, Bt bf16 row-major
// with pitches lda / ldb (elements).
__device__ __forceinline__ void tile_mma(float (&acc)[4], const bf16* A, int lda, int m0,
                                         const bf16* Bt, int ldb, int n0, int K) {
  const int lane = threadIdx.x % 32;
  const bf16* ap = A + (m0 + (lane % 16)) * lda + (lane / 16) * 8;
  const bf16* bp = Bt + (n0 + (lane % 8)) * ldb + ((lane / 8) % 2) * 8;
  for (int k = 0; k < K; k += 16) {
    uint32_t a[4], b[2];
    ldm_x4(a, ap + k);
    ldm_x2(b, bp + k);
    mma16816(acc, a, b);
  }
}

// Copy the column slices [p*W, (p+1)*W) of buf (MT rows, pitch elements) from every
// other CTA p of the cluster into this CTA's buf; four 16-byte loads in flight per thread.
__device__ __forceinline__ void gather_peers(cg::cluster_group& cluster, bf16* buf, int pitch,
                                             int W, int q, int tid) {
  const int chunks = W / 8;
  const int total = (CL - 1) * MT * chunks;
  for (int i0 = tid; i0 < total; i0 += 4 * THREADS) {
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

__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS, 1) latent_mma_kernel(
    const int64_t* __restrict__ blk, const int64_t* __restrict__ am1, const float* __restrict__ xh,
    const bf16* __restrict__ w1, const bf16* __restrict__ wlat, const bf16* __restrict__ mix,
    const bf16* __restrict__ wg, const bf16* __restrict__ wu, const bf16* __restrict__ wd,
    bf16* __restrict__ lat, int N, int B, int r, int H, int V, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t sm[];
  cg::cluster_group cluster = cg::this_cluster();
  const int q = (int)cluster.block_rank();
  const int cid = blockIdx.x / CL;
  const int CS = r / CL, HS = H / CL;
  const Smem P = smem_plan(r, H, B);
  bf16* sWl = (bf16*)(sm + P.wlat);
  bf16* sWg = (bf16*)(sm + P.wg);
  bf16* sWu = (bf16*)(sm + P.wu);
  bf16* sWd = (bf16*)(sm + P.wd);
  float* sMix = (float*)(sm + P.mix);
  bf16* sU = (bf16*)(sm + P.ufull);
  bf16* sA = (bf16*)(sm + P.afull);        // embeddings first, activations later
  float* sX = (float*)(sm + P.xs);
  float* sUs = (float*)(sm + P.us);
  int64_t* sPrev = (int64_t*)(sm + P.prev);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int nb = MT / B;                   // blocks per cluster
  const int n0 = cid * nb;
  const int rows = std::min(nb, N - n0) * B;   // valid rows of this cluster

  // ---- weight slices -> smem (independent of the previous pass) ----
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
  // mixer slice, transposed to [b][j][c] so that neighbouring channels hit neighbouring banks
  for (int i = tid; i < CS * B * B; i += THREADS) {
    const int c = i / (B * B), bj = i % (B * B);
    sMix[bj * (CS + 1) + c] = __bfloat162float(mix[(int64_t)q * CS * B * B + i]);
  }

  // ---- token ids and embeddings (written by the previous kernel) ----
  pdl_wait_all();
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

  pdl_trigger();

  // ---- phase 1: x (own channels) = xh + emb . w_lat^T ----
  for (int it = warp; it < (MT / 16) * (CS / 8); it += THREADS / 32) {
    const int mt = it / (CS / 8), nt = it % (CS / 8);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mma(acc, sA, P.pk_r, mt * 16, sWl, P.pk_r, nt * 8, r);
    const int g = lane / 4, t = lane % 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = mt * 16 + g + (e >= 2 ? 8 : 0);
      const int c = nt * 8 + 2 * t + (e & 1);
      float v = acc[e];
      if (m < rows) v += xh[((int64_t)(n0 * B + m)) * r + q * CS + c];
      sX[m * (CS + 1) + c] = v;
    }
  }
  __syncthreads();

  // ---- causal per-channel mixer (fp32): u[b, c] = sum_j mix[c, b, j] x[j, c] ----
  for (int i = tid; i < MT * CS; i += THREADS) {
    const int m = i / CS, c = i % CS;
    float u = 0.f;
    if (m < rows) {
      const int bl = m / B, b = m % B;
      const float* mcol = sMix + b * B * (CS + 1) + c;
      for (int j = 0; j < B; ++j) u = fmaf(mcol[j * (CS + 1)], sX[(bl * B + j) * (CS + 1) + c], u);
    }
    sUs[m * (CS + 1) + c] = u;
    sU[m * P.pk_r + q * CS + c] = __float2bfloat16_rn(u);
  }
  cluster.sync();

  // ---- gather the other CTAs' u slices ----
  gather_peers(cluster, sU, P.pk_r, CS, q, tid);
  __syncthreads();

  // ---- phase 2: SwiGLU on own hidden units: a = silu(u w_gate^T) * (u w_up^T) ----
  for (int it = warp; it < (MT / 16) * (HS / 8); it += THREADS / 32) {
    const int mt = it / (HS / 8), nt = it % (HS / 8);
    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mma(ag, sU, P.pk_r, mt * 16, sWg, P.pk_r, nt * 8, r);
    tile_mma(au, sU, P.pk_r, mt * 16, sWu, P.pk_r, nt * 8, r);
    const int g = lane / 4, t = lane % 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = mt * 16 + g + (e >= 2 ? 8 : 0);
      const int hh = nt * 8 + 2 * t + (e & 1);
      sA[m * P.pk_h + q * HS + hh] = __float2bfloat16_rn(silu(ag[e]) * au[e]);
    }
  }
  cluster.sync();

  // ---- gather the other CTAs' activation slices ----
  gather_peers(cluster, sA, P.pk_h, HS, q, tid);
  __syncthreads();

  // ---- phase 3: lat (own channels) = u + a . w_down^T, slots 1..B-1 ----
  for (int it = warp; it < (MT / 16) * (CS / 8); it += THREADS / 32) {
    const int mt = it / (CS / 8), nt = it % (CS / 8);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    tile_mma(acc, sA, P.pk_h, mt * 16, sWd, P.pk_h, nt * 8, H);
    const int g = lane / 4, t = lane % 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = mt * 16 + g + (e >= 2 ? 8 : 0);
      const int c = nt * 8 + 2 * t + (e & 1);
      if (m < rows && (m % B) != 0) {
        const int n = n0 + m / B, b = m % B;
        const float v = sUs[m * (CS + 1) + c] + acc[e];
        lat[((int64_t)n * (B - 1) + b - 1) * r + q * CS + c] = __float2bfloat16_rn(v);
      }
    }
  }
  cluster.sync();   // peers may still be reading this CTA's shared memory
}

}  // namespace

bool xp_latent_mma_ok(int r, int H, int B, xp_dtype dt) {
  if (dt != XP_BF16) return false;
  if (r % (8 * CL) != 0 || H % (8 * CL) != 0 || B > MT || B < 2) return false;
  return smem_plan(r, H, B).total <= 227 * 1024;
}

cudaError_t xp_launch_latent_mma(const xp_head* h, const int64_t* blk, const int64_t* am1,
                                 const float* xh, int N, void* lat, cudaStream_t s) {
  const Smem P = smem_plan(h->r, h->H, h->B);
  const int nb = MT / h->B;
  const int clusters = (N + nb - 1) / nb;
  cudaError_t e = cudaFuncSetAttribute(latent_mma_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, P.total);
  if (e != cudaSuccess) return e;
  e = xp_launch_pdl(latent_mma_kernel, dim3(clusters * CL), dim3(THREADS), (size_t)P.total, s, blk,
                    am1, xh, (const bf16*)h->w1, (const bf16*)h->w_lat, (const bf16*)h->mix,
                    (const bf16*)h->w_gate, (const bf16*)h->w_up, (const bf16*)h->w_down,
                    (bf16*)lat, N, h->B, h->r, h->H, h->V, h->err);
  return e != cudaSuccess ? e : cudaGetLastError();
}
