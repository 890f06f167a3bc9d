// Plain CUDA kernels of the pass: the mixer fold, the streaming init argmax, and SIMT versions of the latent stage and of the
// readout (used for fp32 heads and for shapes the tensor-core kernels do not
// tile).  All accumulate in fp32.
#include <math.h>

#include "xp_device.cuh"

using namespace xpd;
typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// fold: mix = raw * tril + I  (qwen3_xpress page, fold_from_raw_), in fp64,
// rounded once to the storage type.  raw * 0 + 0 turns -0 into +0 exactly as
// the tensor expression does.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_d(float* p, double v) { *p = (float)v; }
__device__ __forceinline__ void store_d(bf16* p, double v) { *p = __double2bfloat16(v); }

template <typename T>
__global__ void fold_kernel(const T* __restrict__ raw, T* __restrict__ mix, int r, int B) {
  const int total = r * B * B;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int j = i % B, b = (i / B) % B;
    const double v = (double)to_f(raw[i]);
    const double m = v * (j <= b ? 1.0 : 0.0) + (j == b ? 1.0 : 0.0);
    store_d(mix + i, m);
  }
}

cudaError_t xp_launch_fold(const void* raw, void* mix, int r, int B, xp_dtype dt, cudaStream_t s) {
  const int total = r * B * B;
  const int grid = (total + 255) / 256;
  if (dt == XP_BF16)
    fold_kernel<bf16><<<grid, 256, 0, s>>>((const bf16*)raw, (bf16*)mix, r, B);
  else
    fold_kernel<float><<<grid, 256, 0, s>>>((const float*)raw, (float*)mix, r, B);
  return cudaGetLastError();
}

// mixT[(b*B + j)*r + c] = mix[(c*B + b)*B + j]: the folded mixer with the channel
// innermost (a prepared layout, like the pages' mix_kjc), same storage type
template <typename T>
__global__ void mix_transpose_kernel(const T* __restrict__ mix, T* __restrict__ mixT, int r,
                                     int B) {
  const int total = r * B * B;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int c = i % r, bj = i / r;
    mixT[i] = mix[(int64_t)c * B * B + bj];
  }
}

cudaError_t xp_launch_mix_transpose(const void* mix, void* mixT, int r, int B, xp_dtype dt,
                                    cudaStream_t s) {
  const int grid = (r * B * B + 255) / 256;
  if (dt == XP_BF16)
    mix_transpose_kernel<bf16><<<grid, 256, 0, s>>>((const bf16*)mix, (bf16*)mixT, r, B);
  else
    mix_transpose_kernel<float><<<grid, 256, 0, s>>>((const float*)mix, (float*)mixT, r, B);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// init argmax: blk[n,0] = anchor[n]; blk[n,1+b] = argmax_v base[n,b,v]
// (qwen3_xpress page, jacobi_refine_greedy before the passes).  Grid
// (splits, rows); each CTA reduces one vocabulary chunk of one row, the last
// CTA of a row (ticket) publishes the winner and resets the row's partial.
// ---------------------------------------------------------------------------
template <typename T, bool VEC>
__global__ void __launch_bounds__(256) init_argmax_kernel(
    const T* __restrict__ base, int64_t sn, int64_t sb, int Bm1, int B, int V, int vchunk,
    const int64_t* __restrict__ anchor, int64_t* __restrict__ blk, float* __restrict__ win,
    unsigned long long* __restrict__ packed, unsigned* __restrict__ ticket, uint32_t* err) {
  __shared__ float sv[8];
  __shared__ int si[8];
  __shared__ int s_last;
  const int row = blockIdx.y;
  const int n = row / Bm1, b = row % Bm1;
  const T* p = base + (int64_t)n * sn + (int64_t)b * sb;
  const int v0 = blockIdx.x * vchunk;
  const int v1 = min(V, v0 + vchunk);
  float best = -INFINITY;
  int bi = 0x7FFFFFFF;
  int vtail = v0;
  if (VEC) {
    constexpr int E = 16 / sizeof(T);
    const int nvec = (v1 - v0) / E;
    constexpr int U = 4;                         // 16-byte loads per thread and batch
    const uint4* src = reinterpret_cast<const uint4*>(p + v0);
    const int stride = U * (int)blockDim.x;
    // two batches in flight: the next batch is loaded before this one is reduced
    uint4 q[U], qn[U];
    auto load = [&](uint4 (&dst)[U], int i0) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * (int)blockDim.x;
        dst[u] = i < nvec ? __ldcs(src + i) : make_uint4(0, 0, 0, 0);
      }
    };
    load(q, threadIdx.x);
    for (int i0 = threadIdx.x; i0 < nvec; i0 += stride) {
      load(qn, i0 + stride);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * (int)blockDim.x;
        if (i >= nvec) break;
        const T* e = reinterpret_cast<const T*>(&q[u]);
        if constexpr (sizeof(T) == 2) {
          // the chunk's maximum in packed bf16 first; its lowest index only when it wins
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&q[u]);
          const __nv_bfloat162 m2 = __hmax2(__hmax2(h2[0], h2[1]), __hmax2(h2[2], h2[3]));
          const float m = fmaxf(__low2float(m2), __high2float(m2));
          if (m > best) {
            int first = E - 1;
#pragma unroll
            for (int k = E - 1; k >= 0; --k)
              if (to_f(e[k]) == m) first = k;
            best = m;
            bi = v0 + i * E + first;
          }
        } else {
#pragma unroll
          for (int k = 0; k < E; ++k) {
            const float x = to_f(e[k]);
            if (x > best) { best = x; bi = v0 + i * E + k; }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) q[u] = qn[u];
    }
    vtail = v0 + nvec * E;
  }
  for (int v = vtail + threadIdx.x; v < v1; v += blockDim.x) {
    const float x = to_f(p[v]);
    if (better(x, v, best, bi)) { best = x; bi = v; }
  }
  warp_argmax(best, bi);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) { sv[w] = best; si[w] = bi; }
  __syncthreads();
  if (w == 0) {
    best = l < (int)(blockDim.x / 32) ? sv[l] : -INFINITY;
    bi = l < (int)(blockDim.x / 32) ? si[l] : 0x7FFFFFFF;
    warp_argmax(best, bi);
    if (l == 0) atomicMax(packed + row, pack_best(best, (uint32_t)bi));
  }
  if (arrive_last(ticket + row, gridDim.x, &s_last) && threadIdx.x == 0) {
    const unsigned long long pk = atomicExch(packed + row, 0ull);
    ticket[row] = 0u;
    blk[(int64_t)n * B + 1 + b] = (int64_t)packed_idx(pk);
    if (win) win[row] = packed_val(pk);
    if (b == 0 && anchor) blk[(int64_t)n * B] = checked_token(anchor[n], V, err);
  }
  // launched to overlap an independent predecessor: finish only after it has, so that
  // the kernels after this one see its results too (a no-op without the dependency)
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

cudaError_t xp_launch_init_argmax(const xp_head* h, const void* base, int64_t sn, int64_t sb,
                                  const int64_t* anchor, int N, int64_t* blk, float* win,
                                  unsigned long long* packed, unsigned* ticket, cudaStream_t s,
                                  bool overlap_prev) {
  const int Bm1 = h->B - 1, rows = N * Bm1, V = h->V;
  const size_t es = xp_elem(h->dtype);
  const int E = (int)(16 / es);
  // vectorised loads need every row start 16-byte aligned
  const bool vec = ((uintptr_t)base % 16 == 0) && (sn % E == 0) && (sb % E == 0);
  // at least two CTAs per SM, in chunks as long as possible (a multiple of 256*E): a
  // CTA's start and its reduction cost more than an uneven last wave (batched-decode,
  // 480 rows: one CTA per row, 28.2 us; two per row 31.2 us; five per row 32.8 us)
  const int unit = 256 * E;
  int splits = (2 * h->num_sms + rows - 1) / rows;
  int vchunk = (V + splits - 1) / splits;
  vchunk = ((vchunk + unit - 1) / unit) * unit;
  splits = (V + vchunk - 1) / vchunk;
  dim3 grid(splits, rows);
#define XP_INIT_LAUNCH(T, VEC)                                                                  \
  do {                                                                                          \
    if (overlap_prev)                                                                           \
      return xp_launch_pdl(init_argmax_kernel<T, VEC>, grid, dim3(256), 0, s, (const T*)base, sn, \
                           sb, Bm1, h->B, V, vchunk, anchor, blk, win, packed, ticket, h->err);  \
    init_argmax_kernel<T, VEC><<<grid, 256, 0, s>>>((const T*)base, sn, sb, Bm1, h->B, V,       \
                                                    vchunk, anchor, blk, win, packed, ticket,   \
                                                    h->err);                                    \
  } while (0)
  if (h->dtype == XP_BF16) {
    if (vec) XP_INIT_LAUNCH(bf16, true); else XP_INIT_LAUNCH(bf16, false);
  } else {
    if (vec) XP_INIT_LAUNCH(float, true); else XP_INIT_LAUNCH(float, false);
  }
#undef XP_INIT_LAUNCH
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SIMT latent: one CTA per block, fp32 in shared memory (xpress kernels page,
// _xpress_latent_kernel; qwen3_xpress page, _refine_latent).
//   prev[0] = am1[n], prev[b] = blk[n, b-1]
//   x[b]   = xh[n, b] + w_lat w1[prev[b]]
//   u[b,c] = sum_j mix[c, b, j] x[j, c]        (stored mixer is lower-triangular)
//   lat[b] = u[b] + w_down (silu(w_gate u[b]) * (w_up u[b]))   for b = 1..B-1
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) latent_simt_kernel(
    const int64_t* __restrict__ blk, const int64_t* __restrict__ am1, const float* __restrict__ xh,
    const T* __restrict__ w1, const T* __restrict__ wlat, const T* __restrict__ mix,
    const T* __restrict__ wg, const T* __restrict__ wu, const T* __restrict__ wd,
    T* __restrict__ lat, int B, int r, int H, int V, uint32_t* err) {
  extern __shared__ float sm[];
  float* e = sm;              // [B][r]  embeddings
  float* x = e + B * r;       // [B][r]  in_proj output
  float* u = x + B * r;       // [B][r]  mixed
  float* act = u + B * r;     // [B][H]  SwiGLU activations
  __shared__ int64_t prev[64];
  const int n = blockIdx.x;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int64_t t = b == 0 ? am1[n] : blk[(int64_t)n * B + b - 1];
    prev[b] = checked_token(t, V, err);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < B * r; i += blockDim.x) {
    const int b = i / r, k = i % r;
    e[i] = to_f(w1[prev[b] * r + k]);
  }
  __syncthreads();
  for (int c = threadIdx.x; c < r; c += blockDim.x) {
    for (int b = 0; b < B; ++b) {
      float a = xh[((int64_t)n * B + b) * r + c];
      for (int k = 0; k < r; ++k) a = fmaf(to_f(wlat[(int64_t)c * r + k]), e[b * r + k], a);
      x[b * r + c] = a;
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < r; c += blockDim.x) {
    for (int b = 0; b < B; ++b) {
      float a = 0.f;
      for (int j = 0; j < B; ++j) a = fmaf(to_f(mix[((int64_t)c * B + b) * B + j]), x[j * r + c], a);
      u[b * r + c] = a;
    }
  }
  __syncthreads();
  for (int q = threadIdx.x; q < H; q += blockDim.x) {
    for (int b = 1; b < B; ++b) {
      float g = 0.f, up = 0.f;
      for (int c = 0; c < r; ++c) {
        g = fmaf(to_f(wg[(int64_t)q * r + c]), u[b * r + c], g);
        up = fmaf(to_f(wu[(int64_t)q * r + c]), u[b * r + c], up);
      }
      act[b * H + q] = silu(g) * up;
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < r; c += blockDim.x) {
    for (int b = 1; b < B; ++b) {
      float a = u[b * r + c];
      for (int q = 0; q < H; ++q) a = fmaf(to_f(wd[(int64_t)c * H + q]), act[b * H + q], a);
      lat[((int64_t)n * (B - 1) + (b - 1)) * r + c] = from_f<T>(a);
    }
  }
}

cudaError_t xp_launch_latent_simt(const xp_head* h, const int64_t* blk, const int64_t* am1,
                                  const float* xh, int N, void* lat, cudaStream_t s) {
  const size_t smem = sizeof(float) * (size_t)h->B * (3 * h->r + h->H);
  cudaError_t e;
  if (h->dtype == XP_BF16) {
    e = cudaFuncSetAttribute(latent_simt_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    latent_simt_kernel<bf16><<<N, 256, smem, s>>>(
        blk, am1, xh, (const bf16*)h->w1, (const bf16*)h->w_lat, (const bf16*)h->mix,
        (const bf16*)h->w_gate, (const bf16*)h->w_up, (const bf16*)h->w_down, (bf16*)lat, h->B,
        h->r, h->H, h->V, h->err);
  } else {
    e = cudaFuncSetAttribute(latent_simt_kernel<float>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    latent_simt_kernel<float><<<N, 256, smem, s>>>(
        blk, am1, xh, (const float*)h->w1, (const float*)h->w_lat, (const float*)h->mix,
        (const float*)h->w_gate, (const float*)h->w_up, (const float*)h->w_down, (float*)lat,
        h->B, h->r, h->H, h->V, h->err);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SIMT readout + argmax (xpress kernels page, fused_add_argmax_to_blk, with
// the w2 matmul fused in): tile of 32 rows x 128 vocabulary ids, fp32 FMA.
// The logits live in registers only; per-row (max, id) partials merge with
// atomicMax and the last CTA of a row tile writes blk.  EMIT: the same tile writes
// the fp32 logits (the bias alone when base is null) instead.
// ---------------------------------------------------------------------------
constexpr int SR_RT = 32, SR_VT = 128, SR_KC = 32;

template <typename T, bool EMIT>
__global__ void __launch_bounds__(256) readout_simt_kernel(
    const T* __restrict__ lat, const T* __restrict__ base, int64_t sn, int64_t sb,
    const T* __restrict__ w2, int rows, int Bm1, int B, int V, int r, int64_t* __restrict__ blk,
    float* __restrict__ win, unsigned long long* __restrict__ packed, unsigned* __restrict__ ticket,
    float* __restrict__ out, int64_t ldo) {
  __shared__ float Ls[SR_KC][SR_RT];
  __shared__ float Ws[SR_KC][SR_VT + 1];
  __shared__ int s_last;
  const int tid = threadIdx.x, w = tid / 32, l = tid % 32;
  const int v0 = blockIdx.x * SR_VT, row0 = blockIdx.y * SR_RT;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < r; k0 += SR_KC) {
    for (int i = tid; i < SR_RT * SR_KC; i += 256) {
      const int rr = i / SR_KC, kk = i % SR_KC;
      const int gr = row0 + rr, gk = k0 + kk;
      Ls[kk][rr] = (gr < rows && gk < r) ? to_f(lat[(int64_t)gr * r + gk]) : 0.f;
    }
    for (int i = tid; i < SR_VT * SR_KC; i += 256) {
      const int vv = i / SR_KC, kk = i % SR_KC;
      const int gv = v0 + vv, gk = k0 + kk;
      Ws[kk][vv] = (gv < V && gk < r) ? to_f(w2[(int64_t)gv * r + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < SR_KC; ++kk) {
      float a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = Ls[kk][w * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bb[j] = Ws[kk][l + 32 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }
  if constexpr (EMIT) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = row0 + w * 4 + i;
      if (row >= rows) continue;
      const int n = row / Bm1, b = row % Bm1;
      const T* bp = base ? base + (int64_t)n * sn + (int64_t)b * sb : nullptr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = v0 + l + 32 * j;
        if (v < V) out[(int64_t)row * ldo + v] = acc[i][j] + (bp ? to_f(bp[v]) : 0.f);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = row0 + w * 4 + i;
      float best = -INFINITY;
      int bi = 0x7FFFFFFF;
      if (row < rows) {
        const int n = row / Bm1, b = row % Bm1;
        const T* bp = base + (int64_t)n * sn + (int64_t)b * sb;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int v = v0 + l + 32 * j;
          if (v < V) {
            const float sc = acc[i][j] + to_f(bp[v]);
            if (better(sc, v, best, bi)) { best = sc; bi = v; }
          }
        }
      }
      warp_argmax(best, bi);
      if (l == 0 && row < rows) atomicMax(packed + row, pack_best(best, (uint32_t)bi));
    }
    if (arrive_last(ticket + blockIdx.y, gridDim.x, &s_last)) {
      if (tid < SR_RT) {
        const int row = row0 + tid;
        if (row < rows) {
          const unsigned long long pk = atomicExch(packed + row, 0ull);
          const int n = row / Bm1, b = row % Bm1;
          blk[(int64_t)n * B + 1 + b] = (int64_t)packed_idx(pk);
          if (win) win[row] = packed_val(pk);
        }
      }
      if (tid == 0) ticket[blockIdx.y] = 0u;
    }
  }
}

cudaError_t xp_launch_readout_simt(const xp_head* h, const void* lat, const void* base, int64_t sn,
                                   int64_t sb, int N, int64_t* blk, float* win,
                                   unsigned long long* packed, unsigned* ticket, cudaStream_t s) {
  const int Bm1 = h->B - 1, rows = N * Bm1;
  dim3 grid((h->V + SR_VT - 1) / SR_VT, (rows + SR_RT - 1) / SR_RT);
  if (h->dtype == XP_BF16)
    readout_simt_kernel<bf16, false><<<grid, 256, 0, s>>>(
        (const bf16*)lat, (const bf16*)base, sn, sb, (const bf16*)h->w2, rows, Bm1, h->B, h->V,
        h->r, blk, win, packed, ticket, nullptr, 0);
  else
    readout_simt_kernel<float, false><<<grid, 256, 0, s>>>(
        (const float*)lat, (const float*)base, sn, sb, (const float*)h->w2, rows, Bm1, h->B, h->V,
        h->r, blk, win, packed, ticket, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t xp_launch_logits_simt(const xp_head* h, const void* lat, const void* base, int64_t sn,
                                  int64_t sb, int N, float* out, int64_t ldo, cudaStream_t s) {
  const int Bm1 = h->B - 1, rows = N * Bm1;
  dim3 grid((h->V + SR_VT - 1) / SR_VT, (rows + SR_RT - 1) / SR_RT);
  if (h->dtype == XP_BF16)
    readout_simt_kernel<bf16, true><<<grid, 256, 0, s>>>(
        (const bf16*)lat, (const bf16*)base, sn, sb, (const bf16*)h->w2, rows, Bm1, h->B, h->V,
        h->r, nullptr, nullptr, nullptr, nullptr, out, ldo);
  else
    readout_simt_kernel<float, true><<<grid, 256, 0, s>>>(
        (const float*)lat, (const float*)base, sn, sb, (const float*)h->w2, rows, Bm1, h->B, h->V,
        h->r, nullptr, nullptr, nullptr, nullptr, out, ldo);
  return cudaGetLastError();
}
