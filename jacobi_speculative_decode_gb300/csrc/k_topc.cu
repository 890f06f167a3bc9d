// Top-C path (qwen3_xpress page, the top-C branch of jacobi_refine_greedy;
// xpress kernels page, _xpress_topc_argmax_to_blk_kernel):
//   once per step: per draft row, the C largest base values (ties at the
//   boundary to the lower id) in ascending id order, their base values, and
//   optionally the w2 rows of the candidates;
//   per pass: blk[n, 1+b] = cand[k*], k* = argmax_k base_c[k] + w2[cand[k]] . lat.
#include "xp_device.cuh"

using namespace xpd;
typedef __nv_bfloat16 bf16;

namespace {

constexpr int TS_THREADS = 512;
constexpr int TS_ITEMS = 8;   // contiguous elements per thread per chunk

// Orderable radix keys; -0 shares the key of +0.
__device__ __forceinline__ uint32_t radix_key(bf16 x) {
  uint32_t u = __bfloat16_as_ushort(x);
  if (u == 0x8000u) u = 0u;
  return (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
}
__device__ __forceinline__ uint32_t radix_key(float x) { return f2key(x); }

template <typename T> struct KeyBits;
template <> struct KeyBits<bf16> { static constexpr int value = 16; };
template <> struct KeyBits<float> { static constexpr int value = 32; };

// Inclusive block scan of one uint32 per thread (512 threads = 16 warps).
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t x, uint32_t* s_warp, uint32_t* total) {
  const int l = threadIdx.x % 32, w = threadIdx.x / 32;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (l >= o) x += y;
  }
  if (l == 31) s_warp[w] = x;
  __syncthreads();
  if (w == 0) {
    uint32_t t = l < TS_THREADS / 32 ? s_warp[l] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (l >= o) t += y;
    }
    if (l < TS_THREADS / 32) s_warp[l] = t;   // inclusive warp prefix
  }
  __syncthreads();
  if (w > 0) x += s_warp[w - 1];
  *total = s_warp[TS_THREADS / 32 - 1];
  __syncthreads();
  return x;
}

template <typename T>
__global__ void __launch_bounds__(TS_THREADS) topc_select_kernel(
    const T* __restrict__ base, int64_t sn, int64_t sb, int Bm1, int B, int V, int C,
    int64_t* __restrict__ cand, T* __restrict__ base_c, int64_t* __restrict__ blk,
    const int64_t* __restrict__ anchor, uint32_t* err) {
  constexpr int KB = KeyBits<T>::value;
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_warp[32];
  __shared__ uint32_t s_sel[3];   // prefix, remaining quota, count above the prefix
  __shared__ float s_bv[TS_THREADS / 32];
  __shared__ int s_bi[TS_THREADS / 32];
  const int row = blockIdx.x;
  const int n = row / Bm1, b = row % Bm1;
  const T* p = base + (int64_t)n * sn + (int64_t)b * sb;
  const int tid = threadIdx.x;

  // ---- radix select of the C-th largest key, 8 bits at a time ----
  uint32_t prefix = 0, pmask = 0, remaining = (uint32_t)C, above = 0;
  for (int shift = KB - 8; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += TS_THREADS) hist[i] = 0;
    __syncthreads();
    for (int v = tid; v < V; v += TS_THREADS) {
      const uint32_t k = radix_key(p[v]);
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t cum = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (cum + hist[d] >= remaining) break;
        cum += hist[d];
      }
      s_sel[0] = prefix | ((uint32_t)d << shift);
      s_sel[1] = remaining - cum;
      s_sel[2] = above + cum;
    }
    __syncthreads();
    prefix = s_sel[0];
    remaining = s_sel[1];
    above = s_sel[2];
    pmask |= 255u << shift;
    __syncthreads();
  }
  // keys > prefix: all `above` of them selected; keys == prefix: the first
  // `remaining` in id order.
  const uint32_t thr = prefix, quota = remaining;

  // ---- ordered compaction in id order + the row argmax ----
  uint32_t g_run = 0, e_run = 0;          // gt / eq counts of earlier chunks
  float best = -INFINITY;
  int bi = 0x7FFFFFFF;
  int64_t* crow = cand + (int64_t)row * C;
  T* brow = base_c + (int64_t)row * C;
  for (int c0 = 0; c0 < V; c0 += TS_THREADS * TS_ITEMS) {
    const int v0 = c0 + tid * TS_ITEMS;
    uint32_t keys[TS_ITEMS];
    T vals[TS_ITEMS];
    uint32_t ngt = 0, neq = 0;
#pragma unroll
    for (int i = 0; i < TS_ITEMS; ++i) {
      const int v = v0 + i;
      if (v < V) {
        vals[i] = p[v];
        keys[i] = radix_key(vals[i]);
        ngt += keys[i] > thr;
        neq += keys[i] == thr;
        const float x = to_f(vals[i]);
        if (x > best) { best = x; bi = v; }
      } else {
        keys[i] = 0;
      }
    }
    uint32_t tot;
    const uint32_t incl = block_incl_scan(ngt | (neq << 16), s_warp, &tot);
    const uint32_t excl = incl - (ngt | (neq << 16));
    uint32_t gb = g_run + (excl & 0xFFFFu), eb = e_run + (excl >> 16);
    uint32_t pos = gb + min(eb, quota);
#pragma unroll
    for (int i = 0; i < TS_ITEMS; ++i) {
      const int v = v0 + i;
      if (v >= V) break;
      bool take = false;
      if (keys[i] > thr) take = true;
      else if (keys[i] == thr) { take = eb < quota; ++eb; }
      if (take) { crow[pos] = v; brow[pos] = vals[i]; ++pos; }
    }
    g_run += tot & 0xFFFFu;
    e_run += tot >> 16;
  }
  if (blk) {
    warp_argmax(best, bi);
    if (tid % 32 == 0) { s_bv[tid / 32] = best; s_bi[tid / 32] = bi; }
    __syncthreads();
    if (tid < 32) {
      best = tid < TS_THREADS / 32 ? s_bv[tid] : -INFINITY;
      bi = tid < TS_THREADS / 32 ? s_bi[tid] : 0x7FFFFFFF;
      warp_argmax(best, bi);
      if (tid == 0) {
        blk[(int64_t)n * B + 1 + b] = bi;
        if (b == 0 && anchor) blk[(int64_t)n * B] = checked_token(anchor[n], V, err);
      }
    }
  }
}

// w2c[row, k, :] = w2[cand[row, k], :]  -- one warp per candidate row, 16-byte copies
template <bool VEC>
__global__ void __launch_bounds__(256) gather_rows_kernel(const char* __restrict__ w2,
                                                          const int64_t* __restrict__ cand,
                                                          char* __restrict__ w2c, int64_t total,
                                                          int row_bytes, int V, uint32_t* err) {
  const int lane = threadIdx.x % 32;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int64_t nwarps = (int64_t)gridDim.x * blockDim.x / 32;
  for (int64_t k = warp0; k < total; k += nwarps) {
    const int64_t id = checked_token(cand[k], V, err);
    const char* src = w2 + id * row_bytes;
    char* dst = w2c + k * row_bytes;
    if (VEC) {
      for (int o = lane * 16; o < row_bytes; o += 32 * 16)
        *reinterpret_cast<uint4*>(dst + o) = __ldg(reinterpret_cast<const uint4*>(src + o));
    } else {
      for (int o = lane; o < row_bytes; o += 32) dst[o] = src[o];
    }
  }
}

// Per pass: one CTA per draft row.  Groups of 8 lanes score one candidate.
template <typename T>
__global__ void __launch_bounds__(256) topc_readout_kernel(
    const T* __restrict__ lat, const T* __restrict__ base_c, const int64_t* __restrict__ cand,
    const T* __restrict__ w2c, const T* __restrict__ w2, int Bm1, int B, int V, int C, int r,
    int64_t* __restrict__ blk, float* __restrict__ win, uint32_t* err) {
  extern __shared__ float s_lat[];
  __shared__ float s_bv[8];
  __shared__ int s_bi[8];
  __shared__ int s_bk[8];
  const int row = blockIdx.x;
  const int n = row / Bm1, b = row % Bm1;
  for (int c = threadIdx.x; c < r; c += blockDim.x) s_lat[c] = to_f(lat[(int64_t)row * r + c]);
  __syncthreads();
  const int g = threadIdx.x / 8, gl = threadIdx.x % 8;   // 32 groups of 8 lanes
  float best = -INFINITY;
  int bid = 0x7FFFFFFF, bk = -1;
  const int64_t* crow = cand + (int64_t)row * C;
  const T* bcrow = base_c + (int64_t)row * C;
  constexpr int E = 16 / sizeof(T);
  const bool vec = (r % (8 * E)) == 0;
  for (int k0 = 0; k0 < C; k0 += 32) {     // uniform trip count: shuffles see full warps
    const int k = k0 + g;
    const bool ok = k < C;
    float acc = 0.f;
    int64_t id = 0;
    if (ok) {
      id = checked_token(crow[k], V, err);
      const T* wr = w2c ? w2c + ((int64_t)row * C + k) * r : w2 + id * r;
      if (vec) {
        for (int q = gl; q < r / E; q += 8) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(wr) + q);
          const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
          for (int i = 0; i < E; ++i) acc = fmaf(to_f(e[i]), s_lat[q * E + i], acc);
        }
      } else {
        for (int c = gl; c < r; c += 8) acc = fmaf(to_f(wr[c]), s_lat[c], acc);
      }
    }
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 2);
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 4);
    if (ok) {
      const float sc = to_f(bcrow[k]) + acc;
      if (better(sc, (int)id, best, bid)) { best = sc; bid = (int)id; bk = k; }
    }
  }
  // reduce over the 8-lane groups of a warp, then over warps (ties -> lower vocab id)
#pragma unroll
  for (int o = 8; o < 32; o <<= 1) {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, best, o);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, bid, o);
    const int ok = __shfl_xor_sync(0xFFFFFFFFu, bk, o);
    if (better(ov, oi, best, bid)) { best = ov; bid = oi; bk = ok; }
  }
  const int w = threadIdx.x / 32;
  if (threadIdx.x % 32 == 0) { s_bv[w] = best; s_bi[w] = bid; s_bk[w] = bk; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i)
      if (better(s_bv[i], s_bi[i], best, bid)) { best = s_bv[i]; bid = s_bi[i]; bk = s_bk[i]; }
    blk[(int64_t)n * B + 1 + b] = bid;
    if (win) win[row] = best;
  }
}

}  // namespace

cudaError_t xp_launch_topc_gather(const xp_head* h, const void* base, int64_t sn, int64_t sb, int N,
                                  int C, int64_t* cand, void* base_c, void* w2c, int64_t* blk,
                                  const int64_t* anchor, cudaStream_t s) {
  const int Bm1 = h->B - 1, rows = N * Bm1;
  if (h->dtype == XP_BF16)
    topc_select_kernel<bf16><<<rows, TS_THREADS, 0, s>>>((const bf16*)base, sn, sb, Bm1, h->B,
                                                         h->V, C, cand, (bf16*)base_c, blk, anchor,
                                                         h->err);
  else
    topc_select_kernel<float><<<rows, TS_THREADS, 0, s>>>((const float*)base, sn, sb, Bm1, h->B,
                                                          h->V, C, cand, (float*)base_c, blk,
                                                          anchor, h->err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !w2c) return e;
  const int row_bytes = (int)(h->r * xp_elem(h->dtype));
  const int64_t total = (int64_t)rows * C;
  const int grid = (int)std::min<int64_t>((total + 7) / 8, (int64_t)h->num_sms * 16);
  const bool vec = row_bytes % 16 == 0 && (uintptr_t)w2c % 16 == 0;
  if (vec)
    gather_rows_kernel<true><<<grid, 256, 0, s>>>((const char*)h->w2, cand, (char*)w2c, total,
                                                  row_bytes, h->V, h->err);
  else
    gather_rows_kernel<false><<<grid, 256, 0, s>>>((const char*)h->w2, cand, (char*)w2c, total,
                                                   row_bytes, h->V, h->err);
  return cudaGetLastError();
}

cudaError_t xp_launch_topc_readout(const xp_head* h, const void* lat, const void* base_c,
                                   const int64_t* cand, const void* w2c, int N, int C,
                                   int64_t* blk, float* win, cudaStream_t s) {
  const int Bm1 = h->B - 1, rows = N * Bm1;
  const size_t smem = sizeof(float) * h->r;
  if (h->dtype == XP_BF16)
    topc_readout_kernel<bf16><<<rows, 256, smem, s>>>(
        (const bf16*)lat, (const bf16*)base_c, cand, (const bf16*)w2c, (const bf16*)h->w2, Bm1,
        h->B, h->V, C, h->r, blk, win, h->err);
  else
    topc_readout_kernel<float><<<rows, 256, smem, s>>>(
        (const float*)lat, (const float*)base_c, cand, (const float*)w2c, (const float*)h->w2,
        Bm1, h->B, h->V, C, h->r, blk, win, h->err);
  return cudaGetLastError();
}
