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

// the value a radix key stands for (+0 for the shared key of -0 and +0)
__device__ __forceinline__ float key_value(uint32_t k, bf16*) {
  const uint32_t u = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
  return __uint_as_float(u << 16);
}
__device__ __forceinline__ float key_value(uint32_t k, float*) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// the stored value a radix key came from (exact; a zero key is read from `p` instead,
// since -0 and +0 share it)
__device__ __forceinline__ bf16 key_store(uint32_t k, bf16*) {
  return __float2bfloat16_rn(key_value(k, (bf16*)nullptr));
}
__device__ __forceinline__ float key_store(uint32_t k, float*) {
  return key_value(k, (float*)nullptr);
}
// bit i set when x[i] >= t (packed bf16 pair compares for bf16)
__device__ __forceinline__ uint32_t ge_mask8(const bf16 (&x)[8], float t) {
  const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(x);
  const __nv_bfloat162 t2 = __float2bfloat162_rn(t);   // t is a bf16 value: exact
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t g = __hge2_mask(v[q], t2);            // 0xFFFF per true half
    m |= ((g & 1u) | ((g >> 15) & 2u)) << (2 * q);
  }
  return m;
}
__device__ __forceinline__ uint32_t ge_mask8(const float (&x)[8], float t) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m |= (x[i] >= t ? 1u : 0u) << i;
  return m;
}
// largest of 8 values (packed bf16 pairs for bf16)
__device__ __forceinline__ float max8(const bf16 (&x)[8]) {
  const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(x);
  const __nv_bfloat162 m = __hmax2(__hmax2(v[0], v[1]), __hmax2(v[2], v[3]));
  return fmaxf(__low2float(m), __high2float(m));
}
__device__ __forceinline__ float max8(const float (&x)[8]) {
  float m = x[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, x[i]);
  return m;
}

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

// 8 consecutive elements of a row, from one or two 16-byte loads when VEC (the row
// start is 16-byte aligned) and the chunk lies inside the row, else element by element
template <typename T, bool VEC>
__device__ __forceinline__ void load8(const T* __restrict__ p, int v0, int V, T (&x)[8]) {
  if (VEC && v0 + 8 <= V) {
    constexpr int E = 16 / sizeof(T);
#pragma unroll
    for (int q = 0; q < 8 / E; ++q) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(p + v0) + q);
      const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int i = 0; i < E; ++i) x[q * E + i] = e[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = v0 + i < V ? p[v0 + i] : T(0);
  }
}

constexpr int TS_CAP = 2048;      // candidates one row may collect on the fast path
constexpr int TS_HISTS = 4;       // radix histograms per CTA (shared by TS_THREADS/32/TS_HISTS warps)
constexpr int TS_SAMPLE = 8192;   // leading elements of a row that estimate a threshold

// prefix|bin of the remaining-th largest key, given this pass's 256-bin histogram
// (called by all 32 lanes of one warp; lane l owns bins [8l, 8l+8); writes
// s_sel = {prefix, remaining, count above})
__device__ __forceinline__ void radix_pick(const uint32_t* hist, uint32_t prefix, int shift,
                                           uint32_t remaining, uint32_t above, uint32_t* s_sel) {
  const int l = threadIdx.x % 32;
  uint32_t h[8], mine = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) { h[i] = hist[8 * l + i]; mine += h[i]; }
  // suffix sums over lanes: sum of bins >= 8l
  uint32_t suf = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, suf, o);
    if (l + o < 32) suf += y;
  }
  // the bin lies in the highest lane whose suffix reaches `remaining` (lane 0 if none)
  const uint32_t reach = __ballot_sync(0xFFFFFFFFu, suf >= remaining);
  const int L = reach ? 31 - __clz(reach) : 0;
  if (l == L) {
    uint32_t cum = suf - mine;             // bins above this lane's range
    int d = 8 * l + 7;
    for (; d > 0; --d) {
      const uint32_t hd = h[d - 8 * l];
      if (cum + hd >= remaining || d == 8 * l) break;
      cum += hd;
    }
    // d == 8l with the target not reached only happens in lane 0 (bin 0 takes the rest)
    s_sel[0] = prefix | ((uint32_t)d << shift);
    s_sel[1] = remaining - cum;
    s_sel[2] = above + cum;
  }
}

// Per draft row (one CTA of 512 threads):
//  fast path (C <= TS_CAP / 2 and the id bitmaps fit in shared memory):
//   1. t0 = the Ts-th largest key of the row's first TS_SAMPLE elements, Ts about
//      twice the share of C the sample should hold, so that about 2C elements of the
//      row have keys >= t0;
//   2. one pass over the row collects (key, id) of every element with key >= t0 and
//      the row's argmax;
//   3. if C <= collected <= TS_CAP, the C-th largest key thr of the row is the C-th
//      largest collected key (every key >= thr is >= t0), found by radix select over
//      the collected keys; the candidates are all keys > thr plus the `quota` lowest
//      ids with key == thr (ranked among themselves), marked in an id bitmap and
//      emitted in id order by a prefix count over the bitmap;
//  otherwise (and as fallback): radix select over the whole row, then an ordered
//  compaction pass.
template <typename T, bool VEC>
__global__ void __launch_bounds__(TS_THREADS, 2) topc_select_kernel(
    const T* __restrict__ base, int64_t sn, int64_t sb, int Bm1, int B, int V, int C, int fast_ok,
    int64_t* __restrict__ cand, T* __restrict__ base_c, int64_t* __restrict__ blk,
    const int64_t* __restrict__ anchor, uint32_t* err) {
  constexpr int KB = KeyBits<T>::value;
  constexpr int NW = TS_THREADS / 32;
  extern __shared__ __align__(16) uint32_t ts_dyn[];
  // TS_HISTS histograms, each shared by the warps w with w % TS_HISTS equal
  uint32_t (*whist)[256] = reinterpret_cast<uint32_t (*)[256]>(ts_dyn);
  uint32_t* ckey = ts_dyn + TS_HISTS * 256;
  int* cid = reinterpret_cast<int*>(ckey + TS_CAP);
  int* eqid = cid + TS_CAP;                                     // ids whose key == thr
  const int W = (V + 31) / 32;
  uint32_t* selm = reinterpret_cast<uint32_t*>(eqid + TS_CAP);  // selected ids, one bit each
  uint16_t* wpre = reinterpret_cast<uint16_t*>(selm + W);         // selected ids below word w
  __shared__ uint32_t s_warp[32];
  __shared__ uint32_t s_sel[3];   // prefix, remaining quota, count above the prefix
  __shared__ uint32_t s_count;
  __shared__ float s_bv[NW];
  __shared__ int s_bi[NW];
  const int row = blockIdx.x;
  const int n = row / Bm1, b = row % Bm1;
  const T* p = base + (int64_t)n * sn + (int64_t)b * sb;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  int64_t* crow = cand + (int64_t)row * C;
  T* brow = base_c + (int64_t)row * C;
  float best = -INFINITY;
  int bi = 0x7FFFFFFF;

  // one radix step over keys supplied by `each(f)` (f(key) for every live key)
  auto radix = [&](auto&& each, uint32_t need, uint32_t& thr_out, uint32_t& quota_out) {
    uint32_t prefix = 0, pmask = 0, remaining = need, above = 0;
    for (int shift = KB - 8; shift >= 0; shift -= 8) {
      for (int i = tid; i < TS_HISTS * 256; i += TS_THREADS) (&whist[0][0])[i] = 0;
      __syncthreads();
      each([&](uint32_t k) {
        if ((k & pmask) == prefix) atomicAdd(&whist[warp % TS_HISTS][(k >> shift) & 255u], 1u);
      });
      __syncthreads();
      if (tid < 256) {
        uint32_t t = 0;
#pragma unroll
        for (int w = 0; w < TS_HISTS; ++w) t += whist[w][tid];
        whist[0][tid] = t;
      }
      __syncthreads();
      if (warp == 0) radix_pick(whist[0], prefix, shift, remaining, above, s_sel);
      __syncthreads();
      prefix = s_sel[0];
      remaining = s_sel[1];
      above = s_sel[2];
      pmask |= 255u << shift;
      __syncthreads();
    }
    thr_out = prefix;
    quota_out = remaining;
  };

  bool fast = fast_ok != 0;
  uint32_t thr = 0, quota = 0;
  if (fast) {
    // ---- 1. threshold estimate from the leading sample ----
    const int Sn = min(TS_SAMPLE, V);
    const uint32_t Ts =
        (uint32_t)min((int64_t)Sn, (2 * (int64_t)C * Sn + V - 1) / V + 16);
    uint32_t sk[TS_SAMPLE / TS_THREADS];
#pragma unroll
    for (int h = 0; h < TS_SAMPLE / TS_THREADS / 8; ++h) {
      T x[8];
      const int v0 = tid * (TS_SAMPLE / TS_THREADS) + h * 8;
      load8<T, VEC>(p, v0, Sn, x);
#pragma unroll
      for (int i = 0; i < 8; ++i) sk[h * 8 + i] = v0 + i < Sn ? radix_key(x[i]) : 0xFFFFFFFFu;
    }
    uint32_t t0, unused;
    radix([&](auto&& f) {
#pragma unroll
      for (int i = 0; i < TS_SAMPLE / TS_THREADS; ++i)
        if (sk[i] != 0xFFFFFFFFu) f(sk[i]);
    }, Ts, t0, unused);

    // ---- 2. collect every element with key >= t0: a chunk of 8 is looked at one by
    // one only when its maximum reaches the threshold (about 2C of V elements do) ----
    if (tid == 0) s_count = 0;
    __syncthreads();
    const float t0v = key_value(t0, (T*)nullptr);
    auto keep = [&](uint32_t k, int v) {
      const uint32_t slot = atomicAdd(&s_count, 1u);
      if (slot < (uint32_t)TS_CAP) { ckey[slot] = k; cid[slot] = v; }
    };
    if constexpr (VEC && sizeof(T) == 2) {
      // bf16 rows: batches of 4 raw 16-byte words per thread, the next batch loaded
      // before this one is tested (two batches in flight), packed-pair tests
      constexpr int U = 4;
      const __nv_bfloat162 t2 = __float2bfloat162_rn(t0v);   // t0v is a bf16 value: exact
      uint4 w[U], wn[U];
      auto load = [&](uint4 (&dst)[U], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v0 = c0 + u * TS_THREADS * 8;
          dst[u] = v0 + 8 <= V ? __ldg(reinterpret_cast<const uint4*>(p + v0))
                               : make_uint4(0, 0, 0, 0);
        }
      };
      load(w, tid * 8);
      for (int c0 = tid * 8; c0 < V; c0 += U * TS_THREADS * 8) {
        load(wn, c0 + U * TS_THREADS * 8);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v0 = c0 + u * TS_THREADS * 8;
          const uint32_t q[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(q);
          const __nv_bfloat162 m2 = __hmax2(__hmax2(h2[0], h2[1]), __hmax2(h2[2], h2[3]));
          if (fmaxf(__low2float(m2), __high2float(m2)) >= t0v && v0 + 8 <= V) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t g = __hge2_mask(h2[e], t2);
              if (g & 1u) keep(radix_key(__low2bfloat16(h2[e])), v0 + 2 * e);
              if (g & 0x10000u) keep(radix_key(__high2bfloat16(h2[e])), v0 + 2 * e + 1);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) w[u] = wn[u];
      }
      // the ragged end of the row (fewer than 8 elements), element by element
      for (int v = (V / 8) * 8 + tid; v < V; v += TS_THREADS)
        if (to_f(p[v]) >= t0v) keep(radix_key(p[v]), v);
    } else {
      constexpr int U = 4;                     // chunks of 8 in flight
      for (int c0 = tid * 8; c0 < V; c0 += U * TS_THREADS * 8) {
        T x[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u)            // past-the-row slots read as 0: checked below
          load8<T, VEC>(p, c0 + u * TS_THREADS * 8, V, x[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v0 = c0 + u * TS_THREADS * 8;
          if (max8(x[u]) >= t0v) {
            uint32_t m = ge_mask8(x[u], t0v);
            if (v0 + 8 > V) m &= (1u << max(0, V - v0)) - 1u;   // slots past the row
#pragma unroll
            for (int i = 0; i < 8; ++i)                          // static indices: registers
              if (m & (1u << i)) keep(radix_key(x[u][i]), v0 + i);
          }
        }
      }
    }
    __syncthreads();
    const uint32_t ncol = s_count;
    fast = ncol >= (uint32_t)C && ncol <= (uint32_t)TS_CAP;   // CTA-uniform

    if (fast) {
      // the row maximum is among the collected keys (it is >= t0): its lowest id
      for (uint32_t j = tid; j < ncol; j += TS_THREADS) {
        const float xv = key_value(ckey[j], (T*)nullptr);
        if (better(xv, cid[j], best, bi)) { best = xv; bi = cid[j]; }
      }
      // ---- 3. the C-th largest collected key, then the id bitmaps ----
      radix([&](auto&& f) {
        for (uint32_t j = tid; j < ncol; j += TS_THREADS) f(ckey[j]);
      }, (uint32_t)C, thr, quota);
      if (tid == 0) s_count = 0;
      for (int w = tid; w < W; w += TS_THREADS) selm[w] = 0;
      __syncthreads();
      for (uint32_t j = tid; j < ncol; j += TS_THREADS) {
        const uint32_t k = ckey[j];
        const int id = cid[j];
        if (k > thr) atomicOr(&selm[id >> 5], 1u << (id & 31));
        else if (k == thr) eqid[atomicAdd(&s_count, 1u)] = id;
      }
      __syncthreads();
      // of the boundary key, the `quota` lowest ids: rank each by the lower ids
      const uint32_t neq = s_count;
      for (uint32_t j = tid; j < neq; j += TS_THREADS) {
        const int id = eqid[j];
        uint32_t rank = 0;
        for (uint32_t i = 0; i < neq; ++i) rank += eqid[i] < id;
        if (rank < quota) atomicOr(&selm[id >> 5], 1u << (id & 31));
      }
      __syncthreads();
      const int wpt = (W + TS_THREADS - 1) / TS_THREADS, w0 = tid * wpt, w1 = min(W, w0 + wpt);
      uint32_t cnt, tot;
      // emit the selection in id order: every bitmap word's exclusive prefix count, then
      // each selected collected entry writes itself at its rank (its value comes from
      // its key, not from another read of the row)
      cnt = 0;
      for (int w = w0; w < w1; ++w) cnt += __popc(selm[w]);
      uint32_t pos = block_incl_scan(cnt, s_warp, &tot) - cnt;
      for (int w = w0; w < w1; ++w) {
        wpre[w] = (uint16_t)pos;
        pos += __popc(selm[w]);
      }
      __syncthreads();
      const uint32_t zkey = radix_key(T(0.0f));
      for (uint32_t j = tid; j < ncol; j += TS_THREADS) {
        const uint32_t k = ckey[j];
        const int id = cid[j];
        const uint32_t word = selm[id >> 5], bit = 1u << (id & 31);
        if (word & bit) {
          const uint32_t at = wpre[id >> 5] + __popc(word & (bit - 1u));
          crow[at] = id;
          brow[at] = k == zkey ? p[id] : key_store(k, (T*)nullptr);
        }
      }
    }
  }

  if (!fast) {
    // ---- fallback: radix select over the whole row ----
    radix([&](auto&& f) {
      for (int c0 = 0; c0 < V; c0 += TS_THREADS * 8) {
        const int v0 = c0 + tid * 8;
        T x[8];
        load8<T, VEC>(p, v0, V, x);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (v0 + i < V) f(radix_key(x[i]));
      }
    }, (uint32_t)C, thr, quota);
    // keys > thr: all selected; keys == thr: the first `quota` in id order

    // ---- ordered compaction in id order + the row argmax ----
    uint32_t g_run = 0, e_run = 0;          // gt / eq counts of earlier chunks
    best = -INFINITY;
    bi = 0x7FFFFFFF;
    for (int c0 = 0; c0 < V; c0 += TS_THREADS * TS_ITEMS) {
      const int v0 = c0 + tid * TS_ITEMS;
      uint32_t keys[TS_ITEMS];
      T vals[TS_ITEMS];
      uint32_t ngt = 0, neq = 0;
      load8<T, VEC>(p, v0, V, vals);
#pragma unroll
      for (int i = 0; i < TS_ITEMS; ++i) {
        const int v = v0 + i;
        if (v < V) {
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
  }
  if (blk) {
    warp_argmax(best, bi);
    if (lane == 0) { s_bv[warp] = best; s_bi[warp] = bi; }
    __syncthreads();
    if (tid < 32) {
      best = tid < NW ? s_bv[tid] : -INFINITY;
      bi = tid < NW ? s_bi[tid] : 0x7FFFFFFF;
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
  if (VEC && row_bytes == 32 * 16) {
    // one 16-byte piece per lane and row; 4 rows per step so that 4 loads are in flight
    constexpr int U = 4;
    for (int64_t k0 = warp0; k0 < total; k0 += U * nwarps) {
      int64_t id[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t k = k0 + u * nwarps;
        id[u] = k < total ? checked_token(cand[k], V, err) : -1;
      }
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (id[u] >= 0) v[u] = __ldg(reinterpret_cast<const uint4*>(w2 + id[u] * row_bytes) + lane);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (id[u] >= 0)
          reinterpret_cast<uint4*>(w2c + (k0 + u * nwarps) * row_bytes)[lane] = v[u];
    }
    return;
  }
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
// NQ > 0: r = NQ * 8 lanes * (16 / sizeof(T)) exactly; every lane issues its NQ
// 16-byte loads of the candidate's w2 row together, the base value is loaded beside
// them, and the next candidate's id is loaded while this one is scored.
template <typename T, int NQ>
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
  int64_t id_next = g < C ? crow[g] : 0;
  for (int k0 = 0; k0 < C; k0 += 32) {     // uniform trip count: shuffles see full warps
    const int k = k0 + g;
    const bool ok = k < C;
    float acc = 0.f, bc = 0.f;
    int64_t id = 0;
    if constexpr (NQ > 0) {
      const int64_t id_raw = id_next;
      if (k + 32 < C) id_next = crow[k + 32];
      if (ok) {
        id = checked_token(id_raw, V, err);
        bc = to_f(bcrow[k]);
        const uint4* wr = reinterpret_cast<const uint4*>(w2c ? w2c + ((int64_t)row * C + k) * r
                                                             : w2 + id * r);
        uint4 u[NQ];
#pragma unroll
        for (int j = 0; j < NQ; ++j) u[j] = __ldg(wr + gl + 8 * j);
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          const T* e = reinterpret_cast<const T*>(&u[j]);
          const float* lq = s_lat + (gl + 8 * j) * E;
#pragma unroll
          for (int i = 0; i < E; ++i) acc = fmaf(to_f(e[i]), lq[i], acc);
        }
      }
    } else if (ok) {
      id = checked_token(crow[k], V, err);
      bc = to_f(bcrow[k]);
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
      const float sc = bc + acc;
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
  const int E = (int)(16 / xp_elem(h->dtype));
  // 16-byte loads need every row start 16-byte aligned
  const bool vec = (uintptr_t)base % 16 == 0 && sn % E == 0 && sb % E == 0;
  // fast path: room for the collected candidates, the boundary ids and an id bitmap
  const size_t smem_hist = (size_t)TS_HISTS * 256 * 4;
  const size_t smem_fast = smem_hist + (size_t)TS_CAP * 12 + (size_t)((h->V + 31) / 32) * 6;
  const bool fast = C <= TS_CAP / 2 && smem_fast <= 160 * 1024;
  const size_t smem = fast ? smem_fast : smem_hist;
  cudaError_t e = cudaSuccess;
#define XP_SELECT(T, VEC)                                                                   \
  do {                                                                                      \
    e = cudaFuncSetAttribute(topc_select_kernel<T, VEC>,                                    \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);       \
    if (e != cudaSuccess) return e;                                                         \
    topc_select_kernel<T, VEC><<<rows, TS_THREADS, smem, s>>>(                              \
        (const T*)base, sn, sb, Bm1, h->B, h->V, C, fast ? 1 : 0, cand, (T*)base_c, blk,    \
        anchor, h->err);                                                                    \
  } while (0)
  if (h->dtype == XP_BF16) {
    if (vec) XP_SELECT(bf16, true); else XP_SELECT(bf16, false);
  } else {
    if (vec) XP_SELECT(float, true); else XP_SELECT(float, false);
  }
#undef XP_SELECT
  e = cudaGetLastError();
  if (e != cudaSuccess || !w2c) return e;
  const int row_bytes = (int)(h->r * xp_elem(h->dtype));
  const int64_t total = (int64_t)rows * C;
  const int grid = (int)std::min<int64_t>((total + 7) / 8, (int64_t)h->num_sms * 16);
  const bool vec_rows = row_bytes % 16 == 0 && (uintptr_t)w2c % 16 == 0;
  if (vec_rows)
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
  // 16-byte loads per lane and candidate when r is a multiple of 8 lanes x 16 bytes
  const int E = (int)(16 / xp_elem(h->dtype));
  const int nq = h->r % (8 * E) == 0 ? h->r / (8 * E) : 0;
#define XP_TOPC_SCORE(T, NQ)                                                                    \
  topc_readout_kernel<T, NQ><<<rows, 256, smem, s>>>((const T*)lat, (const T*)base_c, cand,     \
                                                     (const T*)w2c, (const T*)h->w2, Bm1, h->B, \
                                                     h->V, C, h->r, blk, win, h->err)
  if (h->dtype == XP_BF16) {
    switch (nq) {
      case 1: XP_TOPC_SCORE(bf16, 1); break;
      case 2: XP_TOPC_SCORE(bf16, 2); break;
      case 4: XP_TOPC_SCORE(bf16, 4); break;
      default: XP_TOPC_SCORE(bf16, 0);
    }
  } else {
    switch (nq) {
      case 1: XP_TOPC_SCORE(float, 1); break;
      case 2: XP_TOPC_SCORE(float, 2); break;
      case 4: XP_TOPC_SCORE(float, 4); break;
      default: XP_TOPC_SCORE(float, 0);
    }
  }
#undef XP_TOPC_SCORE
  return cudaGetLastError();
}
