// Hidden cache on tcgen05 (sm_103a): qwen3_xpress model page, hidden_cache and the
// pass-invariant half of in_proj hoisted out of the refinement loop.
//
// The two linear maps in a row are folded into one, once per head:
//   F_h = in_proj[:, :r]   . down_h     [r, hidden]
//   F_g = in_proj[:, r:2r] . down_g     [r, hidden]
// so that  xh[n,b] = F_h h[n,b] + (1/B) sum_b' F_g h[n,b']   (the block mean commutes
// with F_g).  F = [F_h ; F_g] is kept as two bf16 planes, hi = bf16(F) and
// lo = bf16(F - hi), so hi + lo carries F to about 2^-17 relative.  One tcgen05 GEMM
// accumulates h . hi^T and h . lo^T into the same TMEM accumulator:
//   P[z] = h[:, K-split z] . (hi + lo)[:, K-split z]^T     [N*B, 2r] fp32 partials
//   xh[n*B+b, c] = sum_z P[z][n*B+b, c] + (1/B) sum_b' sum_z P[z][n*B+b', r+c]
// The product keeps fp32 grade although both operands are bf16, and the second
// GEMM of the unfolded form (fp32 hc times in_proj) disappears.
//
// GEMM CTA (192 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer,
// warps 2..5 epilogue (warp w reads TMEM lanes 32*(w%4)..+31).  Tile 128 rows x
// 128 output columns, k-chunks of 64 (128-byte swizzled), 4-stage ring of
// {h chunk 16 KB, hi chunk 16 KB, lo chunk 16 KB}; the K range is split over
// about one CTA per SM.
#include <algorithm>

#include "sm100_ptx.cuh"
#include "xp_device.cuh"

typedef __nv_bfloat16 bf16;

namespace {

constexpr int HM = 128;                 // rows per tile (TMEM lanes)
constexpr int HN = 128;                 // output columns per tile (MMA N)
constexpr int HK = 64;                  // k per swizzled chunk
constexpr int STAGES = 4;
constexpr int A_BYTES = HM * HK * 2;    // 16 KB
constexpr int B_BYTES = HN * HK * 2;    // 16 KB
constexpr int STAGE_BYTES = A_BYTES + 2 * B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = HN;
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(HM, HN);
constexpr int MAX_SPLITS = 64;

struct Bars {
  uint64_t full[STAGES], empty[STAGES];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
};

// fold[p][c][k] for p = 0 (hi), 1 (lo):  F[c][k] = sum_j in_proj[c % r][(c / r) * r + j] *
// down_hg[(c / r) * r + j][k].  Products of two bf16 values are exact in fp32; the sum
// over j (r terms) is the only rounding before the split.  4 output rows per thread.
__global__ void hidden_fold_kernel(const bf16* __restrict__ in_proj, const bf16* __restrict__ down_hg,
                                   bf16* __restrict__ fold, int r, int hidden) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  const int c0 = blockIdx.y * 4;                 // 4 consecutive rows, all in one half (r % 4 == 0)
  if (k >= hidden) return;
  const int part = c0 / r;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < r; ++j) {
    const float d = __bfloat162float(down_hg[(int64_t)(part * r + j) * hidden + k]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = c0 + i;
      const float w = __bfloat162float(in_proj[(int64_t)(c % r) * 3 * r + part * r + j]);
      acc[i] = fmaf(w, d, acc[i]);
    }
  }
  const int64_t plane = (int64_t)2 * r * hidden;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bf16 hi = __float2bfloat16_rn(acc[i]);
    const bf16 lo = __float2bfloat16_rn(acc[i] - __bfloat162float(hi));
    fold[(int64_t)(c0 + i) * hidden + k] = hi;
    fold[plane + (int64_t)(c0 + i) * hidden + k] = lo;
  }
}

__global__ void __launch_bounds__(THREADS, 1) hidden_tc_kernel(
    const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_f, int rows,
    int two_r, int nkb, int splits, float* __restrict__ part, int64_t split_stride, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + STAGES * STAGE_BYTES);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n0 = blockIdx.x * HN, m0 = blockIdx.y * HM, z = blockIdx.z;
  const int kb0 = (int)((int64_t)z * nkb / splits), kb1 = (int)((int64_t)(z + 1) * nkb / splits);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->done), 1);
    bars->abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  ptx::pdl_trigger();           // a launch that depends on nothing here may start now

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_h);
      ptx::prefetch_tmap(&tm_f);
      const uint64_t pol_h = ptx::policy_evict_first();
      const uint64_t pol_f = ptx::policy_evict_last();
      uint32_t issued[STAGES] = {};
      bool ok = true;
      for (int kb = kb0, i = 0; kb < kb1 && ok; ++kb, ++i) {
        const int s = i % STAGES;
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->empty[s]), ((i / STAGES) & 1) ^ 1, abort, err);
        if (!ok) break;
        const uint32_t full = ptx::smem_u32(&bars->full[s]);
        const uint32_t st = ptx::smem_u32(smem + s * STAGE_BYTES);
        ptx::mbar_arrive_expect_tx(full, STAGE_BYTES);
        ptx::tma_load_2d(st, &tm_h, full, kb * HK, m0, pol_h);
        ptx::tma_load_2d(st + A_BYTES, &tm_f, full, kb * HK, n0, pol_f);
        ptx::tma_load_2d(st + A_BYTES + B_BYTES, &tm_f, full, kb * HK, two_r + n0, pol_f);
        ++issued[s];
      }
      // nothing may land in smem after the CTA is gone
      volatile int no_abort = 0;
      for (int s = 0; s < STAGES; ++s)
        if (issued[s])
          ptx::mbar_wait(ptx::smem_u32(&bars->full[s]), (issued[s] - 1) & 1, &no_abort, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int kb = kb0, i = 0; kb < kb1 && ok; ++kb, ++i) {
        const int s = i % STAGES;
        ok = ptx::mbar_wait(ptx::smem_u32(&bars->full[s]), (i / STAGES) & 1, abort, err);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t a0 = ptx::smem_u32(smem + s * STAGE_BYTES);
        const uint32_t bh = a0 + A_BYTES, bl = a0 + A_BYTES + B_BYTES;
#pragma unroll
        for (int kk = 0; kk < HK / 16; ++kk)
          ptx::mma_bf16(tmem, ptx::sw128_desc(a0 + kk * 32), ptx::sw128_desc(bh + kk * 32), IDESC,
                        (i | kk) != 0);
#pragma unroll
        for (int kk = 0; kk < HK / 16; ++kk)
          ptx::mma_bf16(tmem, ptx::sw128_desc(a0 + kk * 32), ptx::sw128_desc(bl + kk * 32), IDESC,
                        1u);
        ptx::mma_commit(ptx::smem_u32(&bars->empty[s]));
      }
      // arrives once every MMA issued above has completed (also after an abort)
      ptx::mma_commit(ptx::smem_u32(&bars->done));
    }
  } else {
    // epilogue: TMEM lane group g = rows m0 + 32g .. +31; transpose each 32 x 32 block
    // through a private smem tile so that every global store is one 128-byte row
    const int g = warp & 3;
    const bool ok =
        __all_sync(0xFFFFFFFFu, ptx::mbar_wait(ptx::smem_u32(&bars->done), 0, abort, err));
    if (ok && !*abort) {
      ptx::tc_fence_after();
      // the ring is idle now (every loaded chunk was consumed by a completed MMA)
      float* T = reinterpret_cast<float*>(smem) + (warp - 2) * 32 * 33;
      const uint32_t trow = tmem + ((uint32_t)(g * 32) << 16);
      float* Pz = part + (int64_t)z * split_stride;
      for (int ch = 0; ch < HN / 32; ++ch) {
        uint32_t v[32];
        ptx::tmem_ld32(trow + (uint32_t)(ch * 32), v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) T[lane * 33 + j] = __uint_as_float(v[j]);
        __syncwarp();
        const int col = n0 + ch * 32 + lane;
#pragma unroll 4
        for (int i = 0; i < 32; ++i) {
          const int row = m0 + g * 32 + i;
          if (row < rows) Pz[(int64_t)row * two_r + col] = T[i * 33 + lane];
        }
        __syncwarp();
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// xh[n*B+b, c] = sum_z P[z][n*B+b, c] + (1/B) sum_b' sum_z P[z][n*B+b', r+c].
// Block (32 channels, 8 slot lanes) per (channel slice, block n); fixed summation order.
__global__ void __launch_bounds__(256) xh_reduce_kernel(const float* __restrict__ P,
                                                        int64_t split_stride, int splits,
                                                        float* __restrict__ xh, int B, int r) {
  __shared__ float red[8][32];
  const int tx = threadIdx.x, ty = threadIdx.y;
  ptx::pdl_wait();              // the partials come from an earlier kernel
  const int c = blockIdx.x * 32 + tx, n = blockIdx.y;
  const int two_r = 2 * r;
  float gsum = 0.f;
  if (c < r)
    for (int b = ty; b < B; b += 8) {
      const float* p = P + ((int64_t)n * B + b) * two_r + r + c;
#pragma unroll 8
      for (int zz = 0; zz < splits; ++zz) gsum += __ldg(p + zz * split_stride);
    }
  red[ty][tx] = gsum;
  __syncthreads();
  float total = 0.f;
#pragma unroll
  for (int t = 0; t < 8; ++t) total += red[t][tx];
  const float mean = total / (float)B;
  if (c < r)
    for (int b = ty; b < B; b += 8) {
      const int64_t row = (int64_t)n * B + b;
      const float* p = P + row * two_r + c;
      float s = 0.f;
#pragma unroll 8
      for (int zz = 0; zz < splits; ++zz) s += __ldg(p + zz * split_stride);
      xh[row * r + c] = s + mean;
    }
}

bool encode_bf16_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                    uint32_t box_inner, uint32_t box_outer) {
  xp_encode_tiled_fn fn = xp_get_encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kSmem = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(Bars);

}  // namespace

bool xp_hidden_tc_ok(int r, int hidden, xp_dtype dt) {
  return dt == XP_BF16 && (2 * r) % HN == 0 && hidden % 8 == 0;
}

bool xp_hidden_tc_map(xp_head* h) {
  // rows [0, 2r) the hi plane, [2r, 4r) the lo plane
  return encode_bf16_2d(&h->tm_hfold, h->hfold, (uint64_t)h->hidden, (uint64_t)4 * h->r, HK, HN);
}

cudaError_t xp_launch_hidden_fold(const xp_head* h, const void* in_proj, cudaStream_t s) {
  dim3 grid((h->hidden + 255) / 256, (2 * h->r) / 4);
  hidden_fold_kernel<<<grid, 256, 0, s>>>((const bf16*)in_proj, (const bf16*)h->down_hg,
                                          (bf16*)h->hfold, h->r, h->hidden);
  return cudaGetLastError();
}

bool xp_hidden_tc_call_ok(const xp_head* h, const void* h_full) {
  return h->hidden_tc && (uintptr_t)h_full % 16 == 0;
}

cudaError_t xp_launch_hidden_tc_gemm(const xp_head* h, const void* h_full, int N, float* part,
                                     int part_rows, cudaStream_t s, int* splits_out) {
  const int rows = N * h->B, two_r = 2 * h->r;
  CUtensorMap tm_h;
  if (!encode_bf16_2d(&tm_h, h_full, (uint64_t)h->hidden, (uint64_t)rows, HK, HM))
    return cudaErrorNotSupported;
  const int nkb = (h->hidden + HK - 1) / HK;
  const int m_tiles = (rows + HM - 1) / HM, n_tiles = two_r / HN;
  int splits = std::max(1, h->num_sms / (m_tiles * n_tiles));
  splits = std::min({splits, nkb, MAX_SPLITS, std::max(1, part_rows / rows)});
  cudaError_t e =
      cudaFuncSetAttribute(hidden_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  const int64_t stride = (int64_t)rows * two_r;
  hidden_tc_kernel<<<dim3(n_tiles, m_tiles, splits), THREADS, kSmem, s>>>(
      tm_h, h->tm_hfold, rows, two_r, nkb, splits, part, stride, h->err);
  *splits_out = splits;
  return cudaGetLastError();
}

cudaError_t xp_launch_xh_reduce(const xp_head* h, int N, float* xh, const float* part, int splits,
                                cudaStream_t s, bool pdl) {
  const int64_t stride = (int64_t)N * h->B * 2 * h->r;
  const dim3 grid((h->r + 31) / 32, N), block(32, 8);
  if (pdl) return xp_launch_pdl(xh_reduce_kernel, grid, block, 0, s, part, stride, splits, xh, h->B, h->r);
  xh_reduce_kernel<<<grid, block, 0, s>>>(part, stride, splits, xh, h->B, h->r);
  return cudaGetLastError();
}

cudaError_t xp_launch_hidden_tc(const xp_head* h, const void* h_full, int N, float* xh,
                                float* part, int part_rows, cudaStream_t s) {
  int splits = 0;
  const cudaError_t e = xp_launch_hidden_tc_gemm(h, h_full, N, part, part_rows, s, &splits);
  if (e != cudaSuccess) return e;
  return xp_launch_xh_reduce(h, N, xh, part, splits, s, false);
}
