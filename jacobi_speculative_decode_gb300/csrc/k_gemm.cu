// Dense products of the hidden cache in unfolded form (once per draft step; qwen3_xpress
// page, hidden_cache and the hoisted xh = hcache @ in_proj[:, :2r]^T), for the heads
// and calls the folded tcgen05 path (k_hidden_tc.cu) does not take:
//   G   = h . [down_h ; down_g]^T        [N*B, 2r]   bf16 tensor cores (split-K partials)
//   hc  = [G_h ; mean over the block of G_g]            fp32  (mean commutes with down_g)
//   xh  = hc . in_proj[:, :2r]^T          [N*B, r]    fp32 SIMT (hc is never rounded)
#include <algorithm>

#include "xp_device.cuh"

using namespace xpd;
typedef __nv_bfloat16 bf16;

namespace {

// ---------------------------------------------------------------------------
// C[z][m, n] = sum_{k in split z} A[m, k] B[n, k]; bf16 operands, fp32 out.
// 128 x 128 tile, 8 warps (2 x 4, 64 x 32 each), k-steps of 32, 3-stage cp.async.
// ---------------------------------------------------------------------------
constexpr int GB_M = 128, GB_N = 128, GB_K = 32, GB_STAGES = 3, GB_PITCH = GB_K + 8;

__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__global__ void __launch_bounds__(256) gemm_bf16_kernel(const bf16* __restrict__ A, int lda,
                                                        const bf16* __restrict__ B, int ldb,
                                                        float* __restrict__ C, int ldc,
                                                        int64_t split_stride, int M, int N,
                                                        int ksplit) {
  extern __shared__ __align__(128) uint8_t gsm[];
  bf16 (*sA)[GB_M * GB_PITCH] = reinterpret_cast<bf16 (*)[GB_M * GB_PITCH]>(gsm);
  bf16 (*sB)[GB_N * GB_PITCH] =
      reinterpret_cast<bf16 (*)[GB_N * GB_PITCH]>(gsm + sizeof(bf16) * GB_STAGES * GB_M * GB_PITCH);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int m0 = blockIdx.y * GB_M, n0 = blockIdx.x * GB_N;
  const int kbeg = blockIdx.z * ksplit;
  const int nk = ksplit / GB_K;
  const int wm = (warp / 4) * 64, wn = (warp % 4) * 32;

  auto load = [&](int stage, int kt) {
    const int k0 = kbeg + kt * GB_K;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = tid + i * 256;        // 512 16-byte chunks per operand tile
      const int row = c / 4, kc = (c % 4) * 8;
      const int gm = m0 + row, gn = n0 + row;
      cp_async16_zfill(&sA[stage][row * GB_PITCH + kc],
                       A + (int64_t)(gm < M ? gm : 0) * lda + k0 + kc, gm < M);
      cp_async16_zfill(&sB[stage][row * GB_PITCH + kc],
                       B + (int64_t)(gn < N ? gn : 0) * ldb + k0 + kc, gn < N);
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

#pragma unroll
  for (int s = 0; s < GB_STAGES - 1; ++s) {
    if (s < nk) load(s, s);
    cp_async_commit();
  }
  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<GB_STAGES - 2>();
    __syncthreads();
    const int nxt = kt + GB_STAGES - 1;
    if (nxt < nk) load(nxt % GB_STAGES, nxt);
    cp_async_commit();
    const bf16* a = sA[kt % GB_STAGES];
    const bf16* b = sB[kt % GB_STAGES];
#pragma unroll
    for (int kk = 0; kk < GB_K; kk += 16) {
      uint32_t af[4][4], bfr[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        ldm_x4(af[i], a + (wm + i * 16 + (lane % 16)) * GB_PITCH + kk + (lane / 16) * 8);
#pragma unroll
      for (int j = 0; j < 2; ++j)
        ldm_x4(bfr[j], b + (wn + j * 16 + (lane % 8) + (lane / 16) * 8) * GB_PITCH + kk +
                           ((lane / 8) % 2) * 8);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma16816(acc[i][j], af[i], &bfr[j / 2][(j % 2) * 2]);
    }
  }
  cp_async_wait<0>();
  float* Cz = C + (int64_t)blockIdx.z * split_stride;
  const int g = lane / 4, t = lane % 4;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = m0 + wm + i * 16 + g + (e >= 2 ? 8 : 0);
        const int n = n0 + wn + j * 8 + 2 * t + (e & 1);
        if (m < M && n < N) Cz[(int64_t)m * ldc + n] = acc[i][j][e];
      }
}

// ---------------------------------------------------------------------------
// SIMT fp32 GEMM, C[z][m, n] = sum_k A[m, k] B[n, k] over split z, 32 x 32 tiles
// (fp32 heads, and the second hidden-cache product whose A operand stays fp32)
// ---------------------------------------------------------------------------
template <typename TA, typename TB>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const TA* __restrict__ A, int lda,
                                                        const TB* __restrict__ B, int ldb,
                                                        float* __restrict__ C, int ldc,
                                                        int64_t split_stride, int M, int N,
                                                        int ksplit, int K) {
  __shared__ float As[32][33];
  __shared__ float Bs[32][33];
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const int m0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  const int kbeg = blockIdx.z * ksplit, kend = std::min(K, kbeg + ksplit);
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  for (int k0 = kbeg; k0 < kend; k0 += 32) {
    for (int i = tid; i < 32 * 32; i += 256) {
      const int rr = i / 32, kk = i % 32, gk = k0 + kk;
      As[kk][rr] = (m0 + rr < M && gk < kend) ? to_f(A[(int64_t)(m0 + rr) * lda + gk]) : 0.f;
      Bs[kk][rr] = (n0 + rr < N && gk < kend) ? to_f(B[(int64_t)(n0 + rr) * ldb + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      const float a0 = As[kk][ty], a1 = As[kk][ty + 16];
      const float b0 = Bs[kk][tx], b1 = Bs[kk][tx + 16];
      acc[0][0] = fmaf(a0, b0, acc[0][0]);
      acc[0][1] = fmaf(a0, b1, acc[0][1]);
      acc[1][0] = fmaf(a1, b0, acc[1][0]);
      acc[1][1] = fmaf(a1, b1, acc[1][1]);
    }
    __syncthreads();
  }
  float* Cz = C + (int64_t)blockIdx.z * split_stride;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
      if (m < M && n < N) Cz[(int64_t)m * ldc + n] = acc[i][j];
    }
}

// hc[n*B+b, c] = sum_z G[z][n*B+b, c]                         (c < r)
// hc[n*B+b, r+c] = (1/B) sum_b' sum_z G[z][n*B+b', r+c]       (mean over the block)
__global__ void hc_reduce_kernel(const float* __restrict__ G, int64_t split_stride, int splits,
                                 float* __restrict__ hc, int N, int B, int r) {
  const int64_t total = (int64_t)N * 2 * r;       // one thread per (block, column)
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % (2 * r));
    const int n = (int)(i / (2 * r));
    if (c < r) {
      for (int b = 0; b < B; ++b) {
        const int64_t o = ((int64_t)n * B + b) * 2 * r + c;
        float s = 0.f;
        for (int z = 0; z < splits; ++z) s += G[z * split_stride + o];
        hc[o] = s;
      }
    } else {
      float s = 0.f;
      for (int b = 0; b < B; ++b) {
        const int64_t o = ((int64_t)n * B + b) * 2 * r + c;
        for (int z = 0; z < splits; ++z) s += G[z * split_stride + o];
      }
      const float mean = s / (float)B;
      for (int b = 0; b < B; ++b) hc[((int64_t)n * B + b) * 2 * r + c] = mean;
    }
  }
}

}  // namespace

cudaError_t xp_launch_embed_table(const xp_head* h, cudaStream_t s) {
  const int smem = (int)(sizeof(bf16) * GB_STAGES * (GB_M + GB_N) * GB_PITCH);
  cudaError_t e =
      cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((h->r + GB_N - 1) / GB_N, (h->V + GB_M - 1) / GB_M, 1);
  gemm_bf16_kernel<<<grid, 256, smem, s>>>((const bf16*)h->w1, h->r, (const bf16*)h->w_lat, h->r,
                                           h->E, h->r, 0, h->V, h->r, h->r);
  return cudaGetLastError();
}

int xp_hidden_splits(int rows, int r, int hidden, int num_sms, int cap_rows) {
  const int tiles = ((rows + GB_M - 1) / GB_M) * ((2 * r + GB_N - 1) / GB_N);
  int splits = std::max(1, (2 * num_sms + tiles - 1) / tiles);
  splits = std::min(splits, std::max(1, cap_rows / std::max(rows, 1)));
  while (splits > 1 && (hidden % (splits * GB_K) != 0)) --splits;
  return std::min(splits, 16);
}

cudaError_t xp_launch_hidden(const xp_head* h, const void* h_full, int N, float* xh, float* part,
                             float* hc, int part_rows, cudaStream_t s) {
  if (xp_hidden_tc_call_ok(h, h_full)) {
    const cudaError_t e = xp_launch_hidden_tc(h, h_full, N, xh, part, part_rows, s);
    if (e != cudaErrorNotSupported) return e;
  }
  const int B = h->B, r = h->r, hid = h->hidden, rows = N * B;
  const int64_t stride = (int64_t)rows * 2 * r;
  int splits = 1;
  if (h->dtype == XP_BF16 && hid % GB_K == 0 && (uintptr_t)h_full % 16 == 0) {
    splits = xp_hidden_splits(rows, r, hid, h->num_sms, part_rows);
    dim3 grid((2 * r + GB_N - 1) / GB_N, (rows + GB_M - 1) / GB_M, splits);
    const int smem = (int)(sizeof(bf16) * GB_STAGES * (GB_M + GB_N) * GB_PITCH);
    cudaError_t e =
        cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gemm_bf16_kernel<<<grid, 256, smem, s>>>((const bf16*)h_full, hid, (const bf16*)h->down_hg, hid,
                                          part, 2 * r, stride, rows, 2 * r, hid / splits);
  } else if (h->dtype == XP_BF16) {
    dim3 grid((2 * r + 31) / 32, (rows + 31) / 32, 1);
    gemm_simt_kernel<bf16, bf16><<<grid, 256, 0, s>>>((const bf16*)h_full, hid,
                                                      (const bf16*)h->down_hg, hid, part, 2 * r,
                                                      stride, rows, 2 * r, hid, hid);
  } else {
    dim3 grid((2 * r + 31) / 32, (rows + 31) / 32, 1);
    gemm_simt_kernel<float, float><<<grid, 256, 0, s>>>((const float*)h_full, hid,
                                                        (const float*)h->down_hg, hid, part,
                                                        2 * r, stride, rows, 2 * r, hid, hid);
  }
  const int64_t red = (int64_t)N * 2 * r;
  hc_reduce_kernel<<<(unsigned)std::min<int64_t>((red + 255) / 256, 4096), 256, 0, s>>>(
      part, stride, splits, hc, N, B, r);
  dim3 g2((r + 31) / 32, (rows + 31) / 32, 1);
  if (h->dtype == XP_BF16)
    gemm_simt_kernel<float, bf16><<<g2, 256, 0, s>>>(hc, 2 * r, (const bf16*)h->w_hc, 2 * r, xh,
                                                     r, 0, rows, r, 2 * r, 2 * r);
  else
    gemm_simt_kernel<float, float><<<g2, 256, 0, s>>>(hc, 2 * r, (const float*)h->w_hc, 2 * r,
                                                      xh, r, 0, rows, r, 2 * r, 2 * r);
  return cudaGetLastError();
}
