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
//   1. x = xh + E[prev] for the own channels (every thread loads the token it needs)
//   2. u = per-channel causal mix of x (fp32; item = slot b x channel pair), kept in
//      fp32 for the residual and sent to the 7 peers as fp16 with one bulk copy each;
//      the own slice stays in a buffer of its own, which nothing overwrites before
//      the copies out of it are known to have landed
//   3. [gate ; up] = [w_gate ; w_up][own units] u^T, tcgen05.mma kind::f16 on fp16
//      operands (the head keeps fp16 copies of w_gate and w_up), the weights as the
//      M = 128 side and the group's rows as N = MT; the weight rows are interleaved
//      so that one TMEM lane quadrant holds gate and up of the same 16 units;
//      a = silu(gate) * up as bf16 hi + lo
//   4. partial = w_down[:, own units] a^T for ALL r channels (two M = 128 tiles, the
//      activations' hi rows and lo rows side by side as N = 2*MT, summed when read
//      back; w_down's slice stays resident), staged by the warp whose lanes hold
//      owner p's channels as [channel][row pair] fp16 and sent by that warp to owner
//      p with one bulk copy
//   5. lat = u + the 8 partials of the own channels, added in a fixed order (fp32)
// The fp16 exchanges halve the bytes that cross the cluster network, whose
// bandwidth per SM sets their latency; fp16's 2^-11 relative error is a quarter of
// the bf16 rounding of the stored latent.  Values beyond the fp16 range saturate
// and raise XP_ERR_RANGE.
// The only cluster-wide barrier per group is a split arrive/wait that keeps a
// CTA from sending into buffers a peer is still reading; the first one (barriers
// initialised) is waited on just before the first send, and after its last group a
// CTA arrives as soon as everything addressed to it has landed.
//
// Shared-memory operand layouts (what the TMA writes and tcgen05 reads):
//   128B swizzle: element (row, k) of an R-row matrix, 64-column chunks, at
//     (k/64)*R*128 + row*128 + ((((k%64)/8) ^ (row%8))*16) + (k%8)*2
//   64B swizzle (the exchanged u, fp16): sender p's slice holds columns [32p, 32p+32)
//     of MT rows: (row, c) at row*64 + (((c/8) ^ ((row/2)%4))*16) + (c%8)*2
#include <cooperative_groups.h>
#include <cuda_fp16.h>

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
constexpr int CS = 32;         // own channels (r = 256) == warp size
constexpr int R = CL * CS;     // latent rank handled by this kernel

// bytes of one staged partial block: [CS channels][MT/2 + 1 row pairs] of fp16x2 (odd pitch)
__host__ __device__ constexpr int blk_bytes(int MT) { return ((CS * (MT / 2 + 1) * 4 + 15) / 16) * 16; }

struct Plan {                  // byte offsets into dynamic shared memory
  int MT;
  int wgu, wd, mix, ubuf, uout, act, rcv, sx, us, rowi, bars;
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
  p.wgu = take((R / 64) * 128 * 128, 1024);     // own w_gate / w_up rows (interleaved), 128B swizzle
  p.wd = take(R * HS * 2, 1024);                // w_down[:, own units], R rows x 64, 128B swizzle
  p.mix = take(mparts * mbox * CS * 2, 1024);
  // u (fp16) of the 8 senders (64B swizzle), later the 7 outgoing partial blocks
  p.ubuf = take(std::max(CL * MT * 64, (CL - 1) * blk_bytes(MT)), 1024);
  p.uout = take(MT * 64, 1024);                 // own u: the MMA's and the peers' copy
  p.act = take(2 * MT * 128, 1024);             // activations hi rows then lo rows, 64 units, 128B swizzle
  p.rcv = take(CL * blk_bytes(MT), 16);         // partial blocks by sender (own one at slot q)
  p.sx = take(MT * CS * 4, 16);                 // x = xh + E[prev], own channels
  p.us = take(MT * CS * 4, 16);                 // u fp32, own channels (the residual)
  p.rowi = take(MT * 4, 16);                    // lat row of each group row, -1 = not stored
  p.bars = take(64, 16);                        // 5 mbarriers + the TMEM address
  p.total = o;
  return p;
}

__device__ __forceinline__ int swz128(int row, int k, int Rr) {
  return ((k >> 6) * Rr + row) * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + ((k & 7) << 1);
}
__device__ __forceinline__ int swz64(int row, int c) {      // within one 32-column chunk
  return row * 64 + ((((c >> 3) ^ ((row >> 1) & 3))) << 4) + ((c & 7) << 1);
}

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
// arrive without ordering this thread's earlier memory operations: used where what
// the peers need was already published (mbarrier inits by fence.mbarrier_init, or
// every byte addressed to this CTA observed through its mbarriers before exit)
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// fp16 pair with saturation at the largest finite value; flags a clipped input
__device__ __forceinline__ __half2 to_half2_sat(float2 v, bool& clipped) {
  constexpr float kMax = 65504.0f;
  clipped |= fabsf(v.x) > kMax || fabsf(v.y) > kMax;
  return __floats2half2_rn(fminf(fmaxf(v.x, -kMax), kMax), fminf(fmaxf(v.y, -kMax), kMax));
}

__device__ __forceinline__ void split_bf16(float v, bf16& hi, bf16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// n consecutive TMEM columns (n = 16, 24, 32 or 48) of this warp's 32 lanes
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t ta, float (&out)[NC]) {
  static_assert(NC == 16 || NC == 24 || NC == 32 || NC == 48, "column count");
  if constexpr (NC >= 32) {
    uint32_t a[32];
    ptx::tmem_ld32(ta, a);
    if constexpr (NC == 48) {
      uint32_t b[16];
      ptx::tmem_ld16(ta + 32, b);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) out[32 + i] = __uint_as_float(b[i]);
    } else {
      ptx::tmem_wait_ld();
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) out[i] = __uint_as_float(a[i]);
  } else {
    uint32_t a[16];
    ptx::tmem_ld16(ta, a);
    if constexpr (NC == 24) {
      uint32_t b[8];
      ptx::tmem_ld8(ta + 16, b);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 8; ++i) out[16 + i] = __uint_as_float(b[i]);
    } else {
      ptx::tmem_wait_ld();
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = __uint_as_float(a[i]);
  }
}

struct Maps {
  CUtensorMap wgu, wdk, mix;
};

// u[bl*B + b][c] = sum_{j <= b} mix[b][j][c] x[bl*B + j][c] for blocks bl0 .. bl0+nbv-1
// (nbv <= NB), one item = (slot b, channel pair); the mixer value is loaded once and
// used for every block.  Writes u (fp32) and its fp16 copy for the exchange.  With
// PARTIAL, blocks k >= nbv are neither read nor written (nbv < NB); without it nbv == NB.
template <int NB, bool PARTIAL = false>
__device__ __forceinline__ void mix_slots(const bf16* __restrict__ sMix, const float* sX, float* sUs,
                                          uint8_t* uh, int B, int nbv, int tid, bool& out_of_range,
                                          int bl0 = 0) {
  for (int it = tid; it < B * (CS / 2); it += THREADS) {
    const int b = it / (CS / 2), c = (it % (CS / 2)) * 2;
    const bf16* mrow = sMix + (b * B) * CS + c;
    const float* xr = sX + (bl0 * B) * CS + c;
    float2 acc[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) acc[k] = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int j = 0; j <= b; ++j) {
      const float2 mv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(mrow + j * CS));
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        if (PARTIAL && k >= nbv) break;
        const float2 xv = *reinterpret_cast<const float2*>(xr + (k * B + j) * CS);
        acc[k].x = fmaf(mv.x, xv.x, acc[k].x);
        acc[k].y = fmaf(mv.y, xv.y, acc[k].y);
      }
    }
#pragma unroll
    for (int k = 0; k < NB; ++k)
      if (k < nbv) {
        const int m = (bl0 + k) * B + b;
        *reinterpret_cast<float2*>(sUs + m * CS + c) = acc[k];
        *reinterpret_cast<__half2*>(uh + swz64(m, c)) = to_half2_sat(acc[k], out_of_range);
      }
  }
}

// [gate ; up] (hi columns then lo columns) at 0, the two partial tiles at 128 and 256
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_GU = 0, COL_P = 128;

template <int MTILES>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS, 1) latent_mma_kernel(
    const __grid_constant__ Maps maps, const int64_t* __restrict__ blk,
    const int64_t* __restrict__ am1, const float* __restrict__ xh, const float* __restrict__ E,
    bf16* __restrict__ lat, int N, int B, int V, uint32_t* err) {
  constexpr int MT = MTILES * 16;
  constexpr int HALF = MT / 2;             // TMEM columns per reader warp in the SwiGLU step
  constexpr int LDH = MT / 2 + 1;          // row pitch of a staged partial block (fp16x2 words)
  constexpr int BLK = blk_bytes(MT);
  constexpr uint32_t SLICE = MT * 64;      // bytes of one sender's u
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (ptx::smem_u32(sm_raw) & 1023u)) & 1023u);
  const int q = (int)cg::this_cluster().block_rank();
  const int cid = blockIdx.x / CL, nclusters = gridDim.x / CL;
  const Plan P = make_plan(MT, B);
  const uint32_t s0 = ptx::smem_u32(sm);
  const uint32_t aW = s0 + P.wgu, aU = s0 + P.ubuf;
  const uint32_t aAct = s0 + P.act;
  const bf16* sMix = (const bf16*)(sm + P.mix);
  float* sX = (float*)(sm + P.sx);
  float* sUs = (float*)(sm + P.us);
  int* sRow = (int*)(sm + P.rowi);
  const uint32_t* sRcv = (const uint32_t*)(sm + P.rcv);
  // bar_mix: the mixer slice; bar_w: the weight slices (needed first by the MMAs)
  const uint32_t bar_w = s0 + P.bars, bar_u = bar_w + 8, bar_p = bar_w + 16;
  const uint32_t bar_mma = bar_w + 24, bar_mix = bar_w + 32;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + P.bars + 40);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int nb = MT / B;                   // blocks per group
  const int groups = (N + nb - 1) / nb;
  const uint32_t p_bytes_in = (uint32_t)((CL - 1) * BLK);
  const uint64_t pol = ptx::policy_evict_last();

  // ---- set-up: barriers, the resident weight and mixer slices by TMA (warp 0), TMEM
  // (warp 1); the cluster barrier that lets peers send here is waited on only just
  // before this CTA's first send, so its latency hides behind the first gather ----
  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_init(bar_w, 1);
      ptx::mbar_init(bar_p, 1);
      ptx::mbar_init(bar_mma, 1);
      ptx::mbar_init(bar_u, 1);
      ptx::mbar_init(bar_mix, 1);
      ptx::fence_barrier_init();
      const int mparts = (P.mix_rows + 255) / 256, mbox = std::min(P.mix_rows, 256);
      ptx::mbar_arrive_expect_tx(bar_mix, mparts * mbox * CS * 2);
      for (int pt = 0; pt < mparts; ++pt)
        ptx::tma_load_2d(s0 + P.mix + pt * mbox * CS * 2, &maps.mix, bar_mix, q * CS, pt * mbox,
                         pol);
      ptx::mbar_arrive_expect_tx(bar_w, 2 * HS * R * 2 + R * HS * 2);
      // the first group's incoming u and partial blocks
      ptx::mbar_arrive_expect_tx(bar_u, (CL - 1) * SLICE);
      ptx::mbar_arrive_expect_tx(bar_p, p_bytes_in);
    }
    __syncwarp();
    // the head keeps [w_gate ; w_up] in this CTA's row order (see xp_launch_gu_to_f16):
    // one 128-row box per 64-wide k chunk; w_down's column slice in one box
    if (lane < R / 64)
      ptx::tma_load_2d(aW + lane * 16384, &maps.wgu, bar_w, lane * 64, q * 128, pol);
    else if (lane == R / 64)
      ptx::tma_load_2d(s0 + P.wd, &maps.wdk, bar_w, q * HS, 0, pol);
  } else if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(s_tmem), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  // this CTA's barriers exist (fence.mbarrier_init above published them to the cluster,
  // so the arrive needs no release of its own)
  cluster_arrive_relaxed();
  ptx::pdl_wait();                         // blk (and xh) come from earlier kernels
  ptx::pdl_trigger();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  uint32_t mma_phase = 0;
  const int quad = warp & 3, half = warp >> 2;

  int it = 0;
  for (int grp = cid; grp < groups; grp += nclusters, ++it) {
    const uint32_t ph = it & 1;
    const bool last = grp + nclusters >= groups;
    const int n0 = grp * nb;
    const int rows = std::min(nb, N - n0) * B;   // valid rows of this group

    // ---- 1. x = xh + E[prev] for the own channels: row m, 4 channels per item ----
    for (int m = tid; m < MT; m += THREADS)
      sRow[m] = (m < rows && m % B != 0) ? (n0 + m / B) * (B - 1) + m % B - 1 : -1;
    for (int i0 = tid; i0 < MT * (CS / 4); i0 += 2 * THREADS) {
      float4 e[2], xv[2];
      int mm[2];
      int64_t tok[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {       // token ids and xh first, both in flight together
        const int i = i0 + k * THREADS;
        const int m = i / (CS / 4), c4 = (i % (CS / 4)) * 4;
        mm[k] = i < MT * (CS / 4) ? m : -1;
        e[k] = xv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        tok[k] = 0;
        if (mm[k] >= 0 && m < rows) {
          const int n = n0 + m / B, b = m % B;
          tok[k] = b == 0 ? am1[n] : blk[(int64_t)n * B + b - 1];
          xv[k] = __ldg(reinterpret_cast<const float4*>(xh + (int64_t)(n0 * B + m) * R + q * CS + c4));
        }
      }
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (mm[k] >= 0 && mm[k] < rows) {
          const int c4 = ((i0 + k * THREADS) % (CS / 4)) * 4;
          const int64_t t = checked_token(tok[k], V, err);
          e[k] = __ldg(reinterpret_cast<const float4*>(E + t * R + q * CS + c4));
        }
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (mm[k] >= 0) {
          const int i = i0 + k * THREADS;
          *reinterpret_cast<float4*>(sX + mm[k] * CS + (i % (CS / 4)) * 4) =
              make_float4(e[k].x + xv[k].x, e[k].y + xv[k].y, e[k].z + xv[k].z, e[k].w + xv[k].w);
        }
    }
    __syncthreads();
    // the previous group's peers are done reading this CTA's buffers, and it theirs
    if (it > 0) cluster_wait();

    // ---- 2. u = per-channel causal mix (fp32): item = (slot b, channel pair) ----
    if (it == 0) {
      volatile int no_abort = 0;
      ptx::mbar_wait(bar_mix, 0, &no_abort, err);
    }
    {
      uint8_t* uh = sm + P.uout;                     // own u (fp16)
      bool out_of_range = false;
      switch (nb) {
        case 1: mix_slots<1>(sMix, sX, sUs, uh, B, 1, tid, out_of_range); break;
        case 2: mix_slots<2>(sMix, sX, sUs, uh, B, 2, tid, out_of_range); break;
        case 3: mix_slots<3>(sMix, sX, sUs, uh, B, 3, tid, out_of_range); break;
        case 4: mix_slots<4>(sMix, sX, sUs, uh, B, 4, tid, out_of_range); break;
        case 6: mix_slots<6>(sMix, sX, sUs, uh, B, 6, tid, out_of_range); break;
        default:
          for (int bl0 = 0; bl0 < nb; bl0 += 4)
            mix_slots<4, true>(sMix, sX, sUs, uh, B, std::min(4, nb - bl0), tid, out_of_range,
                               bl0);
      }
      if (out_of_range) atomicOr(err, XP_ERR_RANGE);
      // rows past the last whole block of the group read as zero
      for (int m = nb * B + warp; m < MT; m += THREADS / 32) {
        sUs[m * CS + lane] = 0.f;
        *reinterpret_cast<__half*>(uh + swz64(m, lane)) = __float2half_rn(0.f);
      }
    }
    fence_async_smem();                    // the bulk copies and the MMA read u
    __syncthreads();
    if (it == 0) cluster_wait();           // the set-up arrive: every peer's barriers exist
    if (tid == 0) {
      for (int dp = 1; dp < CL; ++dp) {
        const int p = (q + dp) % CL;
        ptx::bulk_copy_to_peer(mapa(aU + q * SLICE, p), s0 + P.uout, SLICE, mapa(bar_u, p));
      }
    }
    mbar_wait_cluster(bar_u, ph, err);

    // ---- 3. [gate ; up] (units x rows) ----
    if (tid == 0) {
      if (it == 0) {
        volatile int no_abort = 0;
        ptx::mbar_wait(bar_w, 0, &no_abort, err);
      }
      ptx::tc_fence_after();
      constexpr uint32_t ID = ptx::idesc_f16_f32(128, MT);
      const uint64_t dw = ptx::sw128_desc(aW), du = ptx::sw64_desc(aU);
      const uint64_t dq = ptx::sw64_desc(s0 + P.uout);
#pragma unroll
      for (int s = 0; s < R / 16; ++s) {
        const int p = s / 2;               // sender of channels [32p, 32p + 32)
        const uint64_t bd = (p == q ? dq : du + ((p * SLICE) >> 4)) + (s % 2) * 2;
        ptx::mma_bf16(tmem + COL_GU, dw + (((s / 4) * 16384 + (s % 4) * 32) >> 4), bd, ID, s != 0);
      }
      ptx::mma_commit(bar_mma);
    }
    {
      volatile int no_abort = 0;
      ptx::mbar_wait(bar_mma, mma_phase, &no_abort, err);
    }
    mma_phase ^= 1;
    ptx::tc_fence_after();
    {
      // warp (quad g, half h): TMEM lanes 32g.. hold gate (lanes 0-15) and up (16-31) of
      // units 16g..16g+15, for the rows (columns) [h*HALF, (h+1)*HALF); the two lane
      // halves swap values so that each computes HALF/2 rows of all 16 units
      float v[HALF];
      tmem_ld_cols<HALF>(tmem + ((uint32_t)(quad * 32) << 16) + COL_GU + half * HALF, v);
      const bool lo_lane = lane < 16;
      const int unit = quad * 16 + (lane & 15);
#pragma unroll
      for (int i = 0; i < HALF / 2; ++i) {
        const float other = __shfl_xor_sync(0xFFFFFFFFu, lo_lane ? v[i + HALF / 2] : v[i], 16);
        const float gate = lo_lane ? v[i] : other;
        const float up = lo_lane ? other : v[i + HALF / 2];
        const int m = half * HALF + (lo_lane ? i : HALF / 2 + i);
        const float a = silu_fast(gate) * up;
        bf16 hi, lo;
        split_bf16(a, hi, lo);
        const int off = swz128(m, unit, MT);
        *reinterpret_cast<bf16*>(sm + P.act + off) = hi;
        *reinterpret_cast<bf16*>(sm + P.act + MT * 128 + off) = lo;
      }
    }
    ptx::tc_fence_before();
    fence_async_smem();                    // activations seen by the next MMA
    __syncthreads();

    // ---- 4. partial down projection over own units, channels x rows (two M tiles) ----
    if (tid == 0) {
      ptx::tc_fence_after();
      constexpr uint32_t ID = ptx::idesc_bf16_f32(128, 2 * MT);
      const uint64_t dw = ptx::sw128_desc(s0 + P.wd), da = ptx::sw128_desc(aAct);
#pragma unroll
      for (int t = 0; t < R / 128; ++t)
#pragma unroll
        for (int kk = 0; kk < HS / 16; ++kk)
          ptx::mma_bf16(tmem + COL_P + t * 128, dw + ((t * 16384 + kk * 32) >> 4), da + kk * 2, ID,
                        kk != 0);
      ptx::mma_commit(bar_mma);
    }
    {
      volatile int no_abort = 0;
      ptx::mbar_wait(bar_mma, mma_phase, &no_abort, err);
      mma_phase ^= 1;
    }
    ptx::tc_fence_after();
    {
      // warp p stages owner p's block: its lanes hold channels 32p.. of tile p / 4
      const int p = warp;
      const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + COL_P + (p >> 2) * 128;
      uint32_t* dst = p == q ? (uint32_t*)(sm + P.rcv + q * BLK)
                             : (uint32_t*)(sm + P.ubuf + ((p - q - 1 + CL) % CL) * BLK);
      bool out_of_range = false;
#pragma unroll
      for (int c0 = 0; c0 < MT; c0 += 16) {
        float vh[16], vl[16];
        tmem_ld_cols<16>(ta + c0, vh);
        tmem_ld_cols<16>(ta + MT + c0, vl);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const __half2 h2 =
              to_half2_sat(make_float2(vh[i] + vl[i], vh[i + 1] + vl[i + 1]), out_of_range);
          dst[lane * LDH + (c0 + i) / 2] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      if (out_of_range) atomicOr(err, XP_ERR_RANGE);
      if (p != q) {                        // the warp sends its block as soon as it is staged
        fence_async_smem();
        __syncwarp();
        if (lane == 0)
          ptx::bulk_copy_to_peer(mapa(s0 + P.rcv + q * BLK, p), ptx::smem_u32(dst), BLK,
                                 mapa(bar_p, p));
      }
    }
    ptx::tc_fence_before();
    __syncthreads();                       // the own block is visible to the sum
    mbar_wait_cluster(bar_p, ph, err);
    // everything addressed to this CTA has landed: after its last group it can
    // release the peers' exit barrier now
    if (last) cluster_arrive_relaxed();

    // ---- 5. lat (own channels) = u + sum_p partial_p, p = 0..7 in order ----
    for (int i = tid; i < (MT / 2) * CS; i += THREADS) {
      const int mp = i / CS, c = i % CS, m0 = 2 * mp;
      const int r0 = sRow[m0], r1 = sRow[m0 + 1];
      float v0 = sUs[m0 * CS + c], v1 = sUs[(m0 + 1) * CS + c];
#pragma unroll
      for (int p = 0; p < CL; ++p) {
        const uint32_t w = sRcv[p * (BLK / 4) + c * LDH + mp];
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        v0 += f.x;
        v1 += f.y;
      }
      if (r0 >= 0) lat[(int64_t)r0 * R + q * CS + c] = __float2bfloat16_rn(v0);
      if (r1 >= 0) lat[(int64_t)r1 * R + q * CS + c] = __float2bfloat16_rn(v1);
    }
    if (!last) {
      __syncthreads();
      // arm the next group's receive barriers, then tell the peers this CTA's
      // buffers (u, staged and received partials) are free again
      if (tid == 0) {
        ptx::mbar_arrive_expect_tx(bar_u, (CL - 1) * SLICE);
        ptx::mbar_arrive_expect_tx(bar_p, p_bytes_in);
      }
      cluster_arrive();
    }
  }
  cluster_wait();   // no CTA leaves while a peer may still send into it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// co-resident clusters per variant and device, queried once per shared-memory size
constexpr int kMaxDevices = 64;
int g_max_clusters[kMaxDevices][2] = {}, g_max_clusters_smem[kMaxDevices][2] = {};

size_t smem_bytes(int MT, int B) { return (size_t)make_plan(MT, B).total + 1024; }

template <int MTILES>
int max_clusters(int device, int smem) {
  const int d = device >= 0 && device < kMaxDevices ? device : 0;
  int& cached = g_max_clusters[d][MTILES - 2];
  if (cached > 0 && g_max_clusters_smem[d][MTILES - 2] == smem && d == device) return cached;
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
  g_max_clusters_smem[d][MTILES - 2] = smem;
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
  const int clusters = std::min(groups, max_clusters<MTILES>(h->device, smem));
  const Maps maps = {h->tm_wgu, h->tm_wd, h->tm_mixT};
  e = xp_launch_pdl(latent_mma_kernel<MTILES>, dim3(clusters * CL), dim3(THREADS), (size_t)smem,
                    s, maps, blk, am1, xh, (const float*)h->E, (bf16*)lat, N, h->B, h->V, h->err);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool xp_latent_mma_ok(int r, int H, int B, xp_dtype dt) {
  // the production shape of the head: r = 256 (32 channels per CTA), H = 512 (64 units)
  if (dt != XP_BF16 || B < 2 || B > 32 || r != R || H != CL * HS) return false;
  return smem_bytes(32, B) <= 227 * 1024;
}

// Tensor maps of the weight and mixer slices (2-D, bf16).
bool xp_latent_mma_maps(xp_head* h) {
  xp_encode_tiled_fn fn = xp_get_encode_tiled();
  if (!fn) return false;
  const int B = h->B;
  auto enc = [&](CUtensorMap* m, const void* ptr, int rows, int cols, int box_c, int box_r,
                 bool swz128, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_c, (cuuint32_t)box_r};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              swz128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
  };
  return enc(&h->tm_wgu, h->wgu16, CL * 128, R, 64, 128, true, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) &&
         enc(&h->tm_wd, h->w_down, R, CL * HS, 64, R, true) &&
         enc(&h->tm_mixT, h->mixT, B * B, R, CS, std::min(B * B, 256), false);
}

cudaError_t xp_launch_latent_mma(const xp_head* h, const int64_t* blk, const int64_t* am1,
                                 const float* xh, int N, void* lat, cudaStream_t s) {
  // 32-row groups while they fit in one wave of co-resident clusters, else 48-row groups
  const int groups32 = (N + 32 / h->B - 1) / (32 / h->B);
  if (groups32 <= max_clusters<2>(h->device, (int)smem_bytes(32, h->B)) ||
      smem_bytes(48, h->B) > 227 * 1024)
    return launch<2>(h, blk, am1, xh, N, lat, s);
  return launch<3>(h, blk, am1, xh, N, lat, s);
}

namespace {
// [w_gate ; w_up] (bf16) -> fp16 with saturation (exact for magnitudes in fp16's normal
// range), rows reordered for the cluster latent: CTA q's 128 rows are, for g = 0..3,
// gate units q*64 + 16g .. +15 then up units q*64 + 16g .. +15, so that TMEM lane
// quadrant g of its [gate ; up] accumulator holds both halves of 16 units.
__global__ void gu_to_f16_kernel(const bf16* __restrict__ wg, const bf16* __restrict__ wu,
                                 __half* __restrict__ out, int rows, int r, uint32_t* err) {
  bool clipped = false;
  const int64_t n = (int64_t)2 * rows * r;
  for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < n;
       o += (int64_t)gridDim.x * blockDim.x) {
    const int row = (int)(o / r), k = (int)(o % r);
    const int qq = row / 128, rr = row % 128, g = rr / 32, up = (rr / 16) & 1, i = rr % 16;
    const int src = qq * 64 + 16 * g + i;
    const float v = __bfloat162float((up ? wu : wg)[(int64_t)src * r + k]);
    clipped |= fabsf(v) > 65504.0f;
    out[o] = __float2half_rn(fminf(fmaxf(v, -65504.0f), 65504.0f));
  }
  if (clipped) atomicOr(err, XP_ERR_RANGE);
}
}  // namespace

cudaError_t xp_launch_gu_to_f16(const xp_head* h, const void* w_gate, const void* w_up,
                                cudaStream_t s) {
  const int64_t n = (int64_t)h->H * h->r;
  gu_to_f16_kernel<<<(unsigned)std::min<int64_t>((2 * n + 255) / 256, 1024), 256, 0, s>>>(
      (const bf16*)w_gate, (const bf16*)w_up, (__half*)h->wgu16, h->H, h->r, h->err);
  return cudaGetLastError();
}
