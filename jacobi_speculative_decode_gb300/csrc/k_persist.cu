// All K passes of a draft step in one persistent launch (sm_103a): qwen3_xpress page,
// XPressRefinerHead.jacobi_refine_greedy (the loop latent -> readout -> argmax on the same
// blk); xpress kernels page, module docstring (fusing the latent stage removes the launch
// floor) and fused_add_argmax_to_blk.
//
// One CTA per SM, all co-resident (cooperative launch).  Every CTA owns
//   - a readout unit: a row tile of up to 128 draft rows (whole latent groups) and a
//     contiguous range of 192-wide vocabulary tiles, the same for every pass, and
//   - (CTAs of the first 8 * groups) a share of the latent stage: the CTAs are taken in
//     teams of 8; team j computes the latent of row groups j, j + T, j + 2T, ... (T teams),
//     each group being up to 32 rows (whole blocks); CTA q of a team owns latent channels
//     [32q, 32q + 32) (mixer, residual, output) and hidden units [64q, 64q + 64) (SwiGLU).
// Per pass k every CTA runs its latent rounds, then its readout unit:
//   latent (group g of row tile t):
//     1. wait until every readout CTA of tile t finished pass k-1 (done[t]); the tokens
//        are then final: pass 0 reads blk, later passes the packed argmax words
//     2. x = xh + E[prev] and the causal mixer for the own 32 channels; u is kept in fp32
//        for the residual and written as an fp16 slice, already in the 64-byte-swizzled
//        layout of the MMA operand, to shared memory and to a per-group exchange buffer
//     3. once all 8 slices of the group are written (uxc[g]), the 7 other slices arrive by
//        bulk copies straight into the operand; [gate ; up] of the own units on tcgen05
//        (M = 128 weight rows, N = 32 rows)
//     4. a = silu(gate) * up as bf16 hi + lo; the own units' down projection for all 256
//        channels on tcgen05 (two M = 128 tiles, hi and lo rows side by side as N = 64)
//     5. the partial sums for the other CTAs' channels go to an fp32 exchange buffer; once
//        all 8 have written (xc[g]) each CTA bulk-copies the 7 partials of its channels in
//     6. lat (own channels) = u + the 8 partials in sender order, bf16, to global memory;
//        ready[t] += 1
//   readout (row tile t): wait until every latent CTA of tile t's groups finished pass k
//     (ready[t]); the latent tile goes from global memory to TMEM; then the stream of w2
//     and base tiles as in the single-pass readout (tcgen05 MMA with A in TMEM, base added
//     and the running (max, lowest id) kept in the epilogue); the per-row winners merge into
//     packed[k % 2] with a 64-bit atomicMax; done[t] += 1.  After the last pass, the CTA
//     that completes done[t] writes the tile's rows of blk.
// The packed words of pass k-1 are cleared by the latent of pass k once the team has read
// them (they are merged into again in pass k+1).
//
// Shared memory: the w2 ring (6 x 24 KB) shares its region with the latent's operands
// (the w_gate/w_up fp16 slice, the w_down slice, the mixer's channel slice, x, u fp16, the
// activations).  At a pass boundary the w2 producer waits until every w2 stage has been
// consumed, loads the latent operands into the region, and refills the ring only once the
// latent's last MMA has read them.  The incoming partials and the fp32 u live outside the
// ring.  The base ring is never shared: it keeps streaming the next pass's first tile
// while the latent runs.
// TMEM: the readout's accumulators (2 x 192 columns) and latent tile (128 columns) take all
// 512 columns; the latent's accumulators use columns of the readout's, which are idle
// between the last tile of a pass and the first MMA of the next.
//
// Every wait is bounded (~0.5 s): an mbarrier wait or a counter wait that runs out sets
// XP_ERR_TIMEOUT and a global abort word; from then on every wait returns at once, the
// roles skip their work but keep the same sequence of named barriers, in-flight copies are
// awaited and TMEM is released, so every CTA exits.  The counters then stay dirty: after
// XP_ETIMEOUT the caller zeroes the workspace again.
#include <cuda_fp16.h>

#include <algorithm>

#include "sm100_ptx.cuh"
#include "xp_device.cuh"

using namespace xpd;
typedef __nv_bfloat16 bf16;

namespace {

// readout
constexpr int BM = 128;                // rows per MMA (TMEM lanes)
constexpr int BN = 192;                // vocabulary ids per tile
constexpr int BK = 64;                 // k per 128-byte swizzled chunk
constexpr int KCH = 4;                 // k chunks: r = 256
constexpr int R = KCH * BK;            // latent rank
constexpr int QPT = BN / 64;           // 64-id thirds per tile
constexpr int BASE_STAGES = QPT;
constexpr int EPI_WARPS = 4 * QPT;     // 12
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int NUM_THREADS = (3 + EPI_WARPS) * 32;   // 480
constexpr int W2_STAGES = 6;
constexpr int W2_STAGE_BYTES = BN * BK * 2;         // 24 KB
constexpr int BASE_STAGE_BYTES = 128 * 64 * 2;      // 16 KB
// latent
constexpr int TEAM = 8;                // CTAs per latent team
constexpr int MT = 32;                 // rows per latent group
constexpr int HS = 64;                 // own hidden units
constexpr int CS = 32;                 // own channels
constexpr int BMAX = 16;               // largest block the mixer slice is sized for

// shared memory (offsets from the 1024-aligned base).  Inside the w2 ring's region:
constexpr int LW_WGU = 0;                            // [w_gate ; w_up] slice, fp16, 4 x 16 KB
constexpr int LW_WD = LW_WGU + 4 * 16384;            // w_down[:, own units], 256 x 64 bf16
constexpr int LW_MIX = LW_WD + R * HS * 2;           // mixer [b][j][own channels], bf16
constexpr int LW_X = LW_MIX + BMAX * BMAX * CS * 2;  // x, own channels, fp32 [MT][CS]
constexpr int LW_U16 = LW_X + MT * CS * 4;           // u fp16: 8 slices of [MT][CS], 64B swizzle
constexpr int LW_ACT = LW_U16 + TEAM * MT * CS * 2;  // activations hi then lo, 128B swizzle
constexpr int LW_END = LW_ACT + 2 * MT * 128;
constexpr int RING_BYTES = W2_STAGES * W2_STAGE_BYTES;
// outside it
constexpr int LW_PART = std::max(LW_END, RING_BYTES);          // 7 incoming partials, fp32
constexpr int C_OFF = LW_PART + (TEAM - 1) * MT * CS * 4;     // base ring
constexpr int UOWN_OFF = C_OFF + BASE_STAGES * BASE_STAGE_BYTES;   // u, own channels, fp32
constexpr int BARS_OFF = UOWN_OFF + MT * CS * 4;
constexpr int USLICE = MT * CS * 2;                  // bytes of one fp16 u slice
constexpr int PSLICE = MT * CS * 4;                  // bytes of one fp32 partial slice
static_assert(LW_WD % 1024 == 0 && LW_U16 % 1024 == 0 && LW_ACT % 1024 == 0 &&
              C_OFF % 1024 == 0, "TMA and swizzled operands need 1024-byte alignment");
static_assert(LW_END <= RING_BYTES, "the latent's operands fit in the w2 ring's region");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL = 2 * BN;     // latent tile of the readout
constexpr uint32_t COL_GU = 0;         // latent: [gate ; up], MT columns
constexpr uint32_t COL_P = 128;        // latent: partial tiles at 128 and 256, 2*MT columns each
constexpr uint32_t IDESC_RO = ptx::idesc_bf16_f32(BM, BN);

struct Bars {
  uint64_t a_full;
  uint64_t w_full[W2_STAGES], w_empty[W2_STAGES];
  uint64_t c_full[BASE_STAGES], c_empty[BASE_STAGES];
  uint64_t t_full[2], t_empty[2];
  uint64_t mma_done;
  uint64_t lw_full;     // the latent's operands of a round (w_gate/w_up, w_down, mixer)
  uint64_t u_full;      // the other 7 u slices of the group have landed
  uint64_t m1_done, act_ready, m2_done;
  uint64_t p_full;      // the 7 incoming partials have landed
  uint32_t tmem_base;
  int abort;
  // broadcasts among the epilogue warps, one slot per use: each is written by one thread
  // before a named barrier and read after it, and rewritten only several barriers later
  int f_done, f_last;
  uint32_t sink;
  int tok[MT];
};
constexpr size_t SMEM_BYTES = 1024 + BARS_OFF + sizeof(Bars);
static_assert(SMEM_BYTES <= 227 * 1024, "persistent kernel shared memory");

struct Args {
  // readout geometry
  int rows, Bm1, B, V, rpt, bpt, n_rt, n_seg, nvt;
  // latent geometry
  int N, nb, ngroups, teams;
  int K;
  const float* xh;                 // [N, B, R] fp32
  const float* E;                  // [V, R] fp32
  const int64_t* am1;              // [N]
  int64_t* blk;                    // [N, B]: read at pass 0, written after the last pass
  const bf16* mixT;                // [B][B][R]
  bf16* lat;                       // [rows, R]
  unsigned long long* packed0;     // argmax words of even passes
  unsigned long long* packed1;     // of odd passes
  float* xbuf;                     // [ngroups][TEAM owners][TEAM senders][MT][CS]
  uint8_t* ubuf;                   // [ngroups][TEAM senders][USLICE]
  unsigned* done;                  // [n_rt]
  unsigned* ready;                 // [n_rt]
  unsigned* xc;                    // [ngroups]
  unsigned* uxc;                   // [ngroups]
  unsigned* exit_count;
  unsigned* gabort;
  uint32_t* err;
  // optional phase timestamps (globaltimer, ns): [cta][pass][TL_SLOTS], or null
  unsigned long long* tl;
};
// timestamp slots per CTA and pass: 0 latent start (its tokens are final), 1 latent end (its
// last ready count given), 2 readout start (the tile's latent complete), 3 readout end (its
// winners merged, before its done count); inside the first latent round: 8 tokens shared,
// 9 the first thread's x gathered, 4 all u slices of the team written (the copies are
// issued), 5 activations written, 6 partials written, 7 all partials of the team written
// (the copies are issued); 10 its latent tile is in TMEM, 11 its first vocabulary tile
// is reduced
constexpr int TL_SLOTS = 12;

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// 16-byte read-only load that asks L2 to keep the line (the projected-embedding rows of the
// current tokens: the next pass mostly gathers the same rows again)
__device__ __forceinline__ float4 ldg4_keep(const float* p, uint64_t pol) {
  float4 v;
  asm("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(EPI_THREADS) : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// generic-proxy writes of other CTAs, made visible by an acquire, before bulk copies read them
__device__ __forceinline__ void fence_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// bulk copy global -> shared (no tensor map), completing on an mbarrier
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ int swz64(int row, int c) {      // within one 32-channel slice
  return row * 64 + ((((c >> 3) ^ ((row >> 1) & 3))) << 4) + ((c & 7) << 1);
}

// Abort state: the CTA's own flag (shared) and the launch's (global).  A CTA whose wait runs
// out raises both; a CTA learns of another's abort when one of its own waits runs long, and
// from then on every wait returns false at once.
struct Abort {
  volatile int* cta;
  volatile unsigned* grid;
  // this CTA gave up (its own wait, or it saw the launch's word); shared memory only
  __device__ bool on() const { return *cta != 0; }
  __device__ void raise(uint32_t* err) const {
    atomicOr(err, XP_ERR_TIMEOUT);
    *cta = 1;
    *grid = 1u;
  }
};

// The waits below check the CTA's flag (shared memory) as they poll, but the launch's flag
// (a global load of about a microsecond) only once a wait has run for longer than any wait
// of a healthy launch, so that the global read never delays a waiter in normal running.
constexpr uint64_t kLongWaitNs = 100000ull;       // then also watch the other CTAs' aborts
constexpr uint64_t kGiveUpNs = 500000000ull;      // then give up: XP_ETIMEOUT

__device__ __forceinline__ bool wait_step(uint64_t& t0, const Abort& ab, uint32_t* err) {
  if (*ab.cta) return false;
  const uint64_t now = ptx::globaltimer();
  if (t0 == 0) {
    t0 = now;
  } else if (now - t0 > kLongWaitNs) {
    if (*ab.grid) {
      *ab.cta = 1;
      return false;
    }
    if (now - t0 > kGiveUpNs) {
      ab.raise(err);
      return false;
    }
  }
  return true;
}

// mbarrier wait bounded in time; gives up at once when the CTA or the launch aborted
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, const Abort& ab, uint32_t* err) {
  if (*ab.cta) return false;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && !wait_step(t0, ab, err)) return false;
  }
}

// wait until *c >= target (acquire), bounded in time
__device__ __forceinline__ bool cwait(const unsigned* c, unsigned target, const Abort& ab,
                                      uint32_t* err) {
  if (*ab.cta) return false;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire(c) >= target) return true;
    if ((it & 7u) == 7u && !wait_step(t0, ab, err)) return false;
  }
}

__device__ __forceinline__ void stamp(const Args& a, int k, int slot) {
  if (a.tl) a.tl[((int64_t)blockIdx.x * a.K + k) * TL_SLOTS + slot] = ptx::globaltimer();
}

__device__ __forceinline__ int swz128(int row, int k, int rows) {
  return ((k >> 6) * rows + row) * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + ((k & 7) << 1);
}
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__global__ void __launch_bounds__(NUM_THREADS, 1) refine_persist_kernel(
    const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_base,
    const __grid_constant__ CUtensorMap tm_wgu, const __grid_constant__ CUtensorMap tm_wd,
    const __grid_constant__ CUtensorMap tm_mix, const __grid_constant__ Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t s0 = ptx::smem_u32(sm);
  auto* bars = reinterpret_cast<Bars*>(sm + BARS_OFF);
  float* uown = reinterpret_cast<float*>(sm + UOWN_OFF);
  uint8_t* sC = sm + C_OFF;
  const Abort ab{&bars->abort, a.gabort};

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int cta = blockIdx.x;
  const bool has_ro = cta < a.n_rt * a.n_seg;
  const int tile = cta % a.n_rt, seg = cta / a.n_rt;
  const int vt0 = has_ro ? (int)((int64_t)seg * a.nvt / a.n_seg) : 0;
  const int vt1 = has_ro ? (int)((int64_t)(seg + 1) * a.nvt / a.n_seg) : 0;
  const int row0 = tile * a.rpt;
  const int team = cta / TEAM, q = cta % TEAM;
  const int nrounds = team < a.teams && team < a.ngroups ? (a.ngroups - team + a.teams - 1) / a.teams : 0;
  const int K = a.K;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->a_full), EPI_WARPS);
    for (int s = 0; s < W2_STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->w_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->w_empty[s]), 1);
    }
    for (int s = 0; s < BASE_STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->c_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->c_empty[s]), 4);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->t_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->t_empty[s]), EPI_WARPS);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->mma_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->lw_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->u_full), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->m1_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->act_ready), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->m2_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars->p_full), 1);
    bars->abort = 0;
    // a launch that gave up earlier left the counters dirty: report it, change nothing
    if (*a.gabort != 0u) {
      atomicOr(a.err, XP_ERR_TIMEOUT);
      bars->abort = 1;
    }
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

  if (warp == 0) {
    // ---------------- base producer: every pass's tiles, back to back ----------------
    if (lane == 0 && has_ro) {
      ptx::prefetch_tmap(&tm_base);
      const uint64_t pol = ptx::policy_evict_first();
      const uint32_t box_bytes = 64u * (uint32_t)a.Bm1 * (uint32_t)a.bpt * 2u;
      uint32_t issued[BASE_STAGES] = {};
      int ci = 0;
      for (int k = 0; k < K; ++k)
        for (int vt = vt0; vt < vt1; ++vt)
          for (int qt = 0; qt < QPT; ++qt, ++ci) {
            const int s = ci % BASE_STAGES;
            if (!bwait(ptx::smem_u32(&bars->c_empty[s]), ((ci / BASE_STAGES) & 1) ^ 1, ab, a.err))
              continue;
            const uint32_t full = ptx::smem_u32(&bars->c_full[s]);
            ptx::mbar_arrive_expect_tx(full, box_bytes);
            ptx::tma_load_3d(ptx::smem_u32(sC + s * BASE_STAGE_BYTES), &tm_base, full,
                             vt * BN + qt * 64, 0, tile * a.bpt, pol);
            ++issued[s];
          }
      // nothing may land in shared memory after the CTA is gone
      for (int s = 0; s < BASE_STAGES; ++s)
        if (issued[s]) {
          volatile int no_abort = 0;
          ptx::mbar_wait(ptx::smem_u32(&bars->c_full[s]), (issued[s] - 1) & 1, &no_abort, a.err);
        }
    }
  } else if (warp == 2) {
    // ---------------- w2 producer, and the latent's operand loads ----------------
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_w2);
      ptx::prefetch_tmap(&tm_wgu);
      ptx::prefetch_tmap(&tm_wd);
      ptx::prefetch_tmap(&tm_mix);
      const uint64_t pol_keep = ptx::policy_evict_last();
      uint32_t issued[W2_STAGES] = {};
      uint32_t lw_issued = 0;
      int wi = 0, lr = 0;
      for (int k = 0; k < K; ++k) {
        if (nrounds > 0) {
          // the region holds w2 stages: every chunk issued so far must have been consumed
          for (int j = wi; j < wi + W2_STAGES; ++j)
            bwait(ptx::smem_u32(&bars->w_empty[j % W2_STAGES]), ((j / W2_STAGES) & 1) ^ 1, ab,
                  a.err);
          for (int i = 0; i < nrounds; ++i, ++lr) {
            // the previous round's MMAs have read every operand of the region
            if (i > 0) bwait(ptx::smem_u32(&bars->m2_done), (lr - 1) & 1, ab, a.err);
            if (!ab.on()) {
              const uint32_t lb = ptx::smem_u32(&bars->lw_full);
              ptx::mbar_arrive_expect_tx(lb, 4 * 16384 + R * HS * 2 + a.B * a.B * CS * 2);
              for (int kc = 0; kc < KCH; ++kc)
                ptx::tma_load_2d(s0 + LW_WGU + kc * 16384, &tm_wgu, lb, kc * 64, q * 128, pol_keep);
              ptx::tma_load_2d(s0 + LW_WD, &tm_wd, lb, q * HS, 0, pol_keep);
              ptx::tma_load_2d(s0 + LW_MIX, &tm_mix, lb, q * CS, 0, pol_keep);
              ++lw_issued;
            }
          }
          // the ring refills once the last round's second MMA has read its operands
          bwait(ptx::smem_u32(&bars->m2_done), (lr - 1) & 1, ab, a.err);
        }
        if (!has_ro) continue;
        for (int vt = vt0; vt < vt1; ++vt)
          for (int kc = 0; kc < KCH; ++kc, ++wi) {
            const int s = wi % W2_STAGES;
            if (!bwait(ptx::smem_u32(&bars->w_empty[s]), ((wi / W2_STAGES) & 1) ^ 1, ab, a.err))
              continue;
            const uint32_t full = ptx::smem_u32(&bars->w_full[s]);
            ptx::mbar_arrive_expect_tx(full, W2_STAGE_BYTES);
            ptx::tma_load_2d(ptx::smem_u32(sm + s * W2_STAGE_BYTES), &tm_w2, full, kc * BK,
                             vt * BN, pol_keep);
            ++issued[s];
          }
      }
      volatile int no_abort = 0;
      for (int s = 0; s < W2_STAGES; ++s)
        if (issued[s])
          ptx::mbar_wait(ptx::smem_u32(&bars->w_full[s]), (issued[s] - 1) & 1, &no_abort, a.err);
      if (lw_issued)
        ptx::mbar_wait(ptx::smem_u32(&bars->lw_full), (lw_issued - 1) & 1, &no_abort, a.err);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: latent MMAs, then the pass's readout MMAs ----------------
    if (lane == 0) {
      int wi = 0, ti = 0, lr = 0;
      for (int k = 0; k < K; ++k) {
        for (int i = 0; i < nrounds; ++i, ++lr) {
          const bool ok1 = bwait(ptx::smem_u32(&bars->lw_full), lr & 1, ab, a.err) &&
                           bwait(ptx::smem_u32(&bars->u_full), lr & 1, ab, a.err);
          ptx::tc_fence_after();
          if (ok1) {
            // B = u: k step s (16 channels) is half s % 2 of sender slice s / 2
            constexpr uint32_t ID = ptx::idesc_f16_f32(128, MT);
#pragma unroll
            for (int st = 0; st < R / 16; ++st)
              ptx::mma_bf16(tmem + COL_GU,
                            ptx::sw128_desc(s0 + LW_WGU + (st / 4) * 16384 + (st % 4) * 32),
                            ptx::sw64_desc(s0 + LW_U16 + (st / 2) * USLICE + (st % 2) * 32), ID,
                            st != 0);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->m1_done));
          const bool ok2 = bwait(ptx::smem_u32(&bars->act_ready), lr & 1, ab, a.err);
          ptx::tc_fence_after();
          if (ok2) {
            constexpr uint32_t ID = ptx::idesc_bf16_f32(128, 2 * MT);
#pragma unroll
            for (int t = 0; t < R / 128; ++t)
#pragma unroll
              for (int kk = 0; kk < HS / 16; ++kk)
                ptx::mma_bf16(tmem + COL_P + t * 128,
                              ptx::sw128_desc(s0 + LW_WD + t * 16384 + kk * 32),
                              ptx::sw128_desc(s0 + LW_ACT + kk * 32), ID, kk != 0);
          }
          ptx::mma_commit(ptx::smem_u32(&bars->m2_done));
        }
        if (!has_ro) continue;
        const bool oka = bwait(ptx::smem_u32(&bars->a_full), k & 1, ab, a.err);
        ptx::tc_fence_after();
        for (int vt = vt0; vt < vt1; ++vt, ++ti) {
          const int buf = ti & 1;
          bool ok = oka && bwait(ptx::smem_u32(&bars->t_empty[buf]), ((ti >> 1) & 1) ^ 1, ab, a.err);
          ptx::tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(buf * BN);
          for (int kc = 0; kc < KCH; ++kc, ++wi) {
            const int s = wi % W2_STAGES;
            const bool okw = ok && bwait(ptx::smem_u32(&bars->w_full[s]), (wi / W2_STAGES) & 1, ab, a.err);
            ptx::tc_fence_after();
            if (okw) {
              const uint32_t b0 = ptx::smem_u32(sm + s * W2_STAGE_BYTES);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                ptx::mma_bf16_ts(d, tmem + A_COL + (uint32_t)(kc * 32 + kk * 8),
                                 ptx::sw128_desc(b0 + kk * 32), IDESC_RO, (kc | kk) != 0);
            }
            ptx::mma_commit(ptx::smem_u32(&bars->w_empty[s]));
          }
          ptx::mma_commit(ptx::smem_u32(&bars->t_full[buf]));
        }
      }
      ptx::mma_commit(ptx::smem_u32(&bars->mma_done));
      volatile int no_abort = 0;
      ptx::mbar_wait(ptx::smem_u32(&bars->mma_done), 0, &no_abort, a.err);
    }
  } else {
    // ---------------- epilogue warps: the latent rounds, then the readout epilogue ----------
    const int etid = threadIdx.x - 96;
    const int g4 = warp & 3;                 // TMEM lane quadrant this warp may access
    const int third = (warp - 3) >> 2;
    const int i = g4 * 32 + lane;            // readout row within the tile
    const uint32_t trow = tmem + ((uint32_t)(g4 * 32) << 16);
    int lr = 0, ti = 0;
    const uint64_t pol_e = ptx::policy_evict_last();
    for (int k = 0; k < K; ++k) {
      // =========================== latent rounds of pass k ===========================
      for (int rd = 0; rd < nrounds; ++rd, ++lr) {
        const int g = team + rd * a.teams;
        const int n0 = g * a.nb;
        const int nbv = min(a.nb, a.N - n0);           // blocks of this group
        const int gtile = n0 / a.bpt;
        uint8_t* ubuf_g = a.ubuf + (int64_t)g * TEAM * USLICE;
        // 1. the tokens of the pass are final once tile gtile's readout of pass k-1 is done
        // (every epilogue warp of every readout CTA of the tile counted into done); warp 3
        // waits for that, reads the tokens and shares them with one barrier
        if (warp == 3) {
          int ok = 1;
          if (lane == 0) {
            ok = k == 0 || cwait(a.done + gtile, (unsigned)(a.n_seg * k), ab, a.err);
            bars->f_done = ok;
            if (rd == 0) stamp(a, k, 0);
          }
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0) && !ab.on();
          const int m = lane, bl = m / a.B, b = m % a.B;
          int64_t t = 0;
          if (ok && bl < nbv) {
            const int n = n0 + bl;
            if (b == 0) {
              t = a.am1[n];
            } else if (b == 1 || k == 0) {
              t = a.blk[(int64_t)n * a.B + b - 1];
            } else {
              const unsigned long long* pk = (k & 1) ? a.packed0 : a.packed1;   // pass k-1
              t = (int64_t)packed_idx(__ldcg(pk + (int64_t)n * a.Bm1 + b - 2));
            }
            t = checked_token(t, a.V, a.err);
          }
          bars->tok[m] = (int)t;
        }
        epi_sync();
        const bool live = bars->f_done && !ab.on();
        if (etid == 0 && rd == 0) stamp(a, k, 8);
        // 2. x = xh + E[prev] for the own channels (one float4 per thread), then the mixer
        float* sx = reinterpret_cast<float*>(sm + LW_X);
        if (etid < MT * (CS / 4)) {
          const int m = etid >> 3, c4 = (etid & 7) * 4;
          const int bl = m / a.B;
          const bool v = live && m < a.nb * a.B && bl < nbv;
          const int64_t xr = v ? (int64_t)n0 * a.B + m : 0;
          const float4 xv = __ldg(reinterpret_cast<const float4*>(a.xh + xr * R + q * CS + c4));
          const float4 ev = ldg4_keep(a.E + (int64_t)(v ? bars->tok[m] : 0) * R + q * CS + c4, pol_e);
          *reinterpret_cast<float4*>(sx + m * CS + c4) =
              v ? make_float4(xv.x + ev.x, xv.y + ev.y, xv.z + ev.z, xv.w + ev.w)
                : make_float4(0.f, 0.f, 0.f, 0.f);
          if (etid == 0 && rd == 0) stamp(a, k, 9);
        }
        bwait(ptx::smem_u32(&bars->lw_full), lr & 1, ab, a.err);   // the mixer slice
        epi_sync();
        {
          // u[b, c] = sum_{j <= b} mix[c, b, j] x[j, c] for the own channels; slot 0's u and
          // the rows past the group's whole blocks stay zero (never read out)
          const bf16* smix = reinterpret_cast<const bf16*>(sm + LW_MIX);
          uint8_t* uslice = ubuf_g + q * USLICE;
          bool out_of_range = false;
          for (int it = etid; it < MT * CS; it += EPI_THREADS) {
            const int m = it / CS, c = it % CS;
            const int bl = m / a.B, b = m % a.B;
            float u = 0.f;
            if (m < a.nb * a.B && b > 0) {
              const float* xb = sx + (bl * a.B) * CS + c;
              const bf16* mb = smix + (b * a.B) * CS + c;
              for (int j = 0; j <= b; ++j) u = fmaf(__bfloat162float(mb[j * CS]), xb[j * CS], u);
            }
            uown[m * CS + c] = u;
            out_of_range |= fabsf(u) > 65504.0f;
            const __half h = __float2half_rn(fminf(fmaxf(u, -65504.0f), 65504.0f));
            const int off = swz64(m, c);
            *reinterpret_cast<__half*>(sm + LW_U16 + q * USLICE + off) = h;
            *reinterpret_cast<__half*>(uslice + off) = h;
          }
          if (out_of_range) atomicOr(a.err, XP_ERR_RANGE);
        }
        fence_async_smem();
        epi_sync();
        // 3. the team's other u slices straight into the operand, once all 8 are written
        if (etid == 0) {
          red_release_add(a.uxc + g, 1u);
          if (cwait(a.uxc + g, (unsigned)(TEAM * (k + 1)), ab, a.err)) {
            fence_async_global();
            const uint32_t ub = ptx::smem_u32(&bars->u_full);
            ptx::mbar_arrive_expect_tx(ub, (TEAM - 1) * USLICE);
            for (int p = 0; p < TEAM; ++p)
              if (p != q) bulk_g2s(s0 + LW_U16 + p * USLICE, ubuf_g + p * USLICE, USLICE, ub);
          }
          if (rd == 0) stamp(a, k, 4);
        }
        // [gate ; up] -> a = silu(gate) * up as bf16 hi + lo (warps 3..10)
        bwait(ptx::smem_u32(&bars->m1_done), lr & 1, ab, a.err);
        ptx::tc_fence_after();
        if (warp < 11) {
          constexpr int HALF = MT / 2;
          const int half = (warp - 3) >> 2;
          uint32_t raw[16];
          ptx::tmem_ld16(tmem + ((uint32_t)(g4 * 32) << 16) + COL_GU + half * HALF, raw);
          ptx::tmem_wait_ld();
          const bool lo_lane = lane < 16;
          const int unit = g4 * 16 + (lane & 15);
#pragma unroll
          for (int e = 0; e < HALF / 2; ++e) {
            const float v0 = __uint_as_float(raw[e]), v1 = __uint_as_float(raw[e + HALF / 2]);
            const float other = __shfl_xor_sync(0xFFFFFFFFu, lo_lane ? v1 : v0, 16);
            const float gate = lo_lane ? v0 : other;
            const float up = lo_lane ? other : v1;
            const int m = half * HALF + (lo_lane ? e : HALF / 2 + e);
            const float av = silu_fast(gate) * up;
            const bf16 hi = __float2bfloat16_rn(av);
            const bf16 lo = __float2bfloat16_rn(av - __bfloat162float(hi));
            const int off = swz128(m, unit, MT);
            *reinterpret_cast<bf16*>(sm + LW_ACT + off) = hi;
            *reinterpret_cast<bf16*>(sm + LW_ACT + MT * 128 + off) = lo;
          }
        }
        ptx::tc_fence_before();
        fence_async_smem();
        epi_sync();
        if (etid == 0) {
          ptx::mbar_arrive(ptx::smem_u32(&bars->act_ready));
          if (rd == 0) stamp(a, k, 5);
        }
        // 4./5. the down projection's partials: owner p's 32 channels sit in lane quadrant
        // p % 4 of tile p / 4; warp 3 + e (e < 8) reads owner p = (warp & 3) + 4 * (e / 4)
        bwait(ptx::smem_u32(&bars->m2_done), lr & 1, ab, a.err);
        ptx::tc_fence_after();
        float* xg = a.xbuf + (int64_t)g * TEAM * TEAM * MT * CS;
        if (warp < 11) {
          const int p = g4 + 4 * ((warp - 3) >> 2);
          const uint32_t ta = tmem + ((uint32_t)(g4 * 32) << 16) + COL_P + (p >> 2) * 128;
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int c0 = 0; c0 < MT; c0 += 16) {
            ptx::tmem_ld16(ta + c0, hi);
            ptx::tmem_ld16(ta + MT + c0, lo);
            ptx::tmem_wait_ld();
            if (p != q) {
              float* dst = xg + ((int64_t)(p * TEAM + q) * MT) * CS + lane;
#pragma unroll
              for (int e = 0; e < 16; ++e)
                dst[(c0 + e) * CS] = __uint_as_float(hi[e]) + __uint_as_float(lo[e]);
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e)
                uown[(c0 + e) * CS + lane] += __uint_as_float(hi[e]) + __uint_as_float(lo[e]);
            }
          }
          // each of the 8 reading warps counts its partials out as soon as they are stored
          __syncwarp();
          if (lane == 0) red_release_add(a.xc + g, 1u);
        }
        ptx::tc_fence_before();
        epi_sync();
        // the 7 partials of the own channels in by bulk copies, in sender order (own skipped)
        if (etid == 0) {
          if (rd == 0) stamp(a, k, 6);
          if (cwait(a.xc + g, (unsigned)(TEAM * 8 * (k + 1)), ab, a.err)) {
            fence_async_global();
            const uint32_t pb = ptx::smem_u32(&bars->p_full);
            ptx::mbar_arrive_expect_tx(pb, (TEAM - 1) * PSLICE);
            const float* src = xg + (int64_t)q * TEAM * MT * CS;
            if (q > 0) bulk_g2s(s0 + LW_PART, src, q * PSLICE, pb);
            if (q < TEAM - 1)
              bulk_g2s(s0 + LW_PART + q * PSLICE, src + (int64_t)(q + 1) * MT * CS,
                       (TEAM - 1 - q) * PSLICE, pb);
          }
          if (rd == 0) stamp(a, k, 7);
        }
        // 6. lat (own channels) = u + the partials of all 8 CTAs, in sender order
        if (bwait(ptx::smem_u32(&bars->p_full), lr & 1, ab, a.err)) {
          const float* part = reinterpret_cast<const float*>(sm + LW_PART);
          for (int it = etid; it < MT * CS; it += EPI_THREADS) {
            const int m = it / CS, c = it % CS;
            const int bl = m / a.B, b = m % a.B;
            float v = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < TEAM; ++s2)   // senders 0..7; the own partial is in uown
              if (s2 == q) v += uown[m * CS + c];
              else v += part[(s2 - (s2 > q)) * MT * CS + m * CS + c];
            if (m < a.nb * a.B && bl < nbv && b != 0)
              a.lat[((int64_t)(n0 + bl) * a.Bm1 + b - 1) * R + q * CS + c] = __float2bfloat16_rn(v);
          }
          // the argmax words of pass k-1 for this group's rows were read by the whole team
          // (each CTA passed its own token read before it counted into uxc): clear them
          if (k > 0) {
            unsigned long long* pk = (k & 1) ? a.packed0 : a.packed1;
            for (int rr = q + TEAM * etid; rr < nbv * a.Bm1; rr += TEAM * EPI_THREADS)
              pk[(int64_t)n0 * a.Bm1 + rr] = 0ull;
          }
        }
        // one count per CTA: the barrier orders every warp's stores before the release
        epi_sync();
        if (etid == 0) {
          red_release_add(a.ready + gtile, 1u);
          if (rd == nrounds - 1) stamp(a, k, 1);
        }
      }

      // =========================== readout of pass k ===========================
      if (!has_ro) continue;
      const int tile_blocks = min(a.bpt, a.N - tile * a.bpt);
      const int gpt = (tile_blocks + a.nb - 1) / a.nb;
      // each warp waits for the tile's latent itself (every latent CTA of the tile's groups
      // counted into ready once)
      int rok = 1;
      if (lane == 0) rok = cwait(a.ready + tile, (unsigned)(TEAM * gpt * (k + 1)), ab, a.err);
      const bool live = __shfl_sync(0xFFFFFFFFu, rok, 0) && !ab.on();
      if (etid == 0) stamp(a, k, 2);
      {
        // the latent tile into TMEM columns [A_COL, A_COL + r/2)
        const int grow = row0 + i;
        const bool have = live && i < a.rpt && grow < a.rows;
        const uint4* src = reinterpret_cast<const uint4*>(a.lat + (int64_t)(have ? grow : 0) * R);
        uint4 qv[2][8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = third + QPT * j;
          if (c < KCH)
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[j][e] = have ? __ldcg(src + c * 8 + e) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = third + QPT * j;
          if (c < KCH) {
            uint32_t v[32];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              v[4 * e] = qv[j][e].x;
              v[4 * e + 1] = qv[j][e].y;
              v[4 * e + 2] = qv[j][e].z;
              v[4 * e + 3] = qv[j][e].w;
            }
            ptx::tmem_st32(trow + A_COL + (uint32_t)(c * 32), v);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->a_full));
        if (etid == 0) stamp(a, k, 10);
      }
      float best = -INFINITY;
      int bi = 0x7FFFFFFF;
      uint4 bq[8];
      auto lift = [&](int ci) {
        const int st = ci % BASE_STAGES;
        bwait(ptx::smem_u32(&bars->c_full[st]), (ci / BASE_STAGES) & 1, ab, a.err);
        __syncwarp();
        const uint8_t* rowp = sC + st * BASE_STAGE_BYTES + i * 128;
#pragma unroll
        for (int lc = 0; lc < 8; ++lc)
          bq[lc] = *reinterpret_cast<const uint4*>(rowp + ((lc ^ (i & 7)) << 4));
        // the release waits for the data itself (see the single-pass readout): every lane
        // folds its loaded words into one and stores it before the warp releases the stage
        uint32_t dep = 0;
#pragma unroll
        for (int lc = 0; lc < 8; ++lc) dep ^= bq[lc].x ^ bq[lc].y ^ bq[lc].z ^ bq[lc].w;
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(ptx::smem_u32(&bars->sink)), "r"(dep) : "memory");
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->c_empty[st]));
      };
      if (vt0 < vt1) lift(ti * QPT + third);
      for (int vt = vt0; vt < vt1; ++vt, ++ti) {
        const int buf = ti & 1;
        const bool okt = bwait(ptx::smem_u32(&bars->t_full[buf]), (ti >> 1) & 1, ab, a.err);
        const bool ok = __all_sync(0xFFFFFFFFu, okt);
        ptx::tc_fence_after();
        const int vbase = vt * BN;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int col = third * 64 + cc * 32;
          uint32_t acc[32];
          ptx::tmem_ld32(trow + (uint32_t)(buf * BN + col), acc);
          ptx::tmem_wait_ld();
          float sc[32];
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint4 bv = bq[cc * 4 + ch];
            const uint32_t w4[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float bval = (e & 1) ? bf16hi(w4[e >> 1]) : bf16lo(w4[e >> 1]);
              sc[ch * 8 + e] = __uint_as_float(acc[ch * 8 + e]) + bval;
            }
          }
          const int vlim = a.V - (vbase + col);
          if (vlim < 32) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (e >= vlim) sc[e] = -INFINITY;
          }
          float m = sc[0];
#pragma unroll
          for (int e = 1; e < 32; ++e) m = fmaxf(m, sc[e]);
          if (ok && m > best) {
            int first = 31;
#pragma unroll
            for (int e = 31; e >= 0; --e)
              if (sc[e] == m) first = e;
            best = m;
            bi = vbase + col + first;
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->t_empty[buf]));
        if (etid == 0 && vt == vt0) stamp(a, k, 11);
        if (vt + 1 < vt1) lift((ti + 1) * QPT + third);
      }
      unsigned long long* pk = (k & 1) ? a.packed1 : a.packed0;
      const int grow = row0 + i;
      if (!ab.on() && i < a.rpt && grow < a.rows && bi != 0x7FFFFFFF)
        atomicMax(pk + grow, pack_best(best, (uint32_t)bi));
      if (etid == 0) stamp(a, k, 3);
      // one count per CTA once every warp merged its winners; after the last pass the CTA
      // that completes the tile's count writes the tile's tokens into blk
      epi_sync();
      if (etid == 0) {
        const unsigned t = atom_add_acq_rel(a.done + tile, 1u);
        bars->f_last = k == K - 1 && t == (unsigned)(a.n_seg * K - 1);
      }
      epi_sync();
      if (bars->f_last && !ab.on()) {
        for (int rr = etid; rr < a.rpt && row0 + rr < a.rows; rr += EPI_THREADS) {
          const int gr = row0 + rr;
          const unsigned long long w = __ldcg(pk + gr);
          pk[gr] = 0ull;
          a.blk[(int64_t)(gr / a.Bm1) * a.B + 1 + gr % a.Bm1] = (int64_t)packed_idx(w);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
  // the last CTA to leave resets the counters for the next call (unless a wait gave up)
  if (threadIdx.x == 0) {
    const unsigned t = atom_add_acq_rel(a.exit_count, 1u);
    if (t == gridDim.x - 1 && *a.gabort == 0u) {
      for (int j = 0; j < a.n_rt; ++j) {
        a.done[j] = 0u;
        a.ready[j] = 0u;
      }
      for (int j = 0; j < a.ngroups; ++j) {
        a.xc[j] = 0u;
        a.uxc[j] = 0u;
      }
      *a.exit_count = 0u;
    }
  }
}

bool encode_bf16(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box) {
  xp_encode_tiled_fn fn = xp_get_encode_tiled();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Geometry {
  int nb, bpt, rpt, n_rt, n_seg, nvt, ngroups, teams, grid;
};

// CTAs of the launch that can be resident at once, per device (queried once)
constexpr int kMaxDevices = 64;
int g_resident[kMaxDevices] = {};

int resident_ctas(const xp_head* h) {
  const int d = h->device >= 0 && h->device < kMaxDevices ? h->device : -1;
  if (d >= 0 && g_resident[d] > 0) return g_resident[d];
  int per_sm = 0;
  if (cudaFuncSetAttribute(refine_persist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SMEM_BYTES) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, refine_persist_kernel, NUM_THREADS,
                                                    SMEM_BYTES) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int n = per_sm >= 1 ? h->num_sms : 0;   // one CTA per SM
  if (d >= 0) g_resident[d] = n;
  return n;
}

bool geometry(const xp_head* h, int N, Geometry* g) {
  const int Bm1 = h->B - 1;
  g->nb = MT / h->B;
  g->bpt = (BM / Bm1) / g->nb * g->nb;
  if (g->nb < 1 || g->bpt < 1) return false;
  g->rpt = g->bpt * Bm1;
  g->n_rt = (N + g->bpt - 1) / g->bpt;
  g->nvt = (h->V + BN - 1) / BN;
  g->grid = resident_ctas(h);
  if (g->grid < TEAM || g->n_rt > g->grid) return false;
  g->n_seg = std::max(1, std::min(g->nvt, g->grid / g->n_rt));
  g->ngroups = (N + g->nb - 1) / g->nb;
  g->teams = g->grid / TEAM;
  return true;
}

}  // namespace

bool xp_persist_ok(int r, int H, int B, xp_dtype dt) {
  return dt == XP_BF16 && r == R && H == TEAM * HS && B >= 2 && B <= BMAX;
}

// Measured on GB300 (passes/s of a full step): batched decode 19.4-19.9 k per stage against
// 18.6-18.8 k here, max batch 3.1 k against 2.7 k, single request 44 k against 35 k.  The
// per-stage readout overlaps its prologue and the fill of its rings with the latent
// launch before it, while here the latent's dependency chain (about 10 us from the last
// argmax of a row tile to its next latent tile in tensor memory) runs with the streams
// idle; so the automatic choice is the per-stage launches everywhere.
bool xp_persist_preferred(const xp_head* h, int N) {
  (void)h;
  (void)N;
  return false;
}

size_t xp_persist_xbuf_bytes(int B, int max_N) {
  const int nb = MT / B;
  const size_t groups = (size_t)(max_N + nb - 1) / nb;
  // per group: the partials [owner][sender][MT][CS] fp32, then the u slices [sender]
  return groups * ((size_t)TEAM * TEAM * PSLICE + (size_t)TEAM * USLICE);
}

bool xp_persist_call_ok(const xp_head* h, const void* base, int64_t sn, int64_t sb, int N) {
  if (!h->readout_tc || !h->latent_mma || !xp_persist_ok(h->r, h->H, h->B, h->dtype)) return false;
  if ((uintptr_t)base % 16 != 0 || sn % 8 != 0 || sb % 8 != 0 || sb < h->V ||
      sn < (int64_t)(h->B - 1) * sb)
    return false;
  Geometry g;
  return geometry(h, N, &g);
}

cudaError_t xp_launch_persist(const xp_head* h, const void* base, int64_t sn, int64_t sb, int N,
                              int K, const float* xh, const int64_t* am1, int64_t* blk, void* lat,
                              unsigned long long* packed0, unsigned long long* packed1,
                              void* xbuf, unsigned* counters, cudaStream_t s) {
  Geometry g;
  if (K <= 0 || !xp_persist_call_ok(h, base, sn, sb, N) || !geometry(h, N, &g))
    return cudaErrorNotSupported;
  const int Bm1 = h->B - 1;
  CUtensorMap tb;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)h->V, (cuuint64_t)Bm1, (cuuint64_t)N};
    const cuuint64_t strides[2] = {(cuuint64_t)sb * 2, (cuuint64_t)sn * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)Bm1, (cuuint32_t)g.bpt};
    if (!encode_bf16(&tb, base, 3, dims, strides, box)) return cudaErrorNotSupported;
  }
  Args a;
  a.rows = N * Bm1;
  a.Bm1 = Bm1;
  a.B = h->B;
  a.V = h->V;
  a.rpt = g.rpt;
  a.bpt = g.bpt;
  a.n_rt = g.n_rt;
  a.n_seg = g.n_seg;
  a.nvt = g.nvt;
  a.N = N;
  a.nb = g.nb;
  a.ngroups = g.ngroups;
  a.teams = g.teams;
  a.K = K;
  a.xh = xh;
  a.E = h->E;
  a.am1 = am1;
  a.blk = blk;
  a.mixT = (const bf16*)h->mixT;
  a.lat = (bf16*)lat;
  a.packed0 = packed0;
  a.packed1 = packed1;
  a.xbuf = reinterpret_cast<float*>(xbuf);
  const int groups_cap = (h->max_N + g.nb - 1) / g.nb;
  a.ubuf = reinterpret_cast<uint8_t*>(xbuf) + (size_t)groups_cap * TEAM * TEAM * PSLICE;
  // counters: done[max_N], ready[max_N], xc[max_N], uxc[max_N], exit, abort
  a.done = counters;
  a.ready = counters + h->max_N;
  a.xc = counters + 2 * h->max_N;
  a.uxc = counters + 3 * h->max_N;
  a.exit_count = counters + 4 * h->max_N;
  a.gabort = counters + 4 * h->max_N + 1;
  a.err = h->err;
  const size_t tl_need = (size_t)g.grid * K * TL_SLOTS * sizeof(unsigned long long);
  a.tl = h->timeline && h->timeline_bytes >= tl_need ? (unsigned long long*)h->timeline : nullptr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident at once, or no launch
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, refine_persist_kernel, h->tm_w2, tb, h->tm_wgu,
                                     h->tm_wd, h->tm_mixT, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

size_t xp_persist_counter_words(int max_N) { return (size_t)4 * max_N + 2; }

size_t xp_persist_timeline_bytes(const xp_head* h, int K) {
  return (size_t)resident_ctas(h) * K * TL_SLOTS * sizeof(unsigned long long);
}
