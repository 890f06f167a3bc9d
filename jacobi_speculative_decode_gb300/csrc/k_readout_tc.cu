// Tensor-core readout + argmax (sm_103a): blk[n, 1+b] = argmax_v base[n,b,v] + lat[n,b].w2[v]
// (xpress kernels page, fused_add_argmax_to_blk with the w2 matmul of refine_bias fused in).
//
// One CTA owns a tile of up to 128 draft rows (whole blocks only) and a
// contiguous range of 192-wide vocabulary tiles.  The latent tile (128 rows x r)
// lives in tensor memory as the MMA's A operand, so shared memory holds only the
// two streams.  Per vocabulary tile:
//   TMA   w2[v-tile, k-chunk]  (192 x 64 bf16, 128B-swizzled)  -> 6-stage smem ring
//         (4 stages in the logits mode, EMIT below, which needs room for its output)
//   TMA   base[rows, 64 ids]   (one box per 64-id third)        -> 3-stage smem ring
//         (one tile; each thread lifts its row's part of a stage into registers as
//         soon as the tile before it has been reduced, which frees the stage for the
//         next tile's base one tile earlier)
//   MMA   tcgen05 M=128 (rows) x N=192 (vocab) x K=r, A from TMEM, fp32 accumulators
//         in TMEM, double-buffered (2 x 192 columns; A takes the last 128 columns)
//   epilogue: each thread owns one row (one TMEM lane), adds base, keeps a
//         running (max, lowest id) -- in the argmax mode the logits never leave the SM.
// Per-row winners of all CTAs of a row tile merge through a packed atomicMax;
// the CTA that arrives last publishes into blk and resets the partials.
//
// Warp roles (480 threads): warp 0 base producer, warp 1 MMA issuer (+ TMEM
// owner), warp 2 w2 producer, warps 3..14 epilogue: warp w reads TMEM lane
// group w % 4 and third (w - 3) / 4 of every tile; the epilogue warps also write
// the latent tile into TMEM before the first MMA.
//
// CTA pairs (PAIR): when the row tiles come in even numbers, the two CTAs of a 2-CTA
// cluster take two neighbouring row tiles over the same vocabulary range and share each
// MMA (tcgen05 .cta_group::2, M = 256): the even CTA issues it, each CTA keeps its own
// 128 rows of A and of the accumulators in its own tensor memory, and each stages only
// half of every w2 tile (96 of the 192 ids) -- the MMA reads both halves.  Per tile a
// CTA then moves 12 KB instead of 24 KB of w2 per k-chunk through shared memory, whose
// bandwidth the w2 writes, the MMA's operand reads and the base traffic share.  The
// odd CTA's MMA warp forwards the completion of its w2 stages to the even CTA's
// barriers, and its epilogue warps arrive on the even CTA's barriers directly; these
// per-stage and per-tile signals carry no fence (a fenced remote arrive costs a memory
// barrier each, and the forwarding thread would serialise on them): what they report --
// a TMA copy seen complete, tensor-memory reads waited for -- is already ordered.
// Pairs are off unless the caller asks for them: the vocabulary loop is bound by the
// streams from HBM, and on GB300 the pair was not faster than one CTA per row tile.
//
// Every base stage is consumed by one fixed group of four warps (the ring size is a
// multiple of the thirds per tile), and a group consumes its stages in order, so no
// consumer ever waits on a stage more than one phase ahead of the phase it is in:
// an mbarrier parity wait cannot tell a later phase from the previous one.
#include <algorithm>

#include "sm100_ptx.cuh"
#include "xp_device.cuh"

using namespace xpd;

namespace {

constexpr int BM = 128;           // rows per MMA (TMEM lanes)
constexpr int BN = 192;           // vocabulary ids per tile (MMA N)
constexpr int BK = 64;            // k per swizzled chunk (128 bytes of bf16)
constexpr int QPT = BN / 64;      // 64-id thirds per tile
constexpr int EPI_WARPS = 4 * QPT;                  // one warp per (lane quadrant, third)
constexpr int BASE_STAGE_BYTES = 128 * 64 * 2;      // 16 KB: one 64-wide box of <= 128 rows
constexpr int NUM_THREADS = (3 + EPI_WARPS) * 32;   // 480
constexpr int OUT_STAGE_BYTES = 32 * 32 * 4;        // logits: one warp's 32 rows x 32 ids

// k-chunks of w2 in flight: the argmax kernel spends all of shared memory on its rings;
// the logits kernel gives part of it to the per-warp staging of its output.  A CTA of a
// pair stages half a tile per k-chunk (12 KB): its w2 ring holds two tiles in 96 KB,
// which leaves room for a base ring twice as deep (base comes from HBM every pass, w2
// mostly from L2).
template <bool EMIT, bool PAIR>
struct Smem {
  static_assert(!(EMIT && PAIR), "the logits kernel runs unpaired");
  static constexpr int W2_ROWS = PAIR ? BN / 2 : BN;      // w2 rows this CTA stages per tile
  static constexpr int W2_STAGE_BYTES = W2_ROWS * BK * 2;
  static constexpr int W2_STAGES = EMIT ? 4 : (PAIR ? 8 : 6);
  // base: one tile in smem (a pair: two), one more lifted into registers; stage s always
  // holds third s % QPT, so each stage has a single consumer group
  static constexpr int BASE_STAGES = PAIR ? 2 * QPT : QPT;
  static constexpr int OUT_BYTES = EMIT ? EPI_WARPS * OUT_STAGE_BYTES : 0;
  static_assert(BASE_STAGES % QPT == 0, "a base stage always holds the same third");
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL = 2 * BN;                  // latent tile: columns [384, 384 + r/2)
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN);
constexpr uint32_t IDESC_PAIR = ptx::idesc_bf16_f32(2 * BM, BN);   // M = 256 over the pair
static_assert(A_COL + 128 <= TMEM_COLS, "accumulators and the latent tile share TMEM");

template <int W2_STAGES, int BASE_STAGES>
struct Bars {
  uint64_t a_full;
  uint64_t w_full[W2_STAGES], w_empty[W2_STAGES];
  uint64_t c_full[BASE_STAGES], c_empty[BASE_STAGES];
  uint64_t t_full[2], t_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int last;
  uint32_t sink;      // see lift() in the epilogue
};

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// EMIT: instead of the argmax, write the logits base + lat.w2 (or the bias lat.w2 alone
// when has_base is 0) as fp32 rows of `out`; every thread stages its row's 32 values of
// a chunk in the warp's swizzled 4 KB buffer, and the warp then stores four full
// 128-byte row segments per instruction.
template <int KCH, bool EMIT, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1) readout_tc_kernel(
    const __nv_bfloat16* __restrict__ lat, const __grid_constant__ CUtensorMap tm_w2,
    const __grid_constant__ CUtensorMap tm_base, int rows, int Bm1, int B, int V, int rpt, int bpt,
    int n_rt, int n_seg, int nvt, int64_t* __restrict__ blk, float* __restrict__ win,
    const float* __restrict__ pf_rows, int pf_row_bytes,
    unsigned long long* __restrict__ packed, unsigned* __restrict__ ticket, uint32_t* err,
    float* __restrict__ out, int64_t ldo, int has_base) {
  constexpr int W2_STAGES = Smem<EMIT, PAIR>::W2_STAGES;
  constexpr int W2_STAGE_BYTES = Smem<EMIT, PAIR>::W2_STAGE_BYTES;
  constexpr int BASE_STAGES = Smem<EMIT, PAIR>::BASE_STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sW = smem;                                    // W2_STAGES x 24 (pair: 12) KB
  uint8_t* sC = sW + W2_STAGES * W2_STAGE_BYTES;         // BASE_STAGES x 16 KB
  uint8_t* sO = sC + BASE_STAGES * BASE_STAGE_BYTES;    // EMIT: EPI_WARPS x 4 KB
  auto* bars = reinterpret_cast<Bars<W2_STAGES, BASE_STAGES>*>(sO + Smem<EMIT, PAIR>::OUT_BYTES);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tile = blockIdx.x % n_rt, seg = blockIdx.x / n_rt;
  const int vt0 = (int)((int64_t)seg * nvt / n_seg), vt1 = (int)((int64_t)(seg + 1) * nvt / n_seg);
  const int row0 = tile * rpt;
  // pair: rank 0 (even row tile) issues the MMAs; its a_full and t_empty also count the
  // odd CTA's epilogue warps, its w_full the odd CTA's forwarded w2 stage
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
  const uint32_t pair_n = PAIR ? 2u : 1u;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars->a_full), pair_n * EPI_WARPS);   // every epilogue warp
    for (int s = 0; s < W2_STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->w_full[s]), rank == 0 ? pair_n : 1u);
      ptx::mbar_init(ptx::smem_u32(&bars->w_empty[s]), 1);    // the MMA issuer's commit
    }
    for (int s = 0; s < BASE_STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->c_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->c_empty[s]), 4);   // the 4 warps of one third
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->t_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->t_empty[s]), pair_n * EPI_WARPS);
    }
    ptx::mbar_init(ptx::smem_u32(&bars->mma_done), 1);
    bars->abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(ptx::smem_u32(&bars->tmem_base), TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  if constexpr (PAIR) {            // both CTAs' barriers exist before either signals the other
    __syncwarp();
    ptx::cluster_arrive_release();
    ptx::cluster_wait();
  } else {
    __syncthreads();
  }
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  ptx::pdl_trigger();

  if (warp == 0) {
    // ---------------- base producer ----------------
    if (lane == 0 && has_base) {
      ptx::prefetch_tmap(&tm_base);
      const uint64_t pol = ptx::policy_evict_first();
      const uint32_t box_bytes = 64u * (uint32_t)Bm1 * (uint32_t)bpt * 2u;
      uint32_t issued[BASE_STAGES] = {};
      int ci = 0;
      bool ok = true;
      for (int vt = vt0; vt < vt1 && ok; ++vt) {
        for (int qt = 0; qt < QPT && ok; ++qt, ++ci) {
          const int s = ci % BASE_STAGES;
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->c_empty[s]), ((ci / BASE_STAGES) & 1) ^ 1,
                              abort, err);
          if (!ok) break;
          const uint32_t full = ptx::smem_u32(&bars->c_full[s]);
          ptx::mbar_arrive_expect_tx(full, box_bytes);
          ptx::tma_load_3d(ptx::smem_u32(sC + s * BASE_STAGE_BYTES), &tm_base, full,
                           vt * BN + qt * 64, 0, tile * bpt, pol);
          ++issued[s];
        }
      }
      // nothing may land in smem after the CTA is gone: wait for each stage's last load
      for (int s = 0; s < BASE_STAGES; ++s)
        if (issued[s]) {
          volatile int no_abort = 0;
          ptx::mbar_wait(ptx::smem_u32(&bars->c_full[s]), (issued[s] - 1) & 1, &no_abort, err);
        }
    }
  } else if (warp == 2) {
    // ---------------- w2 producer (w2 depends on nothing earlier in the stream) ----------
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_w2);
      const uint64_t pol_keep = ptx::policy_evict_last();
      uint32_t issued[W2_STAGES] = {};
      int wi = 0;
      bool ok = true;
      for (int vt = vt0; vt < vt1 && ok; ++vt) {
        for (int kc = 0; kc < KCH; ++kc, ++wi) {
          const int s = wi % W2_STAGES;
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->w_empty[s]), ((wi / W2_STAGES) & 1) ^ 1, abort,
                              err);
          if (!ok) break;
          const uint32_t full = ptx::smem_u32(&bars->w_full[s]);
          ptx::mbar_arrive_expect_tx(full, W2_STAGE_BYTES);
          ptx::tma_load_2d(ptx::smem_u32(sW + s * W2_STAGE_BYTES), &tm_w2, full, kc * BK,
                           vt * BN + (int)rank * Smem<EMIT, PAIR>::W2_ROWS, pol_keep);
          ++issued[s];
        }
      }
      volatile int no_abort = 0;
      for (int s = 0; s < W2_STAGES; ++s)
        if (issued[s])
          ptx::mbar_wait(ptx::smem_u32(&bars->w_full[s]), (issued[s] - 1) & 1, &no_abort, err);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (pair: the even CTA; the odd one forwards) ----------------
    if (lane == 0 && rank == 0) {
      auto wait_in = [&](uint64_t* b, uint32_t parity) {
        return ptx::mbar_wait(ptx::smem_u32(b), parity, abort, err);
      };
      // a commit arrives on this CTA's barrier and, in a pair, on the odd CTA's
      auto commit = [&](uint64_t* b) {
        if constexpr (PAIR) {
          ptx::mma_commit_pair(ptx::smem_u32(b));
          ptx::mma_commit_pair(ptx::peer_addr(ptx::smem_u32(b), 1));
        } else {
          ptx::mma_commit(ptx::smem_u32(b));
        }
      };
      // a_full: the odd CTA's A rows come with a cluster-scope release
      bool ok = PAIR ? ptx::mbar_wait_acq_cluster(ptx::smem_u32(&bars->a_full), 0, abort, err)
                     : ptx::mbar_wait(ptx::smem_u32(&bars->a_full), 0, abort, err);
      ptx::tc_fence_after();
      int wi = 0, ti = 0;
      for (int vt = vt0; vt < vt1 && ok; ++vt, ++ti) {
        const int buf = ti & 1;
        ok = wait_in(&bars->t_empty[buf], ((ti >> 1) & 1) ^ 1);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * BN);
        for (int kc = 0; kc < KCH && ok; ++kc, ++wi) {
          const int s = wi % W2_STAGES;
          ok = wait_in(&bars->w_full[s], (wi / W2_STAGES) & 1);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t b0 = ptx::smem_u32(sW + s * W2_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {  // A: 16 k = 8 columns per step
            const uint32_t a = tmem + A_COL + (uint32_t)(kc * 32 + kk * 8);
            if constexpr (PAIR)
              ptx::mma_bf16_ts_pair(d, a, ptx::sw128_desc(b0 + kk * 32), IDESC_PAIR, (kc | kk) != 0);
            else
              ptx::mma_bf16_ts(d, a, ptx::sw128_desc(b0 + kk * 32), IDESC, (kc | kk) != 0);
          }
          commit(&bars->w_empty[s]);
        }
        if (ok) commit(&bars->t_full[buf]);
      }
      // every MMA this thread issued has finished before TMEM can be released
      commit(&bars->mma_done);
      volatile int no_abort = 0;
      ptx::mbar_wait(ptx::smem_u32(&bars->mma_done), 0, &no_abort, err);
    } else if (PAIR && lane == 0) {
      // odd CTA: tell the even CTA, in the order its MMAs consume them, that this CTA's
      // half of each w2 stage has landed
      int wi = 0;
      bool ok = true;
      for (int vt = vt0; vt < vt1 && ok; ++vt)
        for (int kc = 0; kc < KCH && ok; ++kc, ++wi) {
          const int s = wi % W2_STAGES;
          ok = ptx::mbar_wait(ptx::smem_u32(&bars->w_full[s]), (wi / W2_STAGES) & 1, abort, err);
          if (ok) ptx::mbar_arrive_remote_relaxed(ptx::peer_addr(ptx::smem_u32(&bars->w_full[s]), 0));
        }
      // the even CTA's last commit: no MMA reads this CTA's shared or tensor memory after it
      volatile int no_abort = 0;
      ptx::mbar_wait(ptx::smem_u32(&bars->mma_done), 0, &no_abort, err);
    }
  } else {
    // ---------------- epilogue: one row per thread, a third of each tile per warp ----------
    const int g = warp & 3;                  // TMEM lane group this warp may access
    const int third = (warp - 3) >> 2;       // which 64 ids of every tile
    const int i = g * 32 + lane;             // row within the tile
    const uint32_t trow = tmem + ((uint32_t)(g * 32) << 16);
    // arrive on a barrier the MMA issuer waits on: in a pair, the even CTA's (a fence-free
    // arrive where it only reports tensor-memory reads that tcgen05.wait::ld has completed)
    auto arrive_issuer = [&](uint64_t* b, bool release) {
      if (PAIR && rank != 0) {
        const uint32_t rb = ptx::peer_addr(ptx::smem_u32(b), 0);
        if (release)
          ptx::mbar_arrive_remote(rb);
        else
          ptx::mbar_arrive_remote_relaxed(rb);
      } else {
        ptx::mbar_arrive(ptx::smem_u32(b));
      }
    };
    {
      // the latent tile into TMEM columns [A_COL, A_COL + r/2): k-chunk c (64 values =
      // 32 columns) of the group's 32 rows is written by the warp with third == c % 3
      ptx::pdl_wait();                       // lat comes from the previous kernel
      const int grow = row0 + i;
      const bool live = i < rpt && grow < rows;
      const uint4* src = reinterpret_cast<const uint4*>(lat + (int64_t)(live ? grow : 0) * (KCH * BK));
      uint4 q[2][8];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = third + QPT * j;
        if (c < KCH)
#pragma unroll
          for (int e = 0; e < 8; ++e) q[j][e] = live ? __ldg(src + c * 8 + e) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = third + QPT * j;
        if (c < KCH) {
          uint32_t v[32];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            v[4 * e] = q[j][e].x;
            v[4 * e + 1] = q[j][e].y;
            v[4 * e + 2] = q[j][e].z;
            v[4 * e + 3] = q[j][e].w;
          }
          ptx::tmem_st32(trow + A_COL + (uint32_t)(c * 32), v);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_issuer(&bars->a_full, true);
    }
    float best = -INFINITY;
    int bi = 0x7FFFFFFF;
    // This thread's 64 base values (its row, its third) of the tile about to be reduced.
    // A base stage is lifted into registers and released as soon as the previous tile
    // has been reduced, not after its own tile: the ring then keeps one more tile in
    // flight than it holds.
    uint4 bq[8] = {};
    auto lift = [&](int ci) -> bool {
      const int st = ci % BASE_STAGES;
      bool got = ptx::mbar_wait(ptx::smem_u32(&bars->c_full[st]), (ci / BASE_STAGES) & 1, abort, err);
      got = __all_sync(0xFFFFFFFFu, got);
      if (!got) return false;
      const uint8_t* rowp = sC + st * BASE_STAGE_BYTES + i * 128;
#pragma unroll
      for (int lc = 0; lc < 8; ++lc)          // logical 16-byte chunk lc sits at lc ^ (row & 7)
        bq[lc] = *reinterpret_cast<const uint4*>(rowp + ((lc ^ (i & 7)) << 4));
      // The release lets TMA overwrite the stage at once, and a shared-memory load that
      // has been issued but has not returned its data can still read it then: on this
      // GPU the last chunks of a row came back as the next tile's base.  So the release
      // waits for the data itself: every lane folds all of it into one word and stores
      // that word, an instruction that cannot issue before every load has returned.
      uint32_t dep = 0;
#pragma unroll
      for (int lc = 0; lc < 8; ++lc) dep ^= bq[lc].x ^ bq[lc].y ^ bq[lc].z ^ bq[lc].w;
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(ptx::smem_u32(&bars->sink)), "r"(dep) : "memory");
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->c_empty[st]));
      return true;
    };
    bool ok = vt0 < vt1 && has_base ? lift(third) : true;
    int ti = 0;
    for (int vt = vt0; vt < vt1 && ok; ++vt, ++ti) {
      const int buf = ti & 1;
      ok = ptx::mbar_wait(ptx::smem_u32(&bars->t_full[buf]), (ti >> 1) & 1, abort, err);
      ok = __all_sync(0xFFFFFFFFu, ok);      // warp-uniform: tcgen05.ld is .sync.aligned
      if (!ok) break;
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
        if constexpr (EMIT) {
          uint8_t* stg = sO + (warp - 3) * OUT_STAGE_BYTES;
          // row `lane` of the warp's 32: eight 16-byte chunks, chunk c at c ^ (lane & 7)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_float4(sc[4 * c], sc[4 * c + 1], sc[4 * c + 2], sc[4 * c + 3]);
          __syncwarp();
          const int c = lane & 7;
          const int v0 = vbase + col + c * 4;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int rl = j * 4 + (lane >> 3);    // row within the warp's 32
            const int it = g * 32 + rl;            // row within the tile
            const float4 q = *reinterpret_cast<const float4*>(stg + rl * 128 + ((c ^ (rl & 7)) << 4));
            if (it < rpt && row0 + it < rows && v0 < V) {
              float* dst = out + (int64_t)(row0 + it) * ldo + v0;
              if (v0 + 4 <= V) {
                __stcs(reinterpret_cast<float4*>(dst), q);
              } else {
                dst[0] = q.x;
                if (v0 + 1 < V) dst[1] = q.y;
                if (v0 + 2 < V) dst[2] = q.z;
              }
            }
          }
          __syncwarp();                            // before the next chunk refills it
          continue;
        }
        const int vlim = V - (vbase + col);          // ids at or past V are padding
        if (vlim < 32) {                             // warp-uniform: only the last tile
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e >= vlim) sc[e] = -INFINITY;
        }
        // chunk maximum first; the lowest index of it only when it beats the row's best
        float m = sc[0];
#pragma unroll
        for (int e = 1; e < 32; ++e) m = fmaxf(m, sc[e]);
        if (m > best) {
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
      if (lane == 0) arrive_issuer(&bars->t_empty[buf], false);
      if (vt + 1 < vt1 && has_base) ok = lift((ti + 1) * QPT + third);
    }
    const int grow = row0 + i;
    if (!EMIT && ok && !*abort && i < rpt && grow < rows && bi != 0x7FFFFFFF)
      atomicMax(packed + grow, pack_best(best, (uint32_t)bi));
  }

  ptx::tc_fence_before();
  if constexpr (PAIR) {            // no remote arrive or MMA read of this CTA is in flight
    __syncwarp();
    ptx::cluster_arrive_release();
    ptx::cluster_wait();
  } else {
    __syncthreads();
  }
  // the TMEM release comes before the publish, which only the last CTA of a row tile does
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (PAIR)
      ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
  // ---------------- publish: the last CTA of this row tile writes blk ----------------
  ptx::pdl_wait();            // blk may still be read by the kernel this one overlapped
  const bool last = !EMIT && arrive_last(ticket + tile, (unsigned)n_seg, &bars->last);
  if (last && threadIdx.x < BM) {
    const int grow = row0 + threadIdx.x;
    if (threadIdx.x < rpt && grow < rows) {
      const unsigned long long pk = atomicExch(packed + grow, 0ull);
      const int n = grow / Bm1, b = grow % Bm1;
      const uint32_t id = packed_idx(pk);
      blk[(int64_t)n * B + 1 + b] = (int64_t)id;
      if (win) win[grow] = packed_val(pk);
      // the next latent stage gathers the row of pf_rows this token selects: ask L2 for
      // it now, while the other row tiles finish
      if (pf_rows) {
        const char* rp = reinterpret_cast<const char*>(pf_rows) + (int64_t)id * pf_row_bytes;
        for (int o = 0; o < pf_row_bytes; o += 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(rp + o));
      }
    }
    if (threadIdx.x == 0) ticket[tile] = 0u;
  }
}

template <bool EMIT, bool PAIR>
constexpr size_t smem_bytes() {
  using S = Smem<EMIT, PAIR>;
  return 1024 + (size_t)S::W2_STAGES * S::W2_STAGE_BYTES + S::BASE_STAGES * BASE_STAGE_BYTES +
         S::OUT_BYTES + sizeof(Bars<S::W2_STAGES, S::BASE_STAGES>);
}
static_assert(smem_bytes<false, false>() <= 227 * 1024, "readout shared memory");
static_assert(smem_bytes<false, true>() <= 227 * 1024, "paired readout shared memory");
static_assert(smem_bytes<true, false>() <= 227 * 1024, "logits shared memory");
static_assert(Smem<false, true>::W2_STAGE_BYTES % 1024 == 0, "128-byte swizzle atoms stay aligned");

bool encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  xp_encode_tiled_fn fn = xp_get_encode_tiled();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Co-resident 4-CTA clusters of the argmax kernel, queried once per device.
constexpr int kMaxDevices = 64;
template <int KCH>
int co_resident_clusters4(int device) {
  constexpr int size = 4;
  static int cached[kMaxDevices] = {};
  auto* kern = readout_tc_kernel<KCH, false, false>;
  const size_t smem = smem_bytes<false, false>();
  const int d = device >= 0 && device < kMaxDevices ? device : 0;
  if (cached[d] > 0 && d == device) return cached[d];
  cudaLaunchConfig_t q = {};
  q.gridDim = dim3(size);
  q.blockDim = dim3(NUM_THREADS);
  q.dynamicSmemBytes = smem;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = size;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  q.attrs = a;
  q.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 0;
  }
  cached[d] = n;
  return n;
}

// Row tiles x vocabulary segments, one CTA each: the row tiles are spread over the SMs
// and every row tile's vocabulary is split into as many segments as there are SMs per
// row tile (block x = segment * n_rt + row tile).
// - When the row tiles come in multiples of 4, groups of 4 row tiles of one segment are
//   launched as 4-CTA clusters, for placement only: the kernel uses no cluster feature,
//   but a cluster is scheduled inside one GPC, so the CTAs that read the same w2 tiles at
//   the same time sit together on one die.  At batched decode (4 row tiles) this took
//   the readout from 44.2 to 40.3 us with the same DRAM bytes; with 8 and 32 row tiles it
//   was within 1% either way.  The segments are capped so that every cluster is resident
//   at once (36 clusters of 4 at this shared-memory size: 144 CTAs).
// - PAIR: neighbouring row tiles of one segment form a 2-CTA cluster that shares its MMAs
//   (the cluster of blocks 2c, 2c + 1 holds row tiles 2p, 2p + 1 of one segment).
template <int KCH, bool PAIR>
cudaError_t launch_argmax(const xp_head* h, const void* lat, const CUtensorMap& tb, int N,
                          int64_t* blk, float* win, unsigned long long* packed,
                          unsigned* ticket, cudaStream_t s) {
  const int Bm1 = h->B - 1, rows = N * Bm1;
  const int bpt = BM / Bm1, rpt = bpt * Bm1;
  const int n_rt = (N + bpt - 1) / bpt;
  const int nvt = (h->V + BN - 1) / BN;
  int n_seg = std::max(1, std::min(nvt, h->num_sms / n_rt));
  const size_t smem = smem_bytes<false, PAIR>();
  auto* kern = readout_tc_kernel<KCH, false, PAIR>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int cluster = PAIR ? 2 : 1;
  if (!PAIR && n_rt % 4 == 0) {
    const int mc = co_resident_clusters4<KCH>(h->device);
    if (mc * 4 >= n_rt) {
      cluster = 4;
      n_seg = std::max(1, std::min(n_seg, mc * 4 / n_rt));
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_rt * n_seg);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, (const __nv_bfloat16*)lat, PAIR ? h->tm_w2_half : h->tm_w2,
                         tb, rows, Bm1, h->B, h->V, rpt, bpt, n_rt, n_seg, nvt, blk, win,
                         h->latent_mma ? (const float*)h->E : (const float*)nullptr, h->r * 4,
                         packed, ticket, h->err, (float*)nullptr, (int64_t)0, 1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int KCH>
cudaError_t launch(const xp_head* h, const void* lat, const CUtensorMap& tb, int N,
                   int64_t* blk, float* win, unsigned long long* packed, unsigned* ticket,
                   cudaStream_t s) {
  if (xp_readout_paired(h, N))
    return launch_argmax<KCH, true>(h, lat, tb, N, blk, win, packed, ticket, s);
  return launch_argmax<KCH, false>(h, lat, tb, N, blk, win, packed, ticket, s);
}

// Logits: row tiles x vocabulary segments as in the argmax launch.
template <int KCH>
cudaError_t launch_logits(const xp_head* h, const void* lat, const CUtensorMap& tb, int has_base,
                          int N, float* out, int64_t ldo, cudaStream_t s) {
  const int Bm1 = h->B - 1, rows = N * Bm1;
  const int bpt = BM / Bm1, rpt = bpt * Bm1;
  const int n_rt = (N + bpt - 1) / bpt;
  const int nvt = (h->V + BN - 1) / BN;
  const int n_seg = std::max(1, std::min(nvt, h->num_sms / n_rt));
  const size_t smem = smem_bytes<true, false>();
  cudaError_t e = cudaFuncSetAttribute(readout_tc_kernel<KCH, true, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_rt * n_seg);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, readout_tc_kernel<KCH, true, false>, (const __nv_bfloat16*)lat,
                         h->tm_w2, tb, rows, Bm1, h->B, h->V, rpt, bpt, n_rt, n_seg, nvt,
                         (int64_t*)nullptr, (float*)nullptr, (const float*)nullptr, 0,
                         (unsigned long long*)nullptr, (unsigned*)nullptr, h->err, out, ldo,
                         has_base);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int xp_readout_tc_tile() { return BN; }

bool xp_readout_paired(const xp_head* h, int N) {
  const int bpt = BM / (h->B - 1);
  const int n_rt = (N + bpt - 1) / bpt;
  return h->readout_pair_ok && h->readout_pairs && N > 0 && n_rt % 2 == 0;
}

bool xp_readout_tc_call_ok(const xp_head* h, const void* lat, const void* base, int64_t sn,
                           int64_t sb, int N) {
  return h->readout_tc && N > 0 && (uintptr_t)lat % 16 == 0 && (uintptr_t)base % 16 == 0 &&
         sn % 8 == 0 && sb % 8 == 0 && sb >= h->V && sn >= (int64_t)(h->B - 1) * sb;
}

cudaError_t xp_launch_readout_tc(const xp_head* h, const void* lat, const void* base, int64_t sn,
                                 int64_t sb, int N, int64_t* blk, float* win,
                                 unsigned long long* packed, unsigned* ticket, cudaStream_t s) {
  if (!xp_readout_tc_call_ok(h, lat, base, sn, sb, N)) return cudaErrorNotSupported;
  const int Bm1 = h->B - 1;
  const int bpt = BM / Bm1;
  CUtensorMap tb;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)h->V, (cuuint64_t)Bm1, (cuuint64_t)N};
    const cuuint64_t strides[2] = {(cuuint64_t)sb * 2, (cuuint64_t)sn * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)Bm1, (cuuint32_t)bpt};
    if (!encode(&tb, base, 3, dims, strides, box)) return cudaErrorNotSupported;
  }
  switch (h->r / BK) {
    case 1: return launch<1>(h, lat, tb, N, blk, win, packed, ticket, s);
    case 2: return launch<2>(h, lat, tb, N, blk, win, packed, ticket, s);
    case 3: return launch<3>(h, lat, tb, N, blk, win, packed, ticket, s);
    case 4: return launch<4>(h, lat, tb, N, blk, win, packed, ticket, s);
  }
  return cudaErrorNotSupported;
}

bool xp_logits_tc_call_ok(const xp_head* h, const void* lat, const void* base, int64_t sn,
                          int64_t sb, int N, const float* out, int64_t ldo) {
  if (!h->readout_tc || N <= 0 || (uintptr_t)lat % 16 != 0 || (uintptr_t)out % 16 != 0 ||
      ldo % 4 != 0)
    return false;
  return !base || xp_readout_tc_call_ok(h, lat, base, sn, sb, N);
}

cudaError_t xp_launch_logits_tc(const xp_head* h, const void* lat, const void* base, int64_t sn,
                                int64_t sb, int N, float* out, int64_t ldo, cudaStream_t s) {
  if (!xp_logits_tc_call_ok(h, lat, base, sn, sb, N, out, ldo)) return cudaErrorNotSupported;
  const int Bm1 = h->B - 1;
  const int bpt = BM / Bm1;
  CUtensorMap tb = h->tm_w2;      // never read when there is no base
  if (base) {
    const cuuint64_t dims[3] = {(cuuint64_t)h->V, (cuuint64_t)Bm1, (cuuint64_t)N};
    const cuuint64_t strides[2] = {(cuuint64_t)sb * 2, (cuuint64_t)sn * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)Bm1, (cuuint32_t)bpt};
    if (!encode(&tb, base, 3, dims, strides, box)) return cudaErrorNotSupported;
  }
  const int hb = base ? 1 : 0;
  switch (h->r / BK) {
    case 1: return launch_logits<1>(h, lat, tb, hb, N, out, ldo, s);
    case 2: return launch_logits<2>(h, lat, tb, hb, N, out, ldo, s);
    case 3: return launch_logits<3>(h, lat, tb, hb, N, out, ldo, s);
    case 4: return launch_logits<4>(h, lat, tb, hb, N, out, ldo, s);
  }
  return cudaErrorNotSupported;
}
