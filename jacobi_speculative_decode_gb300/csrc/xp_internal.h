// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "xp.h"

// Host-side head: shapes, the prepared device copies, device facts.
struct xp_head {
  int V, hidden, r, H, B, max_N;
  xp_dtype dtype;
  int device, num_sms;
  char* prep;            // caller-owned device memory holding everything below
  size_t prep_bytes;
  uint32_t* err;         // device error word (XP_ERR_* bits)
  void *w1, *down_hg, *w_hc, *w_lat, *mix, *w_gate, *w_up, *w_down, *w2;  // down_hg = [down_h ; down_g]
  void* wgu16;           // [w_gate ; w_up] as fp16 in cluster row order (tensor-core latent only)
  void* mixT;            // folded mixer laid out [out slot][in slot][channel]
  float* E;              // w1 . in_proj[:, 2r:]^T, fp32 [V, r] (tensor-core latent only)
  void* hfold;           // [in_proj[:, :r] . down_h ; in_proj[:, r:2r] . down_g] as bf16 hi, lo planes
  int hidden_tc;         // tcgen05 hidden cache usable for this head's shapes
  CUtensorMap tm_hfold;  // hfold viewed as [4r, hidden] (hi rows, then lo rows)
  int readout_tc;        // tcgen05 readout usable for this head's shapes
  int latent_mma;        // cluster tensor-core latent usable for this head's shapes
  CUtensorMap tm_w2;     // W2 [V, r] tiled map for the tcgen05 readout
  CUtensorMap tm_w2_half;  // the same with half-tile boxes (one CTA of a readout pair)
  int readout_pair_ok;   // tm_w2_half could be encoded
  int readout_pairs;     // xp_set_readout_pairs: 2-CTA readout when the row tiles pair up
  CUtensorMap tm_wgu, tm_wd, tm_mixT;  // [w_gate ; w_up] fp16 rows, w_down, mixer slices (TMA)
  void* timeline;        // optional per-CTA per-pass phase timestamps of the persistent refine
  size_t timeline_bytes;
  int pass_mode;         // XP_PASSES_AUTO / _PERSISTENT / _PER_STAGE
};

// device error word bits
enum : uint32_t { XP_ERR_BADTOKEN = 1u, XP_ERR_TIMEOUT = 2u, XP_ERR_RANGE = 4u };

// Workspace layout.  Regions that must stay zero between calls come first and
// are sized by the head's max_N so that the layout never moves with N.
struct xp_ws_layout {
  size_t ro_packed, ro_ticket;        // readout argmax partials, per-row-tile tickets
  size_t in_packed, in_ticket;        // init argmax partials, per-row tickets
  size_t pk1, cnt;                    // persistent refine: odd passes' argmax words, counters
  size_t zero_end;                    // [0, zero_end) must be zero between calls
  size_t xh, lat, part, hc;           // pass data and hidden-cache scratch
  size_t xbuf;                        // persistent refine: latent partial-sum exchange
  int part_rows;                      // rows of fp32 split-K partials the scratch holds
  size_t cand, base_c, w2c;           // top-C tail (sized by the call's N and C)
  size_t total;
};
xp_ws_layout xp_layout(int V, int hidden, int r, int H, int B, int max_N, xp_dtype dt, int N,
                       int C);

static inline size_t xp_elem(xp_dtype d) { return d == XP_BF16 ? 2 : 4; }

// true when the current device is the one the head was created on
bool xp_on_head_device(const xp_head* h);

// ---- launchers (return cudaGetLastError() after launching) -----------------
cudaError_t xp_launch_fold(const void* raw, void* mix, int r, int B, xp_dtype dt, cudaStream_t s);
cudaError_t xp_launch_mix_transpose(const void* mix, void* mixT, int r, int B, xp_dtype dt,
                                    cudaStream_t s);

// E = w1 . w_lat^T, the projected embedding table of the tensor-core latent
cudaError_t xp_launch_embed_table(const xp_head* h, cudaStream_t s);

cudaError_t xp_launch_hidden(const xp_head* h, const void* h_full, int N, float* xh, float* part,
                             float* hc, int part_rows, cudaStream_t s);
// tcgen05 hidden cache over the folded projection (bf16 heads, 2r a multiple of 256)
bool xp_hidden_tc_ok(int r, int hidden, xp_dtype dt);
bool xp_hidden_tc_map(xp_head* h);
cudaError_t xp_launch_hidden_fold(const xp_head* h, const void* in_proj, cudaStream_t s);
bool xp_hidden_tc_call_ok(const xp_head* h, const void* h_full);
// returns cudaErrorNotSupported when h_full cannot be tiled by TMA
cudaError_t xp_launch_hidden_tc(const xp_head* h, const void* h_full, int N, float* xh,
                                float* part, int part_rows, cudaStream_t s);
// the same in two launches, so that independent work can run between them: the GEMM
// lets a programmatically dependent launch start early; the reduce (pdl = true) waits
// for its predecessor before reading the partials
cudaError_t xp_launch_hidden_tc_gemm(const xp_head* h, const void* h_full, int N, float* part,
                                     int part_rows, cudaStream_t s, int* splits_out);
cudaError_t xp_launch_xh_reduce(const xp_head* h, int N, float* xh, const float* part, int splits,
                                cudaStream_t s, bool pdl);

// overlap_prev: launch with a programmatic dependency on the previous kernel, which
// must touch none of base, blk, win or the argmax scratch; the kernel waits for that
// kernel only at its end, so whatever follows sees both completed
cudaError_t xp_launch_init_argmax(const xp_head* h, const void* base, int64_t sn, int64_t sb,
                                  const int64_t* anchor, int N, int64_t* blk, float* win,
                                  unsigned long long* packed, unsigned* ticket, cudaStream_t s,
                                  bool overlap_prev = false);

cudaError_t xp_launch_latent_simt(const xp_head* h, const int64_t* blk, const int64_t* am1,
                                  const float* xh, int N, void* lat, cudaStream_t s);
bool xp_latent_mma_ok(int r, int H, int B, xp_dtype dt);
bool xp_latent_mma_maps(xp_head* h);
// w_gate / w_up copied to fp16 for the tensor-core latent (saturating; XP_ERR_RANGE)
cudaError_t xp_launch_gu_to_f16(const xp_head* h, const void* w_gate, const void* w_up,
                                cudaStream_t s);
cudaError_t xp_launch_latent_mma(const xp_head* h, const int64_t* blk, const int64_t* am1,
                                 const float* xh, int N, void* lat, cudaStream_t s);

cudaError_t xp_launch_readout_simt(const xp_head* h, const void* lat, const void* base,
                                   int64_t sn, int64_t sb, int N, int64_t* blk, float* win,
                                   unsigned long long* packed, unsigned* ticket, cudaStream_t s);
// returns cudaErrorNotSupported when the call's base addressing cannot be tiled by TMA
cudaError_t xp_launch_readout_tc(const xp_head* h, const void* lat, const void* base,
                                 int64_t sn, int64_t sb, int N, int64_t* blk, float* win,
                                 unsigned long long* packed, unsigned* ticket, cudaStream_t s);
int xp_readout_tc_tile();   // vocabulary ids per tile of the tcgen05 readout (w2 map box rows)
// true when the argmax readout of N blocks runs as 2-CTA pairs (even number of row tiles)
bool xp_readout_paired(const xp_head* h, int N);
bool xp_readout_tc_call_ok(const xp_head* h, const void* lat, const void* base, int64_t sn,
                           int64_t sb, int N);
// logits base + lat.w2 (bias alone when base is null) as fp32 rows of out (row stride ldo)
cudaError_t xp_launch_logits_simt(const xp_head* h, const void* lat, const void* base, int64_t sn,
                                  int64_t sb, int N, float* out, int64_t ldo, cudaStream_t s);
// returns cudaErrorNotSupported when the tcgen05 path cannot take the call
cudaError_t xp_launch_logits_tc(const xp_head* h, const void* lat, const void* base, int64_t sn,
                                int64_t sb, int N, float* out, int64_t ldo, cudaStream_t s);
bool xp_logits_tc_call_ok(const xp_head* h, const void* lat, const void* base, int64_t sn,
                          int64_t sb, int N, const float* out, int64_t ldo);

// All K passes in one persistent cooperative launch (bf16, r = 256, H = 512, B <= 16).
bool xp_persist_ok(int r, int H, int B, xp_dtype dt);
size_t xp_persist_xbuf_bytes(int B, int max_N);
size_t xp_persist_counter_words(int max_N);
size_t xp_persist_timeline_bytes(const xp_head* h, int K);
bool xp_persist_call_ok(const xp_head* h, const void* base, int64_t sn, int64_t sb, int N);
// the automatic choice between the persistent and the per-stage passes for N blocks
bool xp_persist_preferred(const xp_head* h, int N);
// returns cudaErrorNotSupported (nothing launched) when the call cannot take this path
cudaError_t xp_launch_persist(const xp_head* h, const void* base, int64_t sn, int64_t sb, int N,
                              int K, const float* xh, const int64_t* am1, int64_t* blk, void* lat,
                              unsigned long long* packed0, unsigned long long* packed1,
                              void* xbuf, unsigned* counters, cudaStream_t s);

cudaError_t xp_launch_topc_gather(const xp_head* h, const void* base, int64_t sn, int64_t sb,
                                  int N, int C, int64_t* cand, void* base_c, void* w2c,
                                  int64_t* blk, const int64_t* anchor, cudaStream_t s);
cudaError_t xp_launch_topc_readout(const xp_head* h, const void* lat, const void* base_c,
                                   const int64_t* cand, const void* w2c, int N, int C,
                                   int64_t* blk, float* win, cudaStream_t s);

// Launch with a programmatic dependency on the previous kernel in the stream:
// the kernel's prologue may overlap that kernel's tail; the kernel itself must
// call griddepcontrol.wait before it touches anything the predecessor writes.
template <typename... KArgs, typename... Args>
cudaError_t xp_launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// tensor-map encoder fetched from the driver at run time (no -lcuda link)
typedef CUresult (*xp_encode_tiled_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                       const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                       const cuuint32_t*, CUtensorMapInterleave,
                                       CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);
xp_encode_tiled_fn xp_get_encode_tiled();
