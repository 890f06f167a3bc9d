/*
 * xp.h -- C ABI of the GB300 (sm_103a) XPress Jacobi refinement pass.
 *
 * One pass over a batch of N draft blocks of B slots (slot 0 = the verified
 * anchor) computes, for every slot b:
 *   latent   x[b] = xh[b] + W_lat w1[prev[b]],  prev[0] = am1, prev[b] = blk[b-1]
 *            u[b] = sum_{j<=b} mix[c,b,j] x[j]  (per channel c, folded mixer)
 *            lat[b] = u[b] + W_down (silu(W_gate u[b]) * (W_up u[b]))
 *   readout  logits[b, v] = base[b, v] + lat[b] . w2[v]
 *   argmax   blk[b] = argmax_v logits[b, v], written in place for the next pass
 * for the draft slots b = 1..B-1, and repeats that K times (Jacobi iteration).
 *
 * Sources: the vLLM API page of vllm.model_executor.models.qwen3_xpress
 * ("qwen3_xpress page": XPressRefinerHead and its methods) and the vLLM API
 * page of vllm.v1.worker.gpu.spec_decode.xpress.kernels ("xpress kernels
 * page": the docstrings of the per-pass kernels).
 *
 * Conventions (all entry points):
 *  - Memory is owned by the caller.  The library never allocates device
 *    memory; pointers marked "device" must be device (or managed) memory,
 *    pointers marked "host" host memory.  Sizes are element counts unless
 *    stated otherwise.
 *  - Every call is asynchronous on the given stream (0 = legacy default) and
 *    performs no host synchronisation, except xp_get_error and
 *    xp_head_create/xp_head_refill (which synchronise nothing either, but
 *    read device properties).  Host-side validation runs before any launch;
 *    a call that returns an error has launched nothing.
 *  - A head belongs to the device that was current when it was created.  Every
 *    call that takes a head refuses (XP_EINVAL) while another device is current.
 *  - Calls that take a workspace also take its size in bytes; a workspace smaller
 *    than the call needs (xp_workspace_bytes for that N and topc) is refused with
 *    XP_ECAPACITY before anything is launched.
 *  - Token ids are int64 at the boundary.  A token id outside [0, V) read by
 *    a kernel is clamped into range and raises XP_EBADTOKEN in the head's
 *    device error word (read with xp_get_error); kernels never trap.
 *  - Dtypes: the head's weights, base logits, h and latents all share the
 *    head dtype (XP_BF16 or XP_F32); accumulation is fp32 throughout.
 *  - Argmax ties go to the lowest vocabulary id (full vocabulary, init and
 *    top-C alike); -0 compares equal to +0.  Inputs are assumed finite.
 */
#ifndef XP_H_
#define XP_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  XP_OK = 0,
  XP_EINVAL = 1,        /* null pointer, bad shape, bad stride or alignment            */
  XP_ECAPACITY = 2,     /* N above the head's max_N, or a buffer too small             */
  XP_ENOTPREPARED = 3,  /* head missing (the weights were never prepared)              */
  XP_ECUDA = 4,         /* a CUDA runtime call failed (launch, copy, attribute)        */
  XP_EBADTOKEN = 5,     /* device flag: a token id outside [0, V) was clamped          */
  XP_ETIMEOUT = 6,      /* device flag: a bounded wait inside a kernel gave up         */
  XP_EUNSUPPORTED = 7,  /* shape not supported by this build                           */
  XP_ERANGE = 8         /* device flag: a latent-stage value left the fp16 range of the
                           tensor-core latent's exchanges (saturated; results unreliable) */
} xp_status;

typedef enum { XP_BF16 = 0, XP_F32 = 1 } xp_dtype;

/* Head weights, torch layouts ([out, in] row-major for linear maps).  All
 * pointers are device pointers, read only during xp_head_create /
 * xp_head_refill (they are copied into the head's prepared memory).
 * qwen3_xpress page, XPressRefinerHead.__init__. */
typedef struct {
  int V;          /* vocabulary size                                   */
  int hidden;     /* target-model hidden size                          */
  int r;          /* refiner rank (latent width)                       */
  int H;          /* SwiGLU hidden size (mlp_hidden)                   */
  int B;          /* block size (slots per draft block, >= 2)          */
  int max_N;      /* most blocks any call will pass (max_num_reqs)     */
  xp_dtype dtype; /* storage type of every tensor below                */
  const void* w1;       /* [V, r]       token embedding                     */
  const void* down_h;   /* [r, hidden]                                      */
  const void* down_g;   /* [r, hidden]                                      */
  const void* in_proj;  /* [r, 3r]      columns: down_h | down_g | embedding */
  const void* mix_L;    /* [r, B, B]    FOLDED mixer (raw*tril + I), index  */
                        /*              [channel, out slot, in slot]        */
  const void* w_gate;   /* [H, r]                                           */
  const void* w_up;     /* [H, r]                                           */
  const void* w_down;   /* [r, H]                                           */
  const void* w2;       /* [V, r]       readout                             */
} xp_weights;

typedef struct xp_head xp_head; /* opaque, host-side */

/* Device bytes the head's prepared copies need (caller allocates them once).
 * Beyond copies of the weights (about 2 * V * r * es for w1 and w2), a bf16 head with
 * r = 256 and H = 512 also keeps the projected embedding table E = w1 . W_lat^T in
 * fp32, V * r * 4 bytes (155 MB at V = 151936), so that each pass gathers one row of
 * it per slot instead of multiplying W_lat; and the folded hidden-cache projection
 * as two bf16 planes, 2 * 2r * hidden * 2 bytes (8 MB at hidden = 4096). */
size_t xp_head_prep_bytes(const xp_weights* w);

/* Device bytes of the per-call workspace for up to N blocks; topc > 0 adds
 * the candidate buffers of the top-C path for C = min(topc, V): cand and base_c,
 * plus w2c only where xp_jacobi_refine copies the candidates' w2 rows (while
 * N*(B-1)*C <= V; beyond that each pass reads them by id from w2). */
size_t xp_workspace_bytes(const xp_weights* w, int N, int topc);

/* Zero a workspace once after allocating it.  The argmax finish keeps its
 * counters at zero between calls; after XP_ETIMEOUT, zero it again. */
xp_status xp_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/* Copy and lay out the weights into prep_dev (device, prep_bytes >=
 * xp_head_prep_bytes) and return a host handle.  qwen3_xpress page,
 * process_weights_after_loading: prepared copies the kernels index directly. */
xp_status xp_head_create(const xp_weights* w, void* prep_dev, size_t prep_bytes,
                         cudaStream_t stream, xp_head** out);

/* Refill the prepared copies in place from new weights of the same shapes, so
 * that captured CUDA graphs keep their addresses (process_weights_after_loading
 * on a reload). */
xp_status xp_head_refill(xp_head* head, const xp_weights* w, cudaStream_t stream);

void xp_head_destroy(xp_head* head);

/* mix_L[c,b,j] = raw_L[c,b,j] * [j <= b] + [j == b], evaluated in fp64 and
 * rounded once to dtype.  raw_L, mix_L: device [r, B, B].
 * qwen3_xpress page, XPressRefinerHead.fold_from_raw_. */
xp_status xp_fold_mix(const void* raw_L, void* mix_L, int r, int B, xp_dtype dtype,
                      cudaStream_t stream);

/* Pass-invariant hidden half of in_proj, once per draft step:
 *   xh[n,b] = in_proj[:, :2r] . [down_h h[n,b] ; down_g mean_b' h[n,b']]
 * h_full: device [N, B, hidden] (head dtype); xh: device [N, B, r] fp32.
 * ws: workspace of ws_bytes >= xp_workspace_bytes(w, N, 0).
 * qwen3_xpress page, hidden_cache and the xh hoist in jacobi_refine_greedy. */
xp_status xp_hidden_cache(const xp_head* head, const void* h_full, int N, float* xh,
                          void* ws, size_t ws_bytes, cudaStream_t stream);

/* Latent stage of one pass (all slots), written for slots 1..B-1:
 * blk: device [N, B] int64; am1: device [N] int64; xh: device [N, B, r] fp32;
 * lat: device [N, B-1, r] head dtype (written).
 * Precision of the bf16 tensor-core path (r = 256, H = 512): the mixed latent u
 * and the down projection's partial sums cross between CTAs as fp16 (relative
 * error 2^-11, about a quarter of the bf16 output rounding); the SwiGLU
 * activations are carried as bf16 hi + lo pairs; everything else is fp32.  A value
 * outside the fp16 range saturates and raises XP_ERANGE.
 * xpress kernels page, _xpress_latent_kernel; qwen3_xpress page, _refine_latent. */
xp_status xp_latent_pass(const xp_head* head, const int64_t* blk, const int64_t* am1,
                         const float* xh, int N, void* lat, cudaStream_t stream);

/* Readout + argmax straight into the block:
 *   blk[n, 1+b] = argmax_v (base[n,b,v] + lat[n,b] . w2[v]),  b = 0..B-2
 * lat: device [N, B-1, r] head dtype.  base: device, draft row (n, b) starts
 * at base + n*stride_n + b*stride_b (elements), unit stride over v.  blk:
 * device [N, B] int64, slots 1..B-1 written.  win_val: device [N*(B-1)]
 * fp32 winning logits, or NULL.  ws: workspace of ws_bytes >=
 * xp_workspace_bytes(w, N, 0) (argmax partials).
 * The [N*(B-1), V] logits are never written to memory.
 * xpress kernels page, fused_add_argmax_to_blk; qwen3_xpress page, refine_bias. */
xp_status xp_readout_argmax(const xp_head* head, const void* lat, const void* base,
                            int64_t stride_n, int64_t stride_b, int N, int64_t* blk,
                            float* win_val, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Unfused readout: the draft rows' logits (or the refiner bias alone) instead of
 * their argmax, for callers that sample or otherwise need the distribution:
 *   out[n*(B-1) + b, v] = base[n,b,v] + lat[n,b] . w2[v]   (base given)
 *   out[n*(B-1) + b, v] = lat[n,b] . w2[v]                 (base == NULL)
 * for b = 0..B-2 (the draft slots 1..B-1; slot 0 holds the anchor, whose bias
 * the method never reads).  lat and base as for xp_readout_argmax; base may be
 * NULL.  out: device fp32, row r of the N*(B-1) rows at out + r*ld_out, ld_out
 * >= V elements; the caller owns it (N*(B-1)*ld_out*4 bytes).  Products are
 * accumulated in fp32 and the base value is added in fp32: out is the exact
 * logit up to fp32 rounding, not rounded to the head dtype.  No workspace.
 * XP_EINVAL: null lat/out, ld_out < V, negative N or strides.
 * qwen3_xpress page, refine_bias (w2 applied to the refined latent) and the
 * base + bias sum that fused_add_argmax_to_blk reduces. */
xp_status xp_refine_logits(const xp_head* head, const void* lat, const void* base,
                           int64_t stride_n, int64_t stride_b, int N, float* out,
                           int64_t ld_out, cudaStream_t stream);

/* xp_readout_argmax for callers that cannot allocate device memory -- no
 * counterpart on the pages; the refinement method itself says nothing about
 * where scratch lives.  Same arguments and results as xp_readout_argmax,
 * without the workspace: the cross-CTA argmax scratch (48 KB) is a fixed array
 * in the library's device memory, present on every GPU that loads the library
 * until the process exits.  Meant for callers that run inside a memory pool
 * they do not own, or on a path where cudaMalloc and the synchronisation it can
 * bring are not acceptable.  Limit: N*(B-1) <= 4096 draft rows, else
 * XP_ECAPACITY.  The first call on a device looks the array up (once per
 * device, on the current device); make that first call before any stream
 * capture.  All calls share the one array, so calls that overlap on the GPU
 * (other streams, other threads) race; each call clears it before use. */
xp_status xp_readout_argmax_noalloc(const xp_head* head, const void* lat, const void* base,
                                    int64_t stride_n, int64_t stride_b, int N, int64_t* blk,
                                    float* win_val, cudaStream_t stream);

/* Initial block: blk[n,0] = anchor[n], blk[n,1+b] = argmax_v base[n,b,v].
 * Same base addressing and workspace as xp_readout_argmax.  anchor: device [N] int64.
 * qwen3_xpress page, jacobi_refine_greedy (before the passes). */
xp_status xp_init_argmax(const xp_head* head, const void* base, int64_t stride_n,
                         int64_t stride_b, const int64_t* anchor, int N, int64_t* blk,
                         float* win_val, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Top-C candidates, once per draft step.  Per draft row: the C largest base
 * values (ties at the boundary to the lower id), stored in ascending id order:
 * cand: device [N, B-1, C] int64; base_c: device [N, B-1, C] head dtype;
 * w2c: device [N, B-1, C, r] head dtype = w2[cand] rows, or NULL to have the
 * top-C readout gather w2 rows itself each pass.  blk: device [N, B] int64 or
 * NULL; when given, slots 1..B-1 receive the base argmax (the init).
 * 1 <= C <= V.  qwen3_xpress page, jacobi_refine_greedy top-C branch. */
xp_status xp_topc_gather(const xp_head* head, const void* base, int64_t stride_n,
                         int64_t stride_b, int N, int C, int64_t* cand, void* base_c,
                         void* w2c, int64_t* blk, cudaStream_t stream);

/* Top-C readout + argmax, per pass:
 *   blk[n, 1+b] = cand[n,b,k*],  k* = argmax_k (base_c[n,b,k] + w2c[n,b,k] . lat[n,b])
 * ties to the lowest vocabulary id.  w2c may be NULL (rows gathered from the
 * head's w2 through cand).  win_val: device [N*(B-1)] fp32 or NULL.
 * xpress kernels page, _xpress_topc_argmax_to_blk_kernel. */
xp_status xp_topc_readout_argmax(const xp_head* head, const void* lat, const void* base_c,
                                 const int64_t* cand, const void* w2c, int N, int C,
                                 int64_t* blk, float* win_val, cudaStream_t stream);

/* Whole draft step: hidden cache, init argmax (or top-C gather when topc > 0),
 * then K passes of latent + readout-argmax.  blk: device [N, B] int64 (out;
 * slot 0 = anchor).  topc >= V scores the full vocabulary through the top-C
 * path with C = V.  ws: workspace of ws_bytes >= xp_workspace_bytes(w, N, topc).
 * Top-C: the candidates' w2 rows are copied once per step while N*(B-1)*C <= V
 * (the copy is no larger than w2); for larger batches every pass reads them by id
 * from w2 instead.  Both give the same blk.
 * qwen3_xpress page, XPressRefinerHead.jacobi_refine_greedy. */
xp_status xp_jacobi_refine(const xp_head* head, const void* base, int64_t stride_n,
                           int64_t stride_b, const void* h_full, const int64_t* anchor,
                           const int64_t* am1, int N, int K, int topc, int64_t* blk,
                           void* ws, size_t ws_bytes, cudaStream_t stream);

/* The K passes of xp_jacobi_refine alone, for callers that prepare the pass-invariant
 * inputs themselves: blk (device [N, B] int64) holds the initial block (slot 0 = anchor,
 * slots 1..B-1 the initial tokens, e.g. from xp_init_argmax) and is refined in place; xh
 * (device [N, B, r] fp32) is the hidden cache of xp_hidden_cache; am1 and the base
 * addressing as for xp_jacobi_refine; ws of ws_bytes >= xp_workspace_bytes(w, N, 0).
 * Full-vocabulary scoring.  Each pass is one latent and one readout launch, or, under
 * XP_PASSES_PERSISTENT with a bf16 head of r = 256, H = 512 and B <= 16, all K passes run
 * in one persistent launch (one CTA per SM, every CTA resident at once).  Both give the
 * same blk up to the latent's rounding (see xp_latent_pass).
 * qwen3_xpress page, XPressRefinerHead.jacobi_refine_greedy (the loop over passes). */
xp_status xp_jacobi_passes(const xp_head* head, const void* base, int64_t stride_n,
                           int64_t stride_b, const float* xh, const int64_t* am1, int N, int K,
                           int64_t* blk, void* ws, size_t ws_bytes, cudaStream_t stream);

/* How xp_jacobi_refine and xp_jacobi_passes run the passes (full vocabulary):
 *  XP_PASSES_AUTO        the faster of the two for the shapes; on GB300 that has been the
 *                        per-stage launches at every measured shape (single request,
 *                        batched decode, max batch), so AUTO runs them
 *  XP_PASSES_PERSISTENT  the persistent launch wherever the shapes allow it
 *  XP_PASSES_PER_STAGE   one latent and one readout launch per pass
 * The choice changes the launches, not the method: blocks agree up to the latent's
 * rounding.  Default XP_PASSES_AUTO.  XP_EINVAL for another value. */
enum { XP_PASSES_AUTO = 0, XP_PASSES_PERSISTENT = 1, XP_PASSES_PER_STAGE = 2 };
xp_status xp_set_pass_mode(xp_head* head, int mode);

/* The tensor-core argmax readout (xp_readout_argmax, the per-stage passes, the
 * workspace-free readout) takes up to 128 draft rows per CTA.  When the row tiles come in
 * an even number, on = 1 runs them as 2-CTA clusters whose two CTAs share every MMA and
 * stage half of each w2 tile each; on = 0 (the default) keeps one CTA per row tile.  Both
 * compute the same fp32 dot products over the same k order.  The readout's vocabulary
 * loop is bound by the HBM stream of base rather than by shared-memory traffic, so pairs
 * have not been faster on GB300; the setting is there for shapes where w2 traffic
 * dominates.  XP_EINVAL for another value.  Host only. */
xp_status xp_set_readout_pairs(xp_head* head, int on);

/* 1 when an argmax readout of N blocks would run as 2-CTA pairs under the head's
 * setting, else 0.  Host only. */
int xp_readout_pairs(const xp_head* head, int N);

/* 1 when a full-vocabulary refine of N blocks over this base addressing would run its
 * passes in the persistent launch under the head's pass mode, else 0.  Host only. */
int xp_passes_persistent(const xp_head* head, const void* base, int64_t stride_n,
                         int64_t stride_b, int N);

/* Synchronise `stream`, read and clear the head's device error word:
 * XP_OK, XP_EBADTOKEN, XP_ERANGE or XP_ETIMEOUT (precedence in reverse order). */
xp_status xp_get_error(const xp_head* head, cudaStream_t stream);

/* Failure-path self-test (no counterpart on the pages): launches one kernel whose
 * mbarrier wait nothing will ever complete.  Like every wait in this library it
 * gives up after about half a second and records XP_ETIMEOUT in the head's error
 * word (read it with xp_get_error); no trap, no fault, the context stays usable.
 * Returns XP_OK when the launch succeeded. */
xp_status xp_selftest_wait_timeout(const xp_head* head, cudaStream_t stream);

/* Measurement aid (no counterpart on the pages): where xp_jacobi_refine runs all K passes
 * in its persistent kernel (bf16 head, r = 256, H = 512, B <= 16, full vocabulary), it can
 * record when each CTA reached each phase of each pass.  With buf (device) set, later
 * refines of at most K passes write, per CTA c and pass k, twelve globaltimer stamps (ns) at
 * buf[(c * K + k) * 12 + slot]: 0 the CTA's latent work of the pass starts (its tokens are
 * final; 0 if it has none), 1 its latent work is done, 2 its readout starts (its row tile's
 * latent is complete), 3 its readout's winners are merged; within its first latent group
 * of the pass, 8 its tokens are read, 9 its first gathered rows have landed, 4 every CTA of
 * its team has written its slice of the mixed latent u, 5 its SwiGLU activations are
 * written, 6 its down-projection partials are written, 7 every CTA of its team has
 * written its partials; in its readout, 10 its latent tile is in tensor memory, 11 its
 * first vocabulary tile is reduced.  Slots a CTA never reaches stay as they were.  *needed (nullable) receives
 * the bytes K passes need.  buf = NULL turns the recording off.  The work done is the same
 * either way.  XP_ECAPACITY when bytes is below *needed. */
xp_status xp_profile_timeline(xp_head* head, void* buf, size_t bytes, int K, size_t* needed);

/* Name of the readout kernel the head uses for its shape (for profiling). */
const char* xp_readout_kernel_name(const xp_head* head);

const char* xp_status_str(xp_status s);

#ifdef __cplusplus
}
#endif

#endif /* XP_H_ */
