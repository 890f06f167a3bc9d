// Host side of the C ABI: validation, prepared weight copies, workspace layout
// and the order of launches.  Every compute step runs in the kernels.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "xp_internal.h"

namespace {

constexpr size_t kAlign = 1024;
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

bool valid_weights(const xp_weights* w) {
  if (!w) return false;
  if (w->V <= 0 || w->hidden <= 0 || w->r <= 0 || w->H <= 0 || w->B < 2 || w->max_N <= 0)
    return false;
  if (w->B > 64) return false;   // the latent kernels keep a block's slots on chip
  if (w->dtype != XP_BF16 && w->dtype != XP_F32) return false;
  return true;
}

bool valid_weight_ptrs(const xp_weights* w) {
  return w->w1 && w->down_h && w->down_g && w->in_proj && w->mix_L && w->w_gate && w->w_up &&
         w->w_down && w->w2;
}

struct PrepLayout {
  size_t err, w1, down_hg, w_hc, w_lat, mix, mixT, w_gate, w_up, w_down, w2, E, hfold, wgu16, total;
};

PrepLayout prep_layout(const xp_weights* w) {
  const size_t es = xp_elem(w->dtype);
  const size_t V = w->V, r = w->r, H = w->H, hid = w->hidden, B = w->B;
  PrepLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  L.err = take(256);
  L.w1 = take(V * r * es);
  L.down_hg = take(2 * r * hid * es);
  L.w_hc = take(r * 2 * r * es);
  L.w_lat = take(r * r * es);
  L.mix = take(r * B * B * es);
  L.mixT = take(r * B * B * es);
  L.w_gate = take(H * r * es);
  L.w_up = take(H * r * es);
  L.w_down = take(r * H * es);
  L.w2 = take(V * r * es);
  // projected embedding table, only where the tensor-core latent runs
  L.E = take(xp_latent_mma_ok(w->r, w->H, w->B, w->dtype) ? V * r * 4 : 0);
  // folded hidden-cache projection (hi and lo bf16 planes), only where the tcgen05 path runs
  L.hfold = take(xp_hidden_tc_ok(w->r, w->hidden, w->dtype) ? 2 * 2 * r * hid * 2 : 0);
  L.wgu16 = take(xp_latent_mma_ok(w->r, w->H, w->B, w->dtype) ? 2 * H * r * 2 : 0);
  L.total = o;
  return L;
}

xp_status copy_weights(xp_head* h, const xp_weights* w, cudaStream_t s) {
  const size_t es = xp_elem(w->dtype);
  const size_t V = w->V, r = w->r, H = w->H, hid = w->hidden, B = w->B;
  cudaError_t e = cudaSuccess;
  auto cp = [&](void* dst, const void* src, size_t bytes) {
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
  };
  cp(h->w1, w->w1, V * r * es);
  cp(h->down_hg, w->down_h, r * hid * es);
  cp((char*)h->down_hg + r * hid * es, w->down_g, r * hid * es);
  // in_proj [r, 3r]: columns [0, 2r) act on the hidden cache, [2r, 3r) on the embedding
  if (e == cudaSuccess)
    e = cudaMemcpy2DAsync(h->w_hc, 2 * r * es, w->in_proj, 3 * r * es, 2 * r * es, r,
                          cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpy2DAsync(h->w_lat, r * es, (const char*)w->in_proj + 2 * r * es, 3 * r * es,
                          r * es, r, cudaMemcpyDeviceToDevice, s);
  cp(h->mix, w->mix_L, r * B * B * es);
  if (e == cudaSuccess) e = xp_launch_mix_transpose(h->mix, h->mixT, (int)r, (int)B, w->dtype, s);
  cp(h->w_gate, w->w_gate, H * r * es);
  cp(h->w_up, w->w_up, H * r * es);
  cp(h->w_down, w->w_down, r * H * es);
  cp(h->w2, w->w2, V * r * es);
  if (e == cudaSuccess && h->latent_mma) e = xp_launch_embed_table(h, s);
  if (e == cudaSuccess && h->latent_mma) e = xp_launch_gu_to_f16(h, w->w_gate, w->w_up, s);
  if (e == cudaSuccess && h->hidden_tc) e = xp_launch_hidden_fold(h, w->in_proj, s);
  return e == cudaSuccess ? XP_OK : XP_ECUDA;
}

inline xp_status cuda_status(cudaError_t e) { return e == cudaSuccess ? XP_OK : XP_ECUDA; }

bool valid_base(const xp_head* h, const void* base, int64_t sn, int64_t sb) {
  return base && sn >= 0 && sb >= 0;
}

bool on_head_device(const xp_head* h) { return xp_on_head_device(h); }

// Workspace bytes a call over N blocks (C candidates, 0 = full vocabulary) needs.
size_t ws_needed(const xp_head* h, int N, int C) {
  return xp_layout(h->V, h->hidden, h->r, h->H, h->B, h->max_N, h->dtype, N, C).total;
}

}  // namespace

// ---------------------------------------------------------------------------
// The head's prepared memory, tensor maps and launch decisions belong to the device it
// was created on; a call made while another device is current is refused.
bool xp_on_head_device(const xp_head* h) {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && dev == h->device;
}

xp_ws_layout xp_layout(int V, int hidden, int r, int H, int B, int max_N, xp_dtype dt, int N,
                       int C) {
  (void)hidden;
  const size_t es = xp_elem(dt);
  const size_t rows_cap = (size_t)max_N * (B - 1);
  xp_ws_layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  L.ro_packed = take(rows_cap * 8);
  L.ro_ticket = take(rows_cap * 4);
  L.in_packed = take(rows_cap * 8);
  L.in_ticket = take(rows_cap * 4);
  const bool persist = xp_persist_ok(r, H, B, dt);
  L.pk1 = take(persist ? rows_cap * 8 : 0);
  L.cnt = take(persist ? xp_persist_counter_words(max_N) * 4 : 0);
  L.zero_end = o;
  L.xh = take((size_t)max_N * B * r * 4);
  L.lat = take(rows_cap * r * es);
  L.part_rows = std::max(8192, 2 * max_N * B);
  L.part = take((size_t)L.part_rows * 2 * r * 4);
  L.hc = take((size_t)max_N * B * 2 * r * 4);
  L.xbuf = take(persist ? xp_persist_xbuf_bytes(B, max_N) : 0);
  const size_t rows = (size_t)std::max(N, 0) * (B - 1);
  const size_t c = (size_t)std::max(C, 0);
  L.cand = take(rows * c * 8);
  L.base_c = take(rows * c * es);
  // the candidates' w2 rows are copied once per step only while the copy is no larger
  // than w2 (rows * C <= V); beyond that the passes read them by id from w2
  L.w2c = take(rows * c <= (size_t)V ? rows * c * r * es : 0);
  L.total = o;
  return L;
}

extern "C" {

const char* xp_status_str(xp_status s) {
  switch (s) {
    case XP_OK: return "ok";
    case XP_EINVAL: return "invalid argument";
    case XP_ECAPACITY: return "capacity exceeded";
    case XP_ENOTPREPARED: return "head not prepared";
    case XP_ECUDA: return "CUDA runtime error";
    case XP_EBADTOKEN: return "token id out of range (clamped)";
    case XP_ETIMEOUT: return "bounded wait in a kernel timed out";
    case XP_EUNSUPPORTED: return "unsupported shape";
    case XP_ERANGE: return "latent value outside the fp16 exchange range (saturated)";
  }
  return "unknown status";
}

size_t xp_head_prep_bytes(const xp_weights* w) {
  if (!valid_weights(w)) return 0;
  return prep_layout(w).total;
}

size_t xp_workspace_bytes(const xp_weights* w, int N, int topc) {
  if (!valid_weights(w) || N < 0 || topc < 0) return 0;
  const int C = topc > 0 ? std::min(topc, w->V) : 0;
  return xp_layout(w->V, w->hidden, w->r, w->H, w->B, w->max_N, w->dtype, N, C).total;
}

xp_status xp_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws || ws_bytes == 0) return XP_EINVAL;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, stream));
}

static void decide_paths(xp_head* h);

xp_status xp_head_create(const xp_weights* w, void* prep_dev, size_t prep_bytes,
                         cudaStream_t stream, xp_head** out) {
  if (!out) return XP_EINVAL;
  *out = nullptr;
  if (!valid_weights(w) || !valid_weight_ptrs(w) || !prep_dev) return XP_EINVAL;
  if ((uintptr_t)prep_dev % 256 != 0) return XP_EINVAL;
  const PrepLayout L = prep_layout(w);
  if (prep_bytes < L.total) return XP_ECAPACITY;
  xp_head* h = new (std::nothrow) xp_head();
  if (!h) return XP_ECAPACITY;
  h->V = w->V; h->hidden = w->hidden; h->r = w->r; h->H = w->H; h->B = w->B;
  h->max_N = w->max_N; h->dtype = w->dtype;
  h->readout_pairs = 0;
  h->prep = (char*)prep_dev;
  h->prep_bytes = prep_bytes;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) !=
          cudaSuccess) {
    delete h;
    return XP_ECUDA;
  }
  char* p = h->prep;
  h->err = (uint32_t*)(p + L.err);
  h->w1 = p + L.w1; h->down_hg = p + L.down_hg;
  h->w_hc = p + L.w_hc; h->w_lat = p + L.w_lat; h->mix = p + L.mix;
  h->mixT = p + L.mixT;
  h->E = (float*)(p + L.E);
  h->hfold = p + L.hfold;
  h->wgu16 = p + L.wgu16;
  h->w_gate = p + L.w_gate; h->w_up = p + L.w_up; h->w_down = p + L.w_down; h->w2 = p + L.w2;
  decide_paths(h);
  // the error word starts clear; the weight preparation below may already flag it
  xp_status st = cuda_status(cudaMemsetAsync(h->err, 0, 256, stream));
  if (st == XP_OK) st = copy_weights(h, w, stream);
  if (st != XP_OK) { delete h; return st; }
  *out = h;
  return XP_OK;
}

xp_status xp_head_refill(xp_head* h, const xp_weights* w, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!valid_weights(w) || !valid_weight_ptrs(w)) return XP_EINVAL;
  if (w->V != h->V || w->hidden != h->hidden || w->r != h->r || w->H != h->H || w->B != h->B ||
      w->dtype != h->dtype || w->max_N != h->max_N)
    return XP_EINVAL;
  return copy_weights(h, w, stream);
}

void xp_head_destroy(xp_head* h) { delete h; }

xp_status xp_fold_mix(const void* raw_L, void* mix_L, int r, int B, xp_dtype dtype,
                      cudaStream_t stream) {
  if (!raw_L || !mix_L || r <= 0 || B <= 0 || (dtype != XP_BF16 && dtype != XP_F32))
    return XP_EINVAL;
  return cuda_status(xp_launch_fold(raw_L, mix_L, r, B, dtype, stream));
}

xp_status xp_hidden_cache(const xp_head* h, const void* h_full, int N, float* xh, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!h_full || !xh || !ws || N < 0 || !on_head_device(h)) return XP_EINVAL;
  if (N > h->max_N || ws_bytes < ws_needed(h, N, 0)) return XP_ECAPACITY;
  if (N == 0) return XP_OK;
  const xp_ws_layout L = xp_layout(h->V, h->hidden, h->r, h->H, h->B, h->max_N, h->dtype, N, 0);
  char* w = (char*)ws;
  return cuda_status(xp_launch_hidden(h, h_full, N, xh, (float*)(w + L.part), (float*)(w + L.hc),
                                      L.part_rows, stream));
}

xp_status xp_latent_pass(const xp_head* h, const int64_t* blk, const int64_t* am1,
                         const float* xh, int N, void* lat, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!blk || !am1 || !xh || !lat || N < 0 || !on_head_device(h)) return XP_EINVAL;
  if (N > h->max_N) return XP_ECAPACITY;
  if (N == 0) return XP_OK;
  // the tensor-core latent reads xh in 16-byte pieces and writes lat in channel pairs
  if (h->latent_mma && (uintptr_t)xh % 16 == 0 && (uintptr_t)lat % 4 == 0)
    return cuda_status(xp_launch_latent_mma(h, blk, am1, xh, N, lat, stream));
  return cuda_status(xp_launch_latent_simt(h, blk, am1, xh, N, lat, stream));
}

static xp_status readout_impl(const xp_head* h, const void* lat, const void* base, int64_t sn,
                              int64_t sb, int N, int64_t* blk, float* win, void* ws,
                              cudaStream_t stream) {
  const xp_ws_layout L = xp_layout(h->V, h->hidden, h->r, h->H, h->B, h->max_N, h->dtype, N, 0);
  char* w = (char*)ws;
  auto* packed = (unsigned long long*)(w + L.ro_packed);
  auto* ticket = (unsigned*)(w + L.ro_ticket);
  if (h->readout_tc && xp_readout_tc_call_ok(h, lat, base, sn, sb, N)) {
    const cudaError_t e =
        xp_launch_readout_tc(h, lat, base, sn, sb, N, blk, win, packed, ticket, stream);
    if (e != cudaErrorNotSupported) return cuda_status(e);
  }
  return cuda_status(
      xp_launch_readout_simt(h, lat, base, sn, sb, N, blk, win, packed, ticket, stream));
}

xp_status xp_readout_argmax(const xp_head* h, const void* lat, const void* base, int64_t sn,
                            int64_t sb, int N, int64_t* blk, float* win, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!lat || !valid_base(h, base, sn, sb) || !blk || !ws || N < 0 || !on_head_device(h))
    return XP_EINVAL;
  if (N > h->max_N || ws_bytes < ws_needed(h, N, 0)) return XP_ECAPACITY;
  if (N == 0) return XP_OK;
  return readout_impl(h, lat, base, sn, sb, N, blk, win, ws, stream);
}

xp_status xp_refine_logits(const xp_head* h, const void* lat, const void* base, int64_t sn,
                           int64_t sb, int N, float* out, int64_t ld_out, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!lat || !out || (base && !valid_base(h, base, sn, sb)) || ld_out < h->V || N < 0 ||
      !on_head_device(h))
    return XP_EINVAL;
  if (N > h->max_N) return XP_ECAPACITY;
  if (N == 0) return XP_OK;
  if (xp_logits_tc_call_ok(h, lat, base, sn, sb, N, out, ld_out)) {
    const cudaError_t e = xp_launch_logits_tc(h, lat, base, sn, sb, N, out, ld_out, stream);
    if (e != cudaErrorNotSupported) return cuda_status(e);
  }
  return cuda_status(xp_launch_logits_simt(h, lat, base, sn, sb, N, out, ld_out, stream));
}

xp_status xp_init_argmax(const xp_head* h, const void* base, int64_t sn, int64_t sb,
                         const int64_t* anchor, int N, int64_t* blk, float* win, void* ws,
                         size_t ws_bytes, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!valid_base(h, base, sn, sb) || !anchor || !blk || !ws || N < 0 || !on_head_device(h))
    return XP_EINVAL;
  if (N > h->max_N || ws_bytes < ws_needed(h, N, 0)) return XP_ECAPACITY;
  if (N == 0) return XP_OK;
  const xp_ws_layout L = xp_layout(h->V, h->hidden, h->r, h->H, h->B, h->max_N, h->dtype, N, 0);
  char* w = (char*)ws;
  return cuda_status(xp_launch_init_argmax(h, base, sn, sb, anchor, N, blk, win,
                                           (unsigned long long*)(w + L.in_packed),
                                           (unsigned*)(w + L.in_ticket), stream));
}

xp_status xp_topc_gather(const xp_head* h, const void* base, int64_t sn, int64_t sb, int N, int C,
                         int64_t* cand, void* base_c, void* w2c, int64_t* blk,
                         cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!valid_base(h, base, sn, sb) || !cand || !base_c || N < 0 || C < 1 || C > h->V ||
      !on_head_device(h))
    return XP_EINVAL;
  if (N > h->max_N) return XP_ECAPACITY;
  if (N == 0) return XP_OK;
  return cuda_status(
      xp_launch_topc_gather(h, base, sn, sb, N, C, cand, base_c, w2c, blk, nullptr, stream));
}

xp_status xp_topc_readout_argmax(const xp_head* h, const void* lat, const void* base_c,
                                 const int64_t* cand, const void* w2c, int N, int C, int64_t* blk,
                                 float* win, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!lat || !base_c || !cand || !blk || N < 0 || C < 1 || C > h->V || !on_head_device(h))
    return XP_EINVAL;
  if (N > h->max_N) return XP_ECAPACITY;
  if (N == 0) return XP_OK;
  return cuda_status(xp_launch_topc_readout(h, lat, base_c, cand, w2c, N, C, blk, win, stream));
}

// K full-vocabulary passes on an initialised block: K x (latent, readout), or the persistent
// kernel when the head's pass mode asks for it and the shapes allow it.
static xp_status passes_impl(const xp_head* h, const void* base, int64_t sn, int64_t sb,
                             const float* xh, const int64_t* am1, int N, int K, int64_t* blk,
                             char* w, const xp_ws_layout& L, cudaStream_t stream) {
  const bool persist = h->pass_mode == XP_PASSES_PERSISTENT ||
                       (h->pass_mode == XP_PASSES_AUTO && xp_persist_preferred(h, N));
  if (K > 0 && persist && L.xbuf && xp_persist_call_ok(h, base, sn, sb, N)) {
    const cudaError_t ep = xp_launch_persist(
        h, base, sn, sb, N, K, xh, am1, blk, w + L.lat, (unsigned long long*)(w + L.ro_packed),
        (unsigned long long*)(w + L.pk1), (void*)(w + L.xbuf), (unsigned*)(w + L.cnt), stream);
    if (ep == cudaSuccess) return XP_OK;
    cudaGetLastError();   // not launched (e.g. not co-resident): the per-pass kernels
  }
  xp_status st = XP_OK;
  for (int k = 0; k < K && st == XP_OK; ++k) {
    st = xp_latent_pass(h, blk, am1, xh, N, w + L.lat, stream);
    if (st == XP_OK) st = readout_impl(h, w + L.lat, base, sn, sb, N, blk, nullptr, w, stream);
  }
  return st;
}

xp_status xp_jacobi_refine(const xp_head* h, const void* base, int64_t sn, int64_t sb,
                           const void* h_full, const int64_t* anchor, const int64_t* am1, int N,
                           int K, int topc, int64_t* blk, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!valid_base(h, base, sn, sb) || !h_full || !anchor || !am1 || !blk || !ws || N < 0 ||
      K < 0 || topc < 0 || !on_head_device(h))
    return XP_EINVAL;
  const int C = topc > 0 ? std::min(topc, h->V) : 0;
  if (N > h->max_N || ws_bytes < ws_needed(h, N, C)) return XP_ECAPACITY;
  if (N == 0) return XP_OK;
  const xp_ws_layout L = xp_layout(h->V, h->hidden, h->r, h->H, h->B, h->max_N, h->dtype, N, C);
  char* w = (char*)ws;
  float* xh = (float*)(w + L.xh);
  void* lat = w + L.lat;
  xp_status st = XP_OK;
  if (C == 0 && xp_hidden_tc_call_ok(h, h_full)) {
    // the hidden-cache GEMM and the init argmax are independent: the init runs beside
    // the GEMM, the reduce of the GEMM's partials after both
    int splits = 0;
    cudaError_t e = xp_launch_hidden_tc_gemm(h, h_full, N, (float*)(w + L.part), L.part_rows,
                                             stream, &splits);
    if (e == cudaSuccess)
      e = xp_launch_init_argmax(h, base, sn, sb, anchor, N, blk, nullptr,
                                (unsigned long long*)(w + L.in_packed),
                                (unsigned*)(w + L.in_ticket), stream, true);
    if (e == cudaSuccess) e = xp_launch_xh_reduce(h, N, xh, (float*)(w + L.part), splits, stream, true);
    if (e != cudaErrorNotSupported) {
      st = cuda_status(e);
      // all K passes in one persistent launch where the shapes allow it
      if (st == XP_OK) st = passes_impl(h, base, sn, sb, xh, am1, N, K, blk, w, L, stream);
      return st;
    }
    cudaGetLastError();   // nothing was launched: take the general path below
  }
  st = cuda_status(xp_launch_hidden(h, h_full, N, xh, (float*)(w + L.part), (float*)(w + L.hc),
                                    L.part_rows, stream));
  if (st != XP_OK) return st;
  if (C == 0) {
    st = cuda_status(xp_launch_init_argmax(h, base, sn, sb, anchor, N, blk, nullptr,
                                           (unsigned long long*)(w + L.in_packed),
                                           (unsigned*)(w + L.in_ticket), stream));
    if (st == XP_OK) st = passes_impl(h, base, sn, sb, xh, am1, N, K, blk, w, L, stream);
    return st;
  }
  int64_t* cand = (int64_t*)(w + L.cand);
  void* base_c = w + L.base_c;
  // the candidates' w2 rows are copied out once per step only while they take less room
  // than w2 itself; beyond that every pass reads them by id from w2, which then stays
  // resident in L2, instead of streaming the larger copy from HBM
  void* w2c = (int64_t)N * (h->B - 1) * C <= (int64_t)h->V ? (void*)(w + L.w2c) : nullptr;
  st = cuda_status(
      xp_launch_topc_gather(h, base, sn, sb, N, C, cand, base_c, w2c, blk, anchor, stream));
  for (int k = 0; k < K && st == XP_OK; ++k) {
    st = xp_latent_pass(h, blk, am1, xh, N, lat, stream);
    if (st == XP_OK)
      st = cuda_status(
          xp_launch_topc_readout(h, lat, base_c, cand, w2c, N, C, blk, nullptr, stream));
  }
  return st;
}

xp_status xp_jacobi_passes(const xp_head* h, const void* base, int64_t sn, int64_t sb,
                           const float* xh, const int64_t* am1, int N, int K, int64_t* blk,
                           void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!valid_base(h, base, sn, sb) || !xh || !am1 || !blk || !ws || N < 0 || K < 0 ||
      !on_head_device(h))
    return XP_EINVAL;
  if (N > h->max_N || ws_bytes < ws_needed(h, N, 0)) return XP_ECAPACITY;
  if (N == 0 || K == 0) return XP_OK;
  const xp_ws_layout L = xp_layout(h->V, h->hidden, h->r, h->H, h->B, h->max_N, h->dtype, N, 0);
  return passes_impl(h, base, sn, sb, xh, am1, N, K, blk, (char*)ws, L, stream);
}

xp_status xp_get_error(const xp_head* h, cudaStream_t stream) {
  if (!h) return XP_ENOTPREPARED;
  if (!on_head_device(h)) return XP_EINVAL;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return XP_ECUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, h->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return XP_ECUDA;
  if (cudaMemset(h->err, 0, sizeof(word)) != cudaSuccess) return XP_ECUDA;
  if (word & XP_ERR_TIMEOUT) return XP_ETIMEOUT;
  if (word & XP_ERR_RANGE) return XP_ERANGE;
  if (word & XP_ERR_BADTOKEN) return XP_EBADTOKEN;
  return XP_OK;
}

xp_status xp_set_pass_mode(xp_head* h, int mode) {
  if (!h) return XP_ENOTPREPARED;
  if (mode != XP_PASSES_AUTO && mode != XP_PASSES_PERSISTENT && mode != XP_PASSES_PER_STAGE)
    return XP_EINVAL;
  h->pass_mode = mode;
  return XP_OK;
}

xp_status xp_set_readout_pairs(xp_head* h, int on) {
  if (!h) return XP_ENOTPREPARED;
  if (on != 0 && on != 1) return XP_EINVAL;
  h->readout_pairs = on;
  return XP_OK;
}

int xp_readout_pairs(const xp_head* h, int N) {
  return h && h->readout_tc && N > 0 && N <= h->max_N && xp_readout_paired(h, N) ? 1 : 0;
}

int xp_passes_persistent(const xp_head* h, const void* base, int64_t sn, int64_t sb, int N) {
  if (!h || N <= 0 || !valid_base(h, base, sn, sb)) return 0;
  const bool persist = h->pass_mode == XP_PASSES_PERSISTENT ||
                       (h->pass_mode == XP_PASSES_AUTO && xp_persist_preferred(h, N));
  return persist && xp_persist_call_ok(h, base, sn, sb, N) ? 1 : 0;
}

xp_status xp_profile_timeline(xp_head* h, void* buf, size_t bytes, int K, size_t* needed) {
  if (!h) return XP_ENOTPREPARED;
  if (K < 0) return XP_EINVAL;
  if (needed) *needed = xp_persist_timeline_bytes(h, K);
  if (buf && bytes < xp_persist_timeline_bytes(h, K)) return XP_ECAPACITY;
  h->timeline = buf;
  h->timeline_bytes = buf ? bytes : 0;
  return XP_OK;
}

const char* xp_readout_kernel_name(const xp_head* h) {
  if (!h) return "";
  return h->readout_tc ? "readout_tc_kernel" : "readout_simt_kernel";
}

}  // extern "C"

// ---------------------------------------------------------------------------
xp_encode_tiled_fn xp_get_encode_tiled() {
  static xp_encode_tiled_fn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (xp_encode_tiled_fn)p;
  }
  return fn;
}

static void decide_paths(xp_head* h) {
  h->readout_tc = 0;
  h->readout_pair_ok = 0;
  h->latent_mma = 0;
  h->hidden_tc = 0;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, h->device);
  const bool blackwell = major == 10 && minor == 3;
  if (!blackwell || h->dtype != XP_BF16) return;
  h->latent_mma = xp_latent_mma_ok(h->r, h->H, h->B, h->dtype) && xp_latent_mma_maps(h);
  h->hidden_tc = xp_hidden_tc_ok(h->r, h->hidden, h->dtype) && xp_hidden_tc_map(h);
  // tcgen05 readout: K = r tiled by 64-wide (128-byte) swizzled chunks, at most 4
  // of them resident; draft rows of one block never straddle a 128-row tile
  if (h->r % 64 == 0 && h->r <= 256 && h->B - 1 <= 128 && xp_get_encode_tiled()) {
    CUtensorMap tm;
    const cuuint64_t dims[2] = {(cuuint64_t)h->r, (cuuint64_t)h->V};
    const cuuint64_t strides[1] = {(cuuint64_t)h->r * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)xp_readout_tc_tile()};
    const cuuint32_t es[2] = {1, 1};
    if (xp_get_encode_tiled()(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, h->w2, dims, strides, box,
                              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      h->tm_w2 = tm;
      h->readout_tc = 1;
      const cuuint32_t half[2] = {64, (cuuint32_t)xp_readout_tc_tile() / 2};
      h->readout_pair_ok =
          xp_get_encode_tiled()(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, h->w2, dims, strides,
                                half, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
      if (h->readout_pair_ok) h->tm_w2_half = tm;
    }
  }
}
