"""Plain, slow, fp64 CPU oracle of one XPress Jacobi refinement pass.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this module.  It shares
no code with the CUDA library and imports nothing from it.

Every input is first widened exactly from its storage type (bf16 bit patterns
or float32) to float64; all arithmetic is float64 with no intermediate
rounding.  Library primitives (matmul, einsum, argmax, sort) serve as single
steps; nothing is blocked, fused or reordered beyond the definitions below.

Sources ("qwen3_xpress page" = the vLLM API page of
``vllm.model_executor.models.qwen3_xpress``; "xpress kernels page" = the vLLM
API page of ``vllm.v1.worker.gpu.spec_decode.xpress.kernels``):

* fold            -- qwen3_xpress page, ``XPressRefinerHead.fold_from_raw_``
* hidden cache    -- qwen3_xpress page, ``XPressRefinerHead.hidden_cache`` and
                     the ``xh = hcache @ whc_t`` hoist in ``jacobi_refine_greedy``
* latent          -- qwen3_xpress page, ``XPressRefinerHead._refine_latent``;
                     xpress kernels page, ``_xpress_latent_kernel`` docstring
* readout         -- qwen3_xpress page, ``refine_bias`` (w2 of the latent);
                     xpress kernels page, module docstring ("readout")
* argmax to blk   -- xpress kernels page, ``fused_add_argmax_to_blk``
* Jacobi loop     -- qwen3_xpress page, ``XPressRefinerHead.jacobi_refine_greedy``
* top-C           -- qwen3_xpress page, the ``if self.topc`` branch of
                     ``jacobi_refine_greedy``; xpress kernels page,
                     ``_xpress_topc_argmax_to_blk_kernel`` docstring

Readings where the pages are silent (also listed in the design notes):
* argmax ties go to the lowest vocabulary id (first occurrence), everywhere;
* top-C keeps the C largest base values, ties at the boundary to the lower
  id, and stores the candidates in ascending id order;
* the folded mixer is rounded once to the storage type and that stored tensor
  is the parameter (both sides fold the same raw tensor);
* the mean feeding down_g runs over all B slots of the block, slot 0 included.

Parity status: every function here is pinned by tests that do not call back
into it (closed forms, special cases, brute force on tiny inputs, invariants).
"""
from __future__ import annotations

import math
from typing import NamedTuple

import numpy as np


# ---------------------------------------------------------------------------
# storage <-> float64
# ---------------------------------------------------------------------------

def decode(a, dtype: str) -> np.ndarray:
    """Exact widening of stored values to float64 (bf16 bit patterns or float32)."""
    if dtype == "bf16":
        u = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return u.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 once, to nearest-even, into the storage type.

    bf16: the 53-bit significand is cut to 8 bits directly from float64 (no
    detour through float32, which could round twice).  Values are assumed
    finite and inside the normal bf16 range (or exactly zero).
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype != "bf16":
        raise ValueError(dtype)
    u = x.view(np.uint64)
    drop = np.uint64(45)                       # 52 - 7 fraction bits dropped
    lsb = (u >> drop) & np.uint64(1)
    bias = (np.uint64(1) << np.uint64(44)) - np.uint64(1) + lsb
    kept = ((u + bias) >> drop) << drop
    y = kept.view(np.float64)                  # exactly representable in bf16
    return (y.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------
# parameters
# ---------------------------------------------------------------------------

class Params(NamedTuple):
    """Head weights in float64, torch layout ([out, in] for linear maps)."""
    w1: np.ndarray        # [V, r]   token embedding
    down_h: np.ndarray    # [r, hidden]
    down_g: np.ndarray    # [r, hidden]
    in_proj: np.ndarray   # [r, 3r]  columns: [down_h part | down_g part | embedding part]
    mix: np.ndarray       # [r, B, B] folded mixer, index [channel, out slot, in slot]
    w_gate: np.ndarray    # [H, r]
    w_up: np.ndarray      # [H, r]
    w_down: np.ndarray    # [r, H]
    w2: np.ndarray        # [V, r]   readout


def fold(raw: np.ndarray) -> np.ndarray:
    """Folded mixer ``raw * tril + I`` per channel (fold_from_raw_), float64."""
    B = raw.shape[-1]
    tril = np.tril(np.ones((B, B)))
    return raw * tril + np.eye(B)


def fold_stored(raw_stored, dtype: str) -> np.ndarray:
    """The folded mixer as the head stores it: fold in float64, round once."""
    return encode(fold(decode(raw_stored, dtype)), dtype)


def params_from_inputs(inp: dict, dtype: str) -> Params:
    """Widen generated storage arrays; the mixer is folded here from the raw draw."""
    g = lambda k: decode(inp[k], dtype)
    mix = decode(fold_stored(inp["raw_mix"], dtype), dtype)
    return Params(g("w1"), g("down_h"), g("down_g"), g("in_proj"), mix,
                  g("w_gate"), g("w_up"), g("w_down"), g("w2"))


# ---------------------------------------------------------------------------
# one pass, stage by stage
# ---------------------------------------------------------------------------

def hidden_cache(h: np.ndarray, down_h: np.ndarray, down_g: np.ndarray) -> np.ndarray:
    """hcache[n,b] = [down_h h[n,b] ; down_g mean_b' h[n,b']]  -> [N, B, 2r]."""
    g = h.mean(axis=1, keepdims=True)
    g = np.broadcast_to(g, h.shape)
    return np.concatenate([h @ down_h.T, g @ down_g.T], axis=-1)


def xh_from_cache(hcache: np.ndarray, in_proj: np.ndarray) -> np.ndarray:
    """The pass-invariant half of in_proj: xh = hcache @ in_proj[:, :2r]^T -> [N, B, r]."""
    r = in_proj.shape[0]
    return hcache @ in_proj[:, : 2 * r].T


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def prev_ids(blk: np.ndarray, am1: np.ndarray) -> np.ndarray:
    """Token each slot embeds: slot 0 reads am1[n], slot b >= 1 reads blk[n, b-1]."""
    prev = np.empty_like(blk)
    prev[:, 0] = am1
    prev[:, 1:] = blk[:, :-1]
    return prev


def latent_all_slots(blk, am1, xh, p: Params) -> np.ndarray:
    """Latent of every slot 0..B-1 (``_refine_latent`` with the hoisted xh) -> [N, B, r]."""
    r = xh.shape[-1]
    e = p.w1[prev_ids(blk, am1)]                      # [N, B, r] embedding gather
    x = xh + e @ p.in_proj[:, 2 * r:].T               # in_proj over [hcache ; embedding]
    # per-channel mix: u[n, b, c] = sum_j mix[c, b, j] * x[n, j, c]  (bmm over channels)
    u = np.einsum("cbj,njc->nbc", p.mix, x)
    act = silu(u @ p.w_gate.T) * (u @ p.w_up.T)       # SwiGLU, [N, B, H]
    return u + act @ p.w_down.T                       # residual around the MLP


def latent(blk, am1, xh, p: Params) -> np.ndarray:
    """Latent read out for slots 1..B-1 -> [N, B-1, r] (slot 0 is the anchor)."""
    return latent_all_slots(blk, am1, xh, p)[:, 1:, :]


def readout(lat: np.ndarray, w2: np.ndarray, base: np.ndarray) -> np.ndarray:
    """logits[n, b, v] = base[n, b, v] + lat[n, b, :] . w2[v, :]  -> [N, B-1, V]."""
    return base + lat @ w2.T


def argmax_lowest(s: np.ndarray):
    """Argmax over the last axis with ties to the lowest index.

    Returns (ids, winning value, top-2 margin); the margin is the winner minus
    the largest value at any other index (0 for an exact tie).
    """
    ids = np.argmax(s, axis=-1)
    win = np.take_along_axis(s, ids[..., None], axis=-1)[..., 0]
    if s.shape[-1] < 2:
        return ids, win, np.full(ids.shape, np.inf)
    top2 = np.partition(s, -2, axis=-1)[..., -2]
    return ids, win, win - top2


def init_blk(base: np.ndarray, anchor: np.ndarray) -> np.ndarray:
    """blk[:, 0] = anchor; blk[:, 1:] = argmax of the base rows."""
    N, Bm1, _ = base.shape
    blk = np.empty((N, Bm1 + 1), np.int64)
    blk[:, 0] = anchor
    blk[:, 1:] = argmax_lowest(base)[0]
    return blk


def full_pass(blk, am1, xh, base, p: Params):
    """One synchronous Jacobi pass with full-vocabulary scoring.

    Every slot's latent is computed from the pre-pass blk; then slots 1..B-1
    are replaced by the argmax.  Returns (new blk, lat, win, margin).
    """
    lat = latent(blk, am1, xh, p)
    ids, win, margin = argmax_lowest(readout(lat, p.w2, base))
    out = blk.copy()
    out[:, 1:] = ids
    return out, lat, win, margin


def jacobi_refine(base, h, anchor, am1, K: int, p: Params):
    """jacobi_refine_greedy, full vocabulary: hidden cache, init argmax, K passes.

    Returns (blk [N, B], list of per-stage top-2 margins [init, pass 1, ..., pass K]).
    """
    xh = xh_from_cache(hidden_cache(h, p.down_h, p.down_g), p.in_proj)
    blk = init_blk(base, anchor)
    margins = [argmax_lowest(base)[2]]
    for _ in range(K):
        blk, _, _, m = full_pass(blk, am1, xh, base, p)
        margins.append(m)
    return blk, margins


# ---------------------------------------------------------------------------
# top-C
# ---------------------------------------------------------------------------

def topc_select(base: np.ndarray, C: int):
    """Per row: the C largest base values (ties to the lower id), ids ascending.

    base [N, B-1, V] -> cand [N, B-1, C] int64, base_c [N, B-1, C] float64.
    """
    N, Bm1, V = base.shape
    C = min(C, V)
    cand = np.empty((N, Bm1, C), np.int64)
    ids = np.arange(V)
    for n in range(N):
        for b in range(Bm1):
            order = np.lexsort((ids, -base[n, b]))   # value descending, id ascending
            cand[n, b] = np.sort(order[:C])
    base_c = np.take_along_axis(base, cand, axis=-1)
    return cand, base_c


def topc_scores(lat, w2, cand, base_c) -> np.ndarray:
    """s_c[n, b, k] = base_c[n, b, k] + w2[cand[n, b, k]] . lat[n, b]."""
    return base_c + np.einsum("nbkc,nbc->nbk", w2[cand], lat)


def topc_argmax(s_c: np.ndarray, cand: np.ndarray):
    """Winner among the candidates: highest score, ties to the lowest vocabulary id.

    Returns (vocab ids, winning score, top-2 margin over the candidates).
    """
    best = s_c.max(axis=-1, keepdims=True)
    big = np.iinfo(np.int64).max
    ids = np.where(s_c == best, cand, big).min(axis=-1)
    win = best[..., 0]
    if s_c.shape[-1] < 2:
        return ids, win, np.full(ids.shape, np.inf)
    top2 = np.partition(s_c, -2, axis=-1)[..., -2]
    return ids, win, win - top2


def topc_pass(blk, am1, xh, cand, base_c, p: Params):
    """One Jacobi pass scored on the candidates only.  Returns (blk, lat, win, margin)."""
    lat = latent(blk, am1, xh, p)
    ids, win, margin = topc_argmax(topc_scores(lat, p.w2, cand, base_c), cand)
    out = blk.copy()
    out[:, 1:] = ids
    return out, lat, win, margin


def jacobi_refine_topc(base, h, anchor, am1, K: int, C: int, p: Params):
    """jacobi_refine_greedy with top-C scoring: candidates gathered once per step."""
    xh = xh_from_cache(hidden_cache(h, p.down_h, p.down_g), p.in_proj)
    blk = init_blk(base, anchor)
    margins = [argmax_lowest(base)[2]]
    cand, base_c = topc_select(base, C)
    for _ in range(K):
        blk, _, _, m = topc_pass(blk, am1, xh, cand, base_c, p)
        margins.append(m)
    return blk, margins


# ---------------------------------------------------------------------------
# brute force: the refiner's own sequential greedy decode (tiny inputs only)
# ---------------------------------------------------------------------------

def sequential_greedy(base, h, anchor, am1, p: Params) -> np.ndarray:
    """Slot-by-slot greedy decode in plain Python loops.

    t[0] = anchor; for s = 1..B-1 the latent of slot s is built from am1 and
    t[0..s-1] alone, and t[s] = argmax_v(base[s-1, v] + w2[v] . lat_s), ties to
    the lowest id.  Written independently of the vectorised pass above (lists
    and scalar loops; the mixer sum runs over j <= s only).
    """
    N, B, hid = h.shape
    r = p.in_proj.shape[0]
    H = p.w_gate.shape[0]
    V = p.w2.shape[0]
    W1, Dh, Dg, Win = p.w1.tolist(), p.down_h.tolist(), p.down_g.tolist(), p.in_proj.tolist()
    Mix, Wg, Wu, Wd, W2 = p.mix.tolist(), p.w_gate.tolist(), p.w_up.tolist(), p.w_down.tolist(), p.w2.tolist()
    out = np.empty((N, B), np.int64)
    for n in range(N):
        hn = h[n].tolist()
        bn = base[n].tolist()
        # hidden cache of this block, slot by slot
        g = [sum(hn[b][k] for b in range(B)) / B for k in range(hid)]
        hg = [sum(Dg[c][k] * g[k] for k in range(hid)) for c in range(r)]
        xh = []
        for b in range(B):
            hh = [sum(Dh[c][k] * hn[b][k] for k in range(hid)) for c in range(r)]
            cache = hh + hg
            xh.append([sum(Win[c][k] * cache[k] for k in range(2 * r)) for c in range(r)])
        toks = [int(anchor[n])]
        for s in range(1, B):
            prev = [int(am1[n])] + toks[:s]          # slots 0..s read am1, t0..t(s-1)
            x = []
            for j in range(s + 1):
                emb = W1[prev[j]]
                x.append([xh[j][c] + sum(Win[c][2 * r + k] * emb[k] for k in range(r))
                          for c in range(r)])
            u = [sum(Mix[c][s][j] * x[j][c] for j in range(s + 1)) for c in range(r)]
            act = []
            for q in range(H):
                gz = sum(Wg[q][c] * u[c] for c in range(r))
                uz = sum(Wu[q][c] * u[c] for c in range(r))
                act.append(gz / (1.0 + math.exp(-gz)) * uz)
            lat = [u[c] + sum(Wd[c][q] * act[q] for q in range(H)) for c in range(r)]
            best_v, best = -1, -math.inf
            row = bn[s - 1]
            for v in range(V):
                wv = W2[v]
                val = row[v] + sum(wv[c] * lat[c] for c in range(r))
                if val > best:
                    best, best_v = val, v
            toks.append(best_v)
        out[n] = toks
    return out
