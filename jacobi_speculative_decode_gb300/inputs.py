"""Seeded synthetic inputs for the XPress Jacobi refinement pass.

This module only draws numbers.  It holds none of the method's arithmetic (no
fold, no projection, no mixer, no readout, no argmax): the CUDA path and the
CPU oracle both receive exactly the arrays built here, as raw storage (bf16 as
uint16 bit patterns, fp32 as float32, token ids as int64).

Workloads (shapes and value distributions follow the XPressRefinerHead
constructor on the qwen3_xpress model page: rank r=256, mlp_hidden=512,
topc=512 defaults; vocabulary 151936 for the Qwen3 family):

  tiny-fp32        V=4096   hidden=256  r=32  H=64  B=4  N=2    K=3   fp32
  single-request   V=151936 hidden=4096 r=256 H=512 B=8  N=1    K=7   bf16
  batched-decode   V=151936 hidden=4096 r=256 H=512 B=16 N=32   K=15  bf16
  topc             V=151936 hidden=4096 r=256 H=512 B=16 N=256  K=15  bf16  C=512
  max-batch        V=151936 hidden=5120 r=256 H=512 B=16 N=256  K=15  bf16

Distributions: h ~ N(0,1); every weight ~ N(0, 1/fan_in) with torch's fan_in
(= weight.shape[1]); the raw (unfolded) mixer ~ N(0, 0.1^2); base logits
~ N(0, 3^2) over the N*(B-1) draft rows, with a +8 peak planted per row
("peak_all"), or on the first half of a seeded row permutation plus
near-ties on the next 5% ("peaks_half_ties"), or Zipf-skewed rows for the
top-C workload ("zipf"); anchor, am1 and the per-stage block tokens are
uniform in [0, V).

Draw order (one numpy PCG64 stream seeded 20260 + workload index):
h_full, w1, down_h, down_g, in_proj, raw_mix, w_gate, w_up, w_down, w2, base,
peaks/ties (or the Zipf permutation), anchor, am1, blk.  Normals are drawn as
float32 in chunks, scaled in float32 and rounded to nearest-even bf16.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_CHUNK = 1 << 22  # elements per normal draw


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    V: int
    hidden: int
    r: int
    H: int
    B: int
    N: int
    K: int
    dtype: str          # "bf16" or "f32": storage and compute type of the head
    topc: int = 0       # candidates per row; 0 = full-vocabulary scoring
    base_kind: str = "peak_all"   # "peak_all" | "peaks_half_ties" | "zipf"
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.N * (self.B - 1)


WORKLOADS = {
    "tiny-fp32": Workload("tiny-fp32", 4096, 256, 32, 64, 4, 2, 3, "f32",
                          0, "peak_all", 20260),
    "single-request": Workload("single-request", 151936, 4096, 256, 512, 8, 1, 7,
                               "bf16", 0, "peak_all", 20261),
    "batched-decode": Workload("batched-decode", 151936, 4096, 256, 512, 16, 32, 15,
                               "bf16", 0, "peaks_half_ties", 20262),
    "topc": Workload("topc", 151936, 4096, 256, 512, 16, 256, 15, "bf16", 512,
                     "zipf", 20263),
    "max-batch": Workload("max-batch", 151936, 5120, 256, 512, 16, 256, 15, "bf16",
                          0, "peaks_half_ties", 20264),
}


def workload(name: str, **overrides) -> Workload:
    """A named workload, optionally with some fields replaced (smaller parity sizes)."""
    return dataclasses.replace(WORKLOADS[name], **overrides)


# ---------------------------------------------------------------------------
# storage helpers (bit-level, no method arithmetic)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16, ties to even; returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (generator-side use only)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if dtype == "bf16" else np.ascontiguousarray(x32, np.float32)


def _normal(rng: np.random.Generator, shape, std: float, dtype: str) -> np.ndarray:
    """N(0, std^2) drawn as float32 in chunks, scaled in float32, stored in `dtype`."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16 if dtype == "bf16" else np.float32)
    s = np.float32(std)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        z = rng.standard_normal(hi - lo, dtype=np.float32) * s
        out[lo:hi] = _store(z, dtype)
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# base logits
# ---------------------------------------------------------------------------

def _base_gaussian(rng, wl: Workload) -> np.ndarray:
    """[rows, V] ~ N(0, 9) kept in float32 until the peaks are planted."""
    rows, V = wl.rows, wl.V
    out = np.empty((rows, V), np.float32)
    flat = out.reshape(-1)
    for lo in range(0, flat.size, _CHUNK):
        hi = min(flat.size, lo + _CHUNK)
        flat[lo:hi] = rng.standard_normal(hi - lo, dtype=np.float32) * np.float32(3.0)
    return out


def _plant_peaks_all(rng, wl, base32):
    ids = rng.integers(0, wl.V, size=wl.rows)
    base32[np.arange(wl.rows), ids] += np.float32(8.0)
    return _store(base32, wl.dtype), {"peak_rows": np.arange(wl.rows), "peak_ids": ids}


def _plant_peaks_half_ties(rng, wl, base32):
    """Peaks on the first half of a seeded row permutation; near-ties on the next 5%.

    A near-tie row gets two distinct ids v1, v2: base[v1] = bf16(rowmax + 1) and
    base[v2] = bf16(base[v1] - U(0, 0.05)), both set after the row was rounded,
    so the stored margin is either 0 (an exact tie) or one bf16 spacing.
    """
    rows, V = wl.rows, wl.V
    perm = rng.permutation(rows)
    n_peak = rows // 2
    n_tie = max(1, (rows * 5) // 100) if rows >= 2 else 0
    peak_rows = perm[:n_peak]
    tie_rows = perm[n_peak:n_peak + n_tie]
    peak_ids = rng.integers(0, V, size=n_peak)
    base32[peak_rows, peak_ids] += np.float32(8.0)
    stored = _store(base32, wl.dtype)
    v1 = rng.integers(0, V, size=n_tie)
    v2 = (v1 + rng.integers(1, V, size=n_tie)) % V       # distinct from v1
    gap = rng.uniform(0.0, 0.05, size=n_tie).astype(np.float32)
    for i, row in enumerate(tie_rows):
        vals = bf16_bits_to_f32(stored[row]) if wl.dtype == "bf16" else stored[row]
        top = np.float32(vals.max() + np.float32(1.0))
        top_s = _store(np.array([top], np.float32), wl.dtype)[0]
        top_v = bf16_bits_to_f32(np.array([top_s]))[0] if wl.dtype == "bf16" else top_s
        sec_s = _store(np.array([top_v - gap[i]], np.float32), wl.dtype)[0]
        stored[row, v1[i]] = top_s
        stored[row, v2[i]] = sec_s
    return stored, {"peak_rows": peak_rows, "peak_ids": peak_ids,
                    "tie_rows": tie_rows, "tie_ids": np.stack([v1, v2], 1)}


def _base_zipf(rng, wl: Workload):
    """Zipf-skewed rows: base[row, pi(k)] = 3 z_k - alpha ln(k+1), pi(k) = (a k + b) mod V.

    a is coprime to V, so pi is a permutation of the ids.
    alpha starts at 4 and rises by 0.5 until the median top-C softmax mass of
    the first 64 rows is at least 0.9 (the mass does not depend on pi).
    """
    rows, V = wl.rows, wl.V
    C = wl.topc if wl.topc else 512
    logk = np.log(np.arange(1, V + 1, dtype=np.float64)).astype(np.float32)
    z = np.empty((rows, V), np.float32)
    flat = z.reshape(-1)
    for lo in range(0, flat.size, _CHUNK):
        hi = min(flat.size, lo + _CHUNK)
        flat[lo:hi] = rng.standard_normal(hi - lo, dtype=np.float32)
    alpha = 4.0
    sample = z[: min(64, rows)]
    while True:
        vals = _store(np.float32(3.0) * sample - np.float32(alpha) * logk, wl.dtype)
        v = (bf16_bits_to_f32(vals) if wl.dtype == "bf16" else vals).astype(np.float64)
        v = v - v.max(axis=1, keepdims=True)
        e = np.exp(v)
        top = np.sort(e, axis=1)[:, ::-1][:, : min(C, V)].sum(axis=1)
        mass = np.median(top / e.sum(axis=1))
        if mass >= 0.9 or alpha > 64:
            break
        alpha += 0.5
    a = rng.integers(0, max(1, V // 2), size=rows) * 2 + 1
    bad = np.gcd(a, V) != 1
    while bad.any():                      # step to the next odd value coprime to V
        a = np.where(bad, (a + 2) % V, a)
        bad = np.gcd(a, V) != 1
    b = rng.integers(0, V, size=rows)
    out = np.empty((rows, V), np.uint16 if wl.dtype == "bf16" else np.float32)
    k = np.arange(V, dtype=np.int64)
    for row in range(rows):
        vals = _store(np.float32(3.0) * z[row] - np.float32(alpha) * logk, wl.dtype)
        out[row, (a[row] * k + b[row]) % V] = vals
    return out, {"alpha": alpha, "zipf_a": a, "zipf_b": b}


# ---------------------------------------------------------------------------

def make_inputs(wl: Workload, with_base: bool = True, with_hidden: bool = True) -> dict:
    """Draw every input of one workload, in the fixed order.

    Returns a dict of numpy arrays in storage form plus "meta".  `with_base` /
    `with_hidden` = False still advance the stream by the same draws but do not
    keep the arrays (keeps memory down for large stage-only tests).
    """
    rng = np.random.default_rng(wl.seed)
    d = wl.dtype
    r, H, V, B, N, hid = wl.r, wl.H, wl.V, wl.B, wl.N, wl.hidden
    out = {}
    out["h_full"] = _normal(rng, (N, B, hid), 1.0, d)
    out["w1"] = _normal(rng, (V, r), 1.0 / math.sqrt(r), d)
    out["down_h"] = _normal(rng, (r, hid), 1.0 / math.sqrt(hid), d)
    out["down_g"] = _normal(rng, (r, hid), 1.0 / math.sqrt(hid), d)
    out["in_proj"] = _normal(rng, (r, 3 * r), 1.0 / math.sqrt(3 * r), d)
    out["raw_mix"] = _normal(rng, (r, B, B), 0.1, d)
    out["w_gate"] = _normal(rng, (H, r), 1.0 / math.sqrt(r), d)
    out["w_up"] = _normal(rng, (H, r), 1.0 / math.sqrt(r), d)
    out["w_down"] = _normal(rng, (r, H), 1.0 / math.sqrt(H), d)
    out["w2"] = _normal(rng, (V, r), 1.0 / math.sqrt(r), d)
    meta = {"workload": wl}
    if wl.base_kind == "zipf":
        base, extra = _base_zipf(rng, wl)
    else:
        base32 = _base_gaussian(rng, wl)
        if wl.base_kind == "peak_all":
            base, extra = _plant_peaks_all(rng, wl, base32)
        elif wl.base_kind == "peaks_half_ties":
            base, extra = _plant_peaks_half_ties(rng, wl, base32)
        else:
            raise ValueError(wl.base_kind)
        del base32
    meta.update(extra)
    out["base"] = base.reshape(N, B - 1, V) if with_base else None
    out["anchor"] = rng.integers(0, V, size=N, dtype=np.int64)
    out["am1"] = rng.integers(0, V, size=N, dtype=np.int64)
    out["blk"] = rng.integers(0, V, size=(N, B), dtype=np.int64)
    if not with_hidden:
        out["h_full"] = None
    out["meta"] = meta
    return out


def random_lat(wl: Workload, seed: int, scale: float = 1.0) -> np.ndarray:
    """Synthetic latents [N, B-1, r] ~ N(0, scale^2) in storage form, for stage-only tests."""
    rng = np.random.default_rng(seed)
    return _normal(rng, (wl.N, wl.B - 1, wl.r), scale, wl.dtype)


def random_xh(wl: Workload, seed: int) -> np.ndarray:
    """Synthetic pass-invariant hidden projections [N, B, r] ~ N(0, 1), float32."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((wl.N, wl.B, wl.r), dtype=np.float32)
