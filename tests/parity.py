"""Shared helpers of the GPU parity tests: device inputs and the comparison rules.

Tolerances: latents and winning logits within 2e-2 absolute for bf16 heads
and 1e-4 for fp32 heads; block token ids bit-exact, except on draft rows whose
oracle top-2 logit margin is below 2e-2 (reported, and in multi-pass runs the
rest of that block from that slot on is excused, since a flipped near-tie
legitimately changes every later slot's input).
"""
import numpy as np
import torch

from jacobi_speculative_decode_gb300 import xp

LAT_TOL = {"bf16": 2e-2, "f32": 1e-4}
MARGIN = 2e-2


class Dev:
    """Device copies of one workload's inputs plus its head."""

    def __init__(self, d, wl, max_N=None):
        self.wl = wl
        self.head, self.w = xp.head_from_inputs(d, wl, max_N=max_N)
        self.base = xp.to_device(d["base"], wl.dtype) if d["base"] is not None else None
        self.h = xp.to_device(d["h_full"], wl.dtype) if d["h_full"] is not None else None
        self.anchor = torch.from_numpy(d["anchor"]).cuda()
        self.am1 = torch.from_numpy(d["am1"]).cuda()
        self.blk_in = torch.from_numpy(d["blk"]).cuda()
        self.ws = self.head.workspace(max_N or wl.N, wl.topc)
        self.sn, self.sb = (wl.B - 1) * wl.V, wl.V

    def close(self):
        self.head.close()


def check_rows(got_ids, want_ids, margins, what=""):
    """Exact ids except rows with margin < MARGIN; returns the number excused."""
    got_ids = np.asarray(got_ids).reshape(-1)
    want_ids = np.asarray(want_ids).reshape(-1)
    margins = np.asarray(margins).reshape(-1)
    bad = got_ids != want_ids
    excused = bad & (margins < MARGIN)
    unexcused = np.nonzero(bad & ~excused)[0]
    assert unexcused.size == 0, (
        f"{what}: {unexcused.size} rows differ with margin >= {MARGIN}: rows {unexcused[:8]}, "
        f"got {got_ids[unexcused[:8]]} want {want_ids[unexcused[:8]]} "
        f"margins {margins[unexcused[:8]]}")
    return int(excused.sum())


def check_blocks(got_blk, want_blk, margins_per_stage, what=""):
    """Multi-pass rule: block n may differ only from the first slot that had a
    margin below MARGIN in some stage (init or a pass); returns excused blocks."""
    got_blk, want_blk = np.asarray(got_blk), np.asarray(want_blk)
    N, B = want_blk.shape
    excused = 0
    for n in range(N):
        small = [b + 1 for m in margins_per_stage for b in np.nonzero(np.asarray(m)[n] < MARGIN)[0]]
        first = min(small) if small else B
        assert np.array_equal(got_blk[n, :first], want_blk[n, :first]), (
            f"{what}: block {n} differs before slot {first}: got {got_blk[n]} want {want_blk[n]}")
        excused += int(first < B and not np.array_equal(got_blk[n], want_blk[n]))
    return excused


def check_close(got, want, tol, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    err = np.abs(got - want)
    assert err.max(initial=0.0) <= tol, f"{what}: max |err| {err.max():.3g} > {tol} at {np.argmax(err)}"
    return float(err.max(initial=0.0))
