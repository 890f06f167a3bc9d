"""Degenerate cases of the refinement and a property that holds at any size.

- K = 0: the block is the init alone (anchor, then the base argmax of every draft row).
- B = 2: one draft slot per block.
- Fixed point (qwen3_xpress page, jacobi_refine_greedy: a settled prefix stays settled):
  slot b's latent reads only slots < b through the causal mixer, so after pass k the
  slots 1..k no longer change, and after B-1 passes the block is a fixed point.  The
  GPU's own arithmetic has the same structure (the stored mixer is zero above the
  diagonal), so one more pass must leave blk unchanged bit for bit, at full size too.
"""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from oracle import xp_oracle as O
from parity import Dev, check_blocks

pytestmark = pytest.mark.gpu


def _refine(dev, wl, K, topc=0):
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, K, topc, blk, dev.ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    return blk.cpu().numpy()


def test_zero_passes_is_the_init():
    wl = I.workload("batched-decode", V=5000, hidden=512, N=20, K=4)
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    got = _refine(dev, wl, 0)
    assert np.array_equal(got, O.init_blk(O.decode(d["base"], wl.dtype), d["anchor"]))
    dev.close()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_one_draft_slot(dtype):
    wl = I.workload("batched-decode", V=4096, hidden=256, r=64, H=128, B=2, N=9, K=2,
                    dtype=dtype)
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    got = _refine(dev, wl, wl.K)
    want, margins = O.jacobi_refine(O.decode(d["base"], wl.dtype), O.decode(d["h_full"], wl.dtype),
                                    d["anchor"], d["am1"], wl.K, p)
    check_blocks(got, want, margins, "B=2")
    dev.close()


@pytest.mark.parametrize("name", ["batched-decode", "single-request"])
def test_one_more_pass_changes_nothing(name):
    wl = I.workload(name)
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    settled = _refine(dev, wl, wl.B - 1)
    assert np.array_equal(_refine(dev, wl, wl.B), settled)
    assert np.array_equal(_refine(dev, wl, wl.B + 3), settled)
    dev.close()
