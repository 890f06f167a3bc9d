"""The persistent multi-pass refinement (all K passes in one cooperative launch).

xp_jacobi_refine can take it for bf16 heads with r = 256, H = 512 and B <= 16; these
tests force it (XP_PASSES_PERSISTENT) on every shape, including those the automatic
choice leaves to the per-stage launches (one row tile; several latent rounds).  It must
reproduce the oracle's blocks under the multi-pass rule (a block may differ only from
the first slot whose oracle top-2 margin fell below 2e-2), leave its counters and
argmax words clean for the next call (so repeated calls on one workspace agree bit for
bit), and, on a workspace that was never zeroed, stop at once with XP_ETIMEOUT instead
of waiting on counters that will never be right.
"""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from oracle import xp_oracle as O
from parity import Dev, check_blocks

pytestmark = pytest.mark.gpu

SHAPES = [
    # latent groups of 2 blocks, 3 row tiles (the last one ragged), 27 vocabulary tiles
    I.workload("batched-decode", V=5000, hidden=256, N=20, K=6),
    # B = 5: groups of 6 blocks, 30 blocks per row tile, a ragged last group
    I.workload("single-request", V=4104, hidden=256, B=5, N=40, K=4, base_kind="peaks_half_ties"),
    # B = 8 with one block: one latent group, one row tile over every SM
    I.workload("single-request", V=6000, hidden=256, K=7),
    # more groups than teams: every team runs several latent rounds per pass
    I.workload("batched-decode", V=3000, hidden=128, N=300, K=3),
    # B = 2: one draft slot, sixteen blocks per latent group
    I.workload("batched-decode", V=4000, hidden=128, B=2, N=50, K=2),
]
IDS = ["B16-N20", "B5-N40", "B8-N1", "B16-N300-rounds", "B2-N50"]


def _persistent_dev(d, wl):
    dev = Dev(d, wl)
    xp.xp_set_pass_mode(dev.head.handle, xp.XP_PASSES_PERSISTENT)
    assert xp.xp_passes_persistent(dev.head.handle, dev.base, dev.sn, dev.sb, wl.N)
    return dev


def _refine(dev, wl, ws=None):
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, wl.K, 0, blk, dev.ws if ws is None else ws)
    return blk


@pytest.mark.parametrize("wl", SHAPES, ids=IDS)
def test_persistent_refine_matches_oracle_and_repeats(wl):
    d = I.make_inputs(wl)
    dev = _persistent_dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    first = _refine(dev, wl)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want, margins = O.jacobi_refine(O.decode(d["base"], wl.dtype), O.decode(d["h_full"], wl.dtype),
                                    d["anchor"], d["am1"], wl.K, p)
    check_blocks(first.cpu().numpy(), want, margins, f"persistent {wl.N}x{wl.B}")
    # the same workspace twice more: counters and argmax words were left at zero
    for _ in range(2):
        again = _refine(dev, wl)
        assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
        assert torch.equal(again, first)
    dev.close()


def test_unzeroed_workspace_fails_fast_then_recovers():
    wl = SHAPES[0]
    d = I.make_inputs(wl)
    dev = _persistent_dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    dirty = torch.full_like(dev.ws, 1)          # every counter and flag word nonzero
    _refine(dev, wl, dirty)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_ETIMEOUT
    xp.xp_workspace_init(dirty)
    blk = _refine(dev, wl, dirty)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want, margins = O.jacobi_refine(O.decode(d["base"], wl.dtype), O.decode(d["h_full"], wl.dtype),
                                    d["anchor"], d["am1"], wl.K, p)
    check_blocks(blk.cpu().numpy(), want, margins, "after re-zeroing")
    dev.close()


@pytest.mark.parametrize("wl", SHAPES[:2], ids=IDS[:2])
def test_passes_entry_point_equals_the_whole_step(wl):
    # xp_hidden_cache + xp_init_argmax + xp_jacobi_passes runs the same kernels on the same
    # data as xp_jacobi_refine: the same block bit for bit (and the oracle's, by the rule above)
    d = I.make_inputs(wl)
    dev = _persistent_dev(d, wl)
    whole = _refine(dev, wl)
    xh = torch.empty(wl.N, wl.B, wl.r, dtype=torch.float32, device="cuda")
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_hidden_cache(dev.head.handle, dev.h, wl.N, xh, dev.ws)
    xp.xp_init_argmax(dev.head.handle, dev.base, dev.sn, dev.sb, dev.anchor, wl.N, blk, None,
                      dev.ws)
    xp.xp_jacobi_passes(dev.head.handle, dev.base, dev.sn, dev.sb, xh, dev.am1, wl.N, wl.K, blk,
                        dev.ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    assert torch.equal(blk, whole)
    dev.close()


def test_pass_modes_agree_with_the_oracle():
    # the same inputs through the persistent launch and through one launch per stage
    wl = SHAPES[0]
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    want, margins = O.jacobi_refine(O.decode(d["base"], wl.dtype), O.decode(d["h_full"], wl.dtype),
                                    d["anchor"], d["am1"], wl.K, p)
    for mode, persistent in ((xp.XP_PASSES_PERSISTENT, True), (xp.XP_PASSES_PER_STAGE, False)):
        xp.xp_set_pass_mode(dev.head.handle, mode)
        assert xp.xp_passes_persistent(dev.head.handle, dev.base, dev.sn, dev.sb, wl.N) == persistent
        blk = _refine(dev, wl)
        assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
        check_blocks(blk.cpu().numpy(), want, margins, f"mode {mode}")
    with pytest.raises(xp.XPError) as e:
        xp.xp_set_pass_mode(dev.head.handle, 7)
    assert e.value.code == xp.XP_EINVAL
    dev.close()
