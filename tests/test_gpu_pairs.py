"""The 2-CTA readout (two neighbouring row tiles of one vocabulary segment share every
tcgen05 MMA; each CTA stages half of each w2 tile) against the fp64 oracle and against
the one-CTA-per-row-tile readout on the same inputs.

Shapes: even numbers of row tiles (paired) with a ragged last row tile, a ragged
vocabulary tail that leaves the odd CTA's half of the last tile entirely past V, one to
four 64-wide k-chunks (r = 64..256), B = 2 (128 one-row blocks per tile) and B = 5; and an
odd number of row tiles, which stays unpaired.
"""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from oracle import xp_oracle as O
from parity import LAT_TOL, Dev, check_blocks, check_close, check_rows

pytestmark = pytest.mark.gpu

PAIRED = [
    # 4 row tiles of 8 blocks, the last one with 4; V = 26 x 192 + 8: the last tile's upper
    # half (the odd CTA's) lies wholly past V
    I.workload("batched-decode", V=5000, hidden=256, N=28, K=3),
    # B = 5: 32 blocks per row tile, 2 row tiles (the second ragged)
    I.workload("single-request", V=4104, hidden=256, B=5, N=40, K=3, base_kind="peaks_half_ties"),
    # B = 2: 128 one-row blocks per row tile
    I.workload("batched-decode", V=3072, hidden=128, B=2, N=256, K=2),
    # r = 128 and r = 64: two and one k-chunks per tile
    I.workload("batched-decode", V=4096, hidden=128, r=128, H=128, N=16, K=2),
    I.workload("batched-decode", V=4096, hidden=128, r=64, H=128, N=16, K=2),
]
PAIRED_IDS = ["B16-N28-tail", "B5-N40", "B2-N256", "r128", "r64"]


def _readout(dev, wl, lat):
    blk = dev.blk_in.clone()
    win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
    xp.xp_readout_argmax(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N, blk, win, dev.ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    return blk, win


@pytest.mark.parametrize("wl", PAIRED, ids=PAIRED_IDS)
def test_paired_readout_matches_oracle_and_single(wl):
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    assert not xp.xp_readout_pairs(dev.head.handle, wl.N)      # off by default
    xp.xp_set_readout_pairs(dev.head.handle, True)
    assert xp.xp_readout_pairs(dev.head.handle, wl.N)
    for seed in (41, 42):
        lat_np = I.random_lat(wl, seed)
        lat = xp.to_device(lat_np, wl.dtype)
        xp.xp_set_readout_pairs(dev.head.handle, True)
        blk2, win2 = _readout(dev, wl, lat)
        xp.xp_set_readout_pairs(dev.head.handle, False)
        assert not xp.xp_readout_pairs(dev.head.handle, wl.N)
        blk1, win1 = _readout(dev, wl, lat)
        xp.xp_set_readout_pairs(dev.head.handle, True)
        s = O.readout(O.decode(lat_np, wl.dtype), p.w2, O.decode(d["base"], wl.dtype))
        ids, vals, margin = O.argmax_lowest(s)
        got = blk2.cpu().numpy()
        assert np.array_equal(got[:, 0], d["blk"][:, 0])
        check_rows(got[:, 1:], ids, margin, f"paired seed {seed}")
        same = got[:, 1:].reshape(-1) == ids.reshape(-1)
        check_close(win2.cpu().numpy()[same], vals.reshape(-1)[same], LAT_TOL[wl.dtype], "win")
        # the same dot products in the same k order as one CTA per row tile
        assert torch.equal(blk2, blk1)
        assert (win2 - win1).abs().max().item() <= 1e-4
    dev.close()


def test_odd_row_tiles_stay_unpaired():
    wl = I.workload("batched-decode", V=5000, hidden=256, N=20, K=2)     # 3 row tiles
    d = I.make_inputs(wl)
    dev = Dev(d, wl, max_N=32)
    xp.xp_set_readout_pairs(dev.head.handle, True)
    assert not xp.xp_readout_pairs(dev.head.handle, wl.N)
    assert xp.xp_readout_pairs(dev.head.handle, 32)                    # 4 row tiles of 8 blocks
    p = O.params_from_inputs(d, wl.dtype)
    lat_np = I.random_lat(wl, 43)
    blk, _ = _readout(dev, wl, xp.to_device(lat_np, wl.dtype))
    ids, _, margin = O.argmax_lowest(O.readout(O.decode(lat_np, wl.dtype), p.w2,
                                               O.decode(d["base"], wl.dtype)))
    check_rows(blk.cpu().numpy()[:, 1:], ids, margin, "unpaired")
    dev.close()


@pytest.mark.parametrize("wl", PAIRED[:2], ids=PAIRED_IDS[:2])
def test_per_stage_refine_with_pairs(wl):
    # every pass's readout paired, chained with the latent launches as in a real step
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    xp.xp_set_pass_mode(dev.head.handle, xp.XP_PASSES_PER_STAGE)
    xp.xp_set_readout_pairs(dev.head.handle, True)
    p = O.params_from_inputs(d, wl.dtype)
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, wl.K, 0, blk, dev.ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want, margins = O.jacobi_refine(O.decode(d["base"], wl.dtype), O.decode(d["h_full"], wl.dtype),
                                    d["anchor"], d["am1"], wl.K, p)
    check_blocks(blk.cpu().numpy(), want, margins, "per-stage paired")
    dev.close()


def test_pair_setting_validation():
    wl = PAIRED[0]
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    assert xp.lib().xp_set_readout_pairs(dev.head.handle, 7) == xp.XP_EINVAL
    assert xp.lib().xp_readout_pairs(dev.head.handle, 0) == 0
    assert xp.lib().xp_readout_pairs(dev.head.handle, wl.N + 10_000) == 0    # above max_N
    dev.close()
