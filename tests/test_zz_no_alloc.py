"""The workspace-free readout (xp_readout_argmax_noalloc) for callers that cannot
allocate device memory -- code inside a memory pool it does not own, or a path
where cudaMalloc's synchronisation is not acceptable.

On two calls in a row with different latents it must give the block tokens and
winning logits of the fp64 oracle (under the same rules as every readout test:
ids exact except near-tie rows, winning logits within the dtype's tolerance) and
agree with the regular readout on the same inputs.  Its fixed scratch array keeps
the previous call's state, so each call has to clear what must start at zero; a
call after a kernel that gave up on a bounded wait must still be correct.

Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from oracle import xp_oracle as O
from parity import LAT_TOL, Dev, check_close, check_rows

pytestmark = pytest.mark.gpu

WORKLOADS = [I.workload("batched-decode", V=5000, hidden=256, N=20, K=1), I.workload("tiny-fp32")]


def _against_oracle(wl, d, p, lat_np, blk, win, what):
    s = O.readout(O.decode(lat_np, wl.dtype), p.w2, O.decode(d["base"], wl.dtype))
    ids, vals, margin = O.argmax_lowest(s)
    got = blk.cpu().numpy()
    assert np.array_equal(got[:, 0], d["blk"][:, 0]), what        # slot 0 untouched
    check_rows(got[:, 1:], ids, margin, what)
    same = got[:, 1:].reshape(-1) == ids.reshape(-1)
    check_close(win.cpu().numpy()[same], vals.reshape(-1)[same], LAT_TOL[wl.dtype], what)


@pytest.mark.parametrize("wl", WORKLOADS, ids=["bf16", "fp32"])
def test_noalloc_matches_oracle_and_workspace_readout(wl):
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    for seed in (31, 32):                         # two calls in a row, different latents
        lat_np = I.random_lat(wl, seed)
        lat = xp.to_device(lat_np, wl.dtype)
        ref_blk, got_blk = dev.blk_in.clone(), dev.blk_in.clone()
        ref_win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
        got_win = torch.empty_like(ref_win)
        xp.xp_readout_argmax(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N, ref_blk,
                             ref_win, dev.ws)
        xp.xp_readout_argmax_noalloc(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N,
                                     got_blk, got_win)
        torch.cuda.synchronize()
        assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
        _against_oracle(wl, d, p, lat_np, got_blk, got_win, f"noalloc call seed {seed}")
        assert np.array_equal(got_blk.cpu().numpy(), ref_blk.cpu().numpy())
        err = (got_win - ref_win).abs().max().item()
        assert err <= LAT_TOL[wl.dtype], err
    dev.close()


def test_noalloc_after_a_timed_out_wait():
    wl = WORKLOADS[0]
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    xp.xp_selftest_wait_timeout(dev.head.handle)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_ETIMEOUT
    lat_np = I.random_lat(wl, 33)
    blk = dev.blk_in.clone()
    win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
    xp.xp_readout_argmax_noalloc(dev.head.handle, xp.to_device(lat_np, wl.dtype), dev.base,
                                 dev.sn, dev.sb, wl.N, blk, win)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    _against_oracle(wl, d, p, lat_np, blk, win, "noalloc after a timeout")
    dev.close()


def test_noalloc_rejects_more_rows_than_its_scratch():
    wl = I.workload("batched-decode", V=512, hidden=64, N=300, K=1)   # 4500 draft rows
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    lat = torch.zeros(wl.N, wl.B - 1, wl.r, dtype=torch.bfloat16, device="cuda")
    blk = dev.blk_in.clone()
    with pytest.raises(xp.XPError) as e:
        xp.xp_readout_argmax_noalloc(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N, blk,
                                     None)
    assert e.value.code == xp.XP_ECAPACITY
    dev.close()
