"""The workspace-free readout (xp_readout_argmax_noalloc) for callers that cannot
allocate device memory -- code inside a memory pool it does not own, or a path
where cudaMalloc's synchronisation is not acceptable.  It must give the same
block tokens and winning logits as the regular readout on the same inputs, on
two calls in a row (its fixed scratch array keeps the previous call's state, so
each call has to clear what must start at zero).

Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from parity import LAT_TOL, Dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", [I.workload("batched-decode", V=5000, hidden=256, N=20, K=1),
                                I.workload("tiny-fp32")], ids=["bf16", "fp32"])
def test_noalloc_matches_workspace_readout(wl):
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    for seed in (31, 32):                         # two calls in a row, different latents
        lat = xp.to_device(I.random_lat(wl, seed), wl.dtype)
        ref_blk, got_blk = dev.blk_in.clone(), dev.blk_in.clone()
        ref_win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
        got_win = torch.empty_like(ref_win)
        xp.xp_readout_argmax(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N, ref_blk,
                             ref_win, dev.ws)
        xp.xp_readout_argmax_noalloc(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N,
                                     got_blk, got_win)
        torch.cuda.synchronize()
        assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
        assert np.array_equal(got_blk.cpu().numpy(), ref_blk.cpu().numpy())
        err = (got_win - ref_win).abs().max().item()
        assert err <= LAT_TOL[wl.dtype], err
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
