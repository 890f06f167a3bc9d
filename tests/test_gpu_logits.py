"""GPU parity of xp_refine_logits (the unfused readout: logits or bias rows).

The oracle is the fp64 readout, base + lat . w2 (qwen3_xpress page, refine_bias and
the base + bias sum fused_add_argmax_to_blk reduces).  Tolerance: both GPU paths
accumulate the r products and add base in fp32, so an element is within
(r + 1) * 2^-23 * (sum_c |lat_c * w2_vc| + |base_v|) of the exact value (twice the
worst-case bound of r + 1 round-to-nearest fp32 additions).  The argmax of the
logits must also equal xp_readout_argmax's block and winning value bit for bit:
the two kernels run the same MMAs over the same operands and add base the same way.
"""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from oracle import xp_oracle as O
from parity import Dev

pytestmark = pytest.mark.gpu

WORKLOADS = [
    I.workload("tiny-fp32"),
    I.workload("batched-decode", V=5000, hidden=512, N=20, K=4),
    I.workload("single-request", V=4104, hidden=256, B=5, N=40, K=4, base_kind="peaks_half_ties"),
    I.workload("batched-decode", V=4099, hidden=128, r=64, H=128, N=6, K=3),
    I.workload("batched-decode", V=2056, hidden=96, r=96, H=80, B=6, N=7, K=3),
]
IDS = ["tiny-fp32", "bf16-V5000-B16", "bf16-B5", "bf16-oddV-r64", "bf16-r96-plain"]


@pytest.fixture(scope="module", params=list(range(len(WORKLOADS))), ids=IDS)
def case(request):
    wl = WORKLOADS[request.param]
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    yield wl, d, dev, p
    dev.close()


def _bound(lat, w2, base, r):
    mag = np.abs(lat) @ np.abs(w2).T + (np.abs(base) if base is not None else 0.0)
    return (r + 1) * 2.0 ** -23 * mag


def _check(got, lat, w2, base, r, what):
    want = lat @ w2.T + (base if base is not None else 0.0)
    err = np.abs(got.astype(np.float64) - want)
    tol = _bound(lat, w2, base, r)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements beyond the fp32 bound; worst "
                           f"{err.max():.3g} (bound there {tol.reshape(-1)[np.argmax(err)]:.3g})")


@pytest.mark.parametrize("with_base", [True, False], ids=["logits", "bias"])
def test_logits_match_oracle(case, with_base):
    wl, d, dev, p = case
    lat_np = I.random_lat(wl, 21)
    lat = xp.to_device(lat_np, wl.dtype)
    ld = (wl.V + 12 + 3) // 4 * 4                    # padded rows: the padding stays untouched
    out = torch.full((wl.rows, ld), 7.0, dtype=torch.float32, device="cuda")
    xp.xp_refine_logits(dev.head.handle, lat, dev.base if with_base else None, dev.sn, dev.sb,
                        wl.N, out, ld)
    got = out.cpu().numpy()
    assert np.all(got[:, wl.V:] == 7.0)
    base = O.decode(d["base"], wl.dtype).reshape(wl.rows, wl.V) if with_base else None
    _check(got[:, :wl.V], O.decode(lat_np, wl.dtype).reshape(wl.rows, wl.r), p.w2, base, wl.r,
           "logits" if with_base else "bias")


def test_logits_argmax_is_readout_argmax(case):
    wl, d, dev, p = case
    lat = xp.to_device(I.random_lat(wl, 22), wl.dtype)
    out = torch.empty(wl.rows, wl.V, dtype=torch.float32, device="cuda")
    xp.xp_refine_logits(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N, out, wl.V)
    blk = dev.blk_in.clone()
    win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
    xp.xp_readout_argmax(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N, blk, win, dev.ws)
    s = out.cpu().numpy()
    ids = np.argmax(s, axis=1)                        # first occurrence: the lowest id
    assert np.array_equal(blk.cpu().numpy()[:, 1:].reshape(-1), ids)
    assert np.array_equal(win.cpu().numpy(), s[np.arange(wl.rows), ids])


def test_logits_strided_base_and_validation(case):
    wl, d, dev, p = case
    full = torch.zeros(wl.N, wl.B, wl.V, dtype=xp.torch_dtype(wl.dtype), device="cuda")
    full[:, 1:, :] = dev.base
    lat_np = I.random_lat(wl, 23)
    lat = xp.to_device(lat_np, wl.dtype)
    out = torch.empty(wl.rows, wl.V, dtype=torch.float32, device="cuda")
    xp.xp_refine_logits(dev.head.handle, lat, full[:, 1:, :].data_ptr(), wl.B * wl.V, wl.V, wl.N,
                        out, wl.V)
    _check(out.cpu().numpy(), O.decode(lat_np, wl.dtype).reshape(wl.rows, wl.r), p.w2,
           O.decode(d["base"], wl.dtype).reshape(wl.rows, wl.V), wl.r, "strided base")
    with pytest.raises(RuntimeError, match="XP_EINVAL"):
        xp.xp_refine_logits(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N, out, wl.V - 1)
    with pytest.raises(RuntimeError, match="XP_EINVAL"):
        xp.xp_refine_logits(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N, None, wl.V)
    with pytest.raises(RuntimeError, match="XP_ECAPACITY"):
        xp.xp_refine_logits(dev.head.handle, lat, dev.base, dev.sn, dev.sb, wl.N + 1, out, wl.V)
    xp.xp_refine_logits(dev.head.handle, lat, dev.base, dev.sn, dev.sb, 0, out, wl.V)   # no-op


def test_logits_full_size_all_rows():
    # batched-decode at full size, in the launch the bench times: every row and every
    # vocabulary id against the oracle (in row chunks), then repeated launches must give
    # the same bits (the kernel has no atomics: any difference is a race on its rings)
    wl = I.workload("batched-decode")
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    lat_np = I.random_lat(wl, 24)
    lat_d = xp.to_device(lat_np, wl.dtype)
    out = torch.empty(wl.rows, wl.V, dtype=torch.float32, device="cuda")
    xp.xp_refine_logits(dev.head.handle, lat_d, dev.base, dev.sn, dev.sb, wl.N, out, wl.V)
    got = out.cpu().numpy()
    lat = O.decode(lat_np, wl.dtype).reshape(wl.rows, wl.r)
    base = O.decode(d["base"], wl.dtype).reshape(wl.rows, wl.V)
    for r0 in range(0, wl.rows, 48):
        sl = slice(r0, r0 + 48)
        _check(got[sl], lat[sl], p.w2, base[sl], wl.r, f"full-size logits rows {r0}+")
    # the argmax kernel (clusters, its own ring depths) against the same logits, bit for bit
    blk = dev.blk_in.clone()
    win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
    xp.xp_readout_argmax(dev.head.handle, lat_d, dev.base, dev.sn, dev.sb, wl.N, blk, win, dev.ws)
    ids = np.argmax(got, axis=1)
    assert np.array_equal(blk.cpu().numpy()[:, 1:].reshape(-1), ids)
    assert np.array_equal(win.cpu().numpy(), got[np.arange(wl.rows), ids])
    again = torch.empty_like(out)
    for _ in range(8):
        xp.xp_refine_logits(dev.head.handle, lat_d, dev.base, dev.sn, dev.sb, wl.N, again, wl.V)
        assert torch.equal(again, out)
    dev.close()
