"""GPU parity at the full workload sizes, in the launch configuration bench.py uses.

The GPU runs the whole batch; the fp64 oracle checks sampled blocks and rows it
can afford (blocks are independent, so a sampled block's oracle run sees exactly
what the GPU saw).  Same tolerances and margin rule as test_gpu_parity.py.
"""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from oracle import xp_oracle as O
from parity import LAT_TOL, Dev, check_blocks, check_close, check_rows

pytestmark = pytest.mark.gpu


def _oracle_jacobi(d, wl, p, blocks, topc=0):
    base = O.decode(d["base"][blocks], wl.dtype)
    h = O.decode(d["h_full"][blocks], wl.dtype)
    if topc:
        return O.jacobi_refine_topc(base, h, d["anchor"][blocks], d["am1"][blocks], wl.K, topc, p)
    return O.jacobi_refine(base, h, d["anchor"][blocks], d["am1"][blocks], wl.K, p)


def _run_jacobi(dev, wl, topc=0, ws=None):
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, wl.K, topc, blk, dev.ws if ws is None else ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    return blk.cpu().numpy()


@pytest.fixture(scope="module")
def single_request():
    wl = I.workload("single-request")
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    yield wl, d, dev, O.params_from_inputs(d, wl.dtype)
    dev.close()


@pytest.fixture(scope="module")
def batched():
    wl = I.workload("batched-decode")
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    yield wl, d, dev, O.params_from_inputs(d, wl.dtype)
    dev.close()


def test_single_request_jacobi(single_request):
    wl, d, dev, p = single_request
    got = _run_jacobi(dev, wl)
    want, margins = _oracle_jacobi(d, wl, p, np.arange(wl.N))
    check_blocks(got, want, margins, "single-request")


def test_batched_readout_all_rows(batched):
    wl, d, dev, p = batched
    lat_np = I.random_lat(wl, 41)
    blk = dev.blk_in.clone()
    win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
    xp.xp_readout_argmax(dev.head.handle, xp.to_device(lat_np, wl.dtype), dev.base, dev.sn,
                         dev.sb, wl.N, blk, win, dev.ws)
    assert xp.xp_readout_kernel_name(dev.head.handle) == "readout_tc_kernel"
    s = O.readout(O.decode(lat_np, wl.dtype), p.w2, O.decode(d["base"], wl.dtype))
    ids, vals, margin = O.argmax_lowest(s)
    got = blk.cpu().numpy()
    check_rows(got[:, 1:], ids, margin, "batched readout")
    same = got[:, 1:].reshape(-1) == ids.reshape(-1)
    check_close(win.cpu().numpy()[same], vals.reshape(-1)[same], LAT_TOL["bf16"], "win")


def test_batched_latent_all_rows(batched):
    wl, d, dev, p = batched
    xh_np = I.random_xh(wl, 42)
    lat = torch.empty(wl.N, wl.B - 1, wl.r, dtype=torch.bfloat16, device="cuda")
    xp.xp_latent_pass(dev.head.handle, dev.blk_in, dev.am1, torch.from_numpy(xh_np).cuda(), wl.N,
                      lat)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want = O.latent(d["blk"], d["am1"], xh_np.astype(np.float64), p)
    check_close(O.decode(xp.to_host_storage(lat), "bf16"), want, LAT_TOL["bf16"], "lat")


def test_batched_jacobi_sampled_blocks(batched):
    wl, d, dev, p = batched
    got = _run_jacobi(dev, wl)
    blocks = np.array([0, 7, 19, 31])
    want, margins = _oracle_jacobi(d, wl, p, blocks)
    check_blocks(got[blocks], want, margins, "batched jacobi")
    # the init and the near-tie rows: every block's slot 0 is its anchor
    assert np.array_equal(got[:, 0], d["anchor"])


def test_max_batch_sampled():
    wl = I.workload("max-batch")
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    blocks = np.array([0, 101, 255])
    want, margins = _oracle_jacobi(d, wl, p, blocks)
    # the launches the workload gets by default, then the persistent launch forced (128 latent
    # groups over its teams: several latent rounds per pass)
    for mode in (xp.XP_PASSES_AUTO, xp.XP_PASSES_PERSISTENT):
        xp.xp_set_pass_mode(dev.head.handle, mode)
        got = _run_jacobi(dev, wl)
        check_blocks(got[blocks], want, margins, f"max-batch jacobi, pass mode {mode}")
    xp.xp_set_pass_mode(dev.head.handle, xp.XP_PASSES_AUTO)
    # hidden cache (hidden = 5120) on the sampled blocks
    xh = torch.empty(wl.N, wl.B, wl.r, dtype=torch.float32, device="cuda")
    xp.xp_hidden_cache(dev.head.handle, dev.h, wl.N, xh, dev.ws)
    want_xh = O.xh_from_cache(O.hidden_cache(O.decode(d["h_full"][blocks], "bf16"), p.down_h,
                                             p.down_g), p.in_proj)
    check_close(xh.cpu().numpy()[blocks], want_xh, LAT_TOL["bf16"] / 4, "xh")
    dev.close()


def test_topc_sampled():
    wl = I.workload("topc")
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    C = wl.topc
    dt = torch.bfloat16
    cand = torch.empty(wl.N, wl.B - 1, C, dtype=torch.int64, device="cuda")
    base_c = torch.empty(wl.N, wl.B - 1, C, dtype=dt, device="cuda")
    w2c = torch.empty(wl.N, wl.B - 1, C, wl.r, dtype=dt, device="cuda")
    blk0 = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_topc_gather(dev.head.handle, dev.base, dev.sn, dev.sb, wl.N, C, cand, base_c, w2c, blk0)
    blocks = np.array([3, 128, 250])
    base_s = O.decode(d["base"][blocks], "bf16")
    want_cand, want_bc = O.topc_select(base_s, C)
    got_cand = cand.cpu().numpy()[blocks]
    assert np.array_equal(got_cand, want_cand)
    assert np.array_equal(O.decode(xp.to_host_storage(base_c[blocks]), "bf16"), want_bc)
    assert np.array_equal(xp.to_host_storage(w2c[blocks]), d["w2"][want_cand])
    assert np.array_equal(blk0.cpu().numpy()[blocks, 1:], O.argmax_lowest(base_s)[0])
    got = _run_jacobi(dev, wl, topc=C)
    want, margins = _oracle_jacobi(d, wl, p, blocks, topc=C)
    check_blocks(got[blocks], want, margins, "topc jacobi")
    dev.close()


def test_max_batch_readout_all_rows():
    # every one of the 3840 draft rows x V logits of the max-batch readout, in the launch
    # geometry the step uses (32 row tiles x 4 vocabulary segments), against fp64 logits
    # computed by the oracle in row chunks
    wl = I.workload("max-batch")
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    lat_np = I.random_lat(wl, 45)
    blk = dev.blk_in.clone()
    win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
    xp.xp_readout_argmax(dev.head.handle, xp.to_device(lat_np, wl.dtype), dev.base, dev.sn,
                         dev.sb, wl.N, blk, win, dev.ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    # the same readout as 2-CTA pairs (16 clusters of two row tiles x 4 segments)
    xp.xp_set_readout_pairs(dev.head.handle, True)
    assert xp.xp_readout_pairs(dev.head.handle, wl.N)
    blk2 = dev.blk_in.clone()
    win2 = torch.empty_like(win)
    xp.xp_readout_argmax(dev.head.handle, xp.to_device(lat_np, wl.dtype), dev.base, dev.sn,
                         dev.sb, wl.N, blk2, win2, dev.ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    assert torch.equal(blk2, blk)
    assert (win2 - win).abs().max().item() <= 1e-4
    got = blk.cpu().numpy()[:, 1:].reshape(-1)
    got_win = win.cpu().numpy()
    lat = O.decode(lat_np, wl.dtype).reshape(wl.rows, wl.r)
    base = d["base"].reshape(wl.rows, wl.V)
    ids = np.empty(wl.rows, np.int64)
    vals = np.empty(wl.rows)
    margin = np.empty(wl.rows)
    for r0 in range(0, wl.rows, 128):
        s = O.readout(lat[r0:r0 + 128], p.w2, O.decode(base[r0:r0 + 128], wl.dtype))
        ids[r0:r0 + 128], vals[r0:r0 + 128], margin[r0:r0 + 128] = O.argmax_lowest(s)
    check_rows(got, ids, margin, "max-batch readout")
    same = got == ids
    check_close(got_win[same], vals[same], LAT_TOL[wl.dtype], "max-batch win")
    dev.close()


def _topc_by_definition(row, C):
    """The C best ids of one row (value descending, ties at the boundary to the lower id),
    ascending: every id above the C-th largest value, then the lowest ids equal to it."""
    t = np.partition(row, row.size - C)[row.size - C]
    above = np.nonzero(row > t)[0]
    equal = np.nonzero(row == t)[0][: C - above.size]
    return np.sort(np.concatenate([above, equal]))


def test_topc_candidates_all_rows():
    # the candidate selection of the top-C workload (3840 rows x V, C = 512, Zipf rows): all
    # rows against the selection's definition, 32 whole blocks against the oracle itself
    wl = I.workload("topc")
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    C = wl.topc
    cand = torch.empty(wl.N, wl.B - 1, C, dtype=torch.int64, device="cuda")
    base_c = torch.empty(wl.N, wl.B - 1, C, dtype=torch.bfloat16, device="cuda")
    xp.xp_topc_gather(dev.head.handle, dev.base, dev.sn, dev.sb, wl.N, C, cand, base_c, None,
                      None)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    got_cand = cand.cpu().numpy().reshape(wl.rows, C)
    got_bc = xp.to_host_storage(base_c).reshape(wl.rows, C)
    base_bits = d["base"].reshape(wl.rows, wl.V)
    base = O.decode(base_bits, "bf16")
    bad = [r for r in range(wl.rows) if not np.array_equal(got_cand[r], _topc_by_definition(base[r], C))]
    assert not bad, f"{len(bad)} rows differ, first {bad[:5]}"
    assert np.array_equal(got_bc, np.take_along_axis(base_bits, got_cand, axis=1))
    blocks = np.arange(0, wl.N, wl.N // 32)[:32]
    want_cand, want_bc = O.topc_select(O.decode(d["base"][blocks], "bf16"), C)
    assert np.array_equal(got_cand.reshape(wl.N, wl.B - 1, C)[blocks], want_cand)
    assert np.array_equal(O.decode(got_bc.reshape(wl.N, wl.B - 1, C)[blocks], "bf16"), want_bc)
    dev.close()
