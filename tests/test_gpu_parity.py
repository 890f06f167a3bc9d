"""GPU parity: every C-ABI entry point against the fp64 CPU oracle on seeded inputs.

Small shapes that still span several row tiles and a ragged vocabulary tail,
in both head dtypes, plus shapes the tensor-core kernels do not tile (odd V,
r = 64) so the plain CUDA kernels are covered too.  Full-size checks live in
test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from oracle import xp_oracle as O
from parity import LAT_TOL, MARGIN, Dev, check_blocks, check_close, check_rows

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


def _oracle_xh(d, wl, p):
    return O.xh_from_cache(O.hidden_cache(O.decode(d["h_full"], wl.dtype), p.down_h, p.down_g),
                           p.in_proj)


def test_fold_bit_exact(case):
    wl, d, dev, p = case
    want = O.fold_stored(d["raw_mix"], wl.dtype)
    got = xp.to_host_storage(dev.w["mix_L"])
    assert np.array_equal(got, want)


def test_fold_signed_zero_and_ties():
    # raw entries -0, midpoints of the bf16 grid around 1: rounding happens once
    raw = np.array([[[-0.0, -0.0, 5.0], [2 ** -8, -2 ** -9, -0.0], [3.0, -0.0, 3 * 2 ** -8]]])
    for dt in ("bf16", "f32"):
        stored = O.encode(raw, dt)
        t = xp.to_device(stored, dt)
        out = torch.empty_like(t)
        xp.xp_fold_mix(t, out, 1, 3, xp.XP_BF16 if dt == "bf16" else xp.XP_F32)
        torch.cuda.synchronize()
        assert np.array_equal(xp.to_host_storage(out), O.fold_stored(stored, dt))


def test_hidden_cache(case):
    wl, d, dev, p = case
    xh = torch.empty(wl.N, wl.B, wl.r, dtype=torch.float32, device="cuda")
    xp.xp_hidden_cache(dev.head.handle, dev.h, wl.N, xh, dev.ws)
    want = _oracle_xh(d, wl, p)
    check_close(xh.cpu().numpy(), want, LAT_TOL[wl.dtype] / 4, "xh")


def test_hidden_cache_fp32_grade(case):
    # bf16 inputs, but every product of the hidden cache is carried in fp32: the folded
    # projection keeps a hi + lo pair of bf16 planes, so a dropped lo plane (error near
    # 2^-9 of |xh|) or a missing mean term fails this bound
    wl, d, dev, p = case
    xh = torch.empty(wl.N, wl.B, wl.r, dtype=torch.float32, device="cuda")
    xp.xp_hidden_cache(dev.head.handle, dev.h, wl.N, xh, dev.ws)
    check_close(xh.cpu().numpy(), _oracle_xh(d, wl, p), 2e-4 if wl.dtype == "bf16" else 1e-4,
                "xh")


def test_hidden_cache_unaligned_input(case):
    # h_full one element past a 16-byte boundary cannot be tiled by TMA: the unfolded
    # path runs and must agree to the same bound
    wl, d, dev, p = case
    buf = torch.empty(dev.h.numel() + 8, dtype=dev.h.dtype, device="cuda")
    h1 = buf[1:1 + dev.h.numel()].view_as(dev.h)
    h1.copy_(dev.h)
    xh = torch.empty(wl.N, wl.B, wl.r, dtype=torch.float32, device="cuda")
    xp.xp_hidden_cache(dev.head.handle, h1, wl.N, xh, dev.ws)
    check_close(xh.cpu().numpy(), _oracle_xh(d, wl, p), 2e-4 if wl.dtype == "bf16" else 1e-4,
                "xh")


def test_latent(case):
    wl, d, dev, p = case
    xh_np = I.random_xh(wl, seed=7)
    xh = torch.from_numpy(xh_np).cuda()
    lat = torch.empty(wl.N, wl.B - 1, wl.r, dtype=xp.torch_dtype(wl.dtype), device="cuda")
    xp.xp_latent_pass(dev.head.handle, dev.blk_in, dev.am1, xh, wl.N, lat)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want = O.latent(d["blk"], d["am1"], xh_np.astype(np.float64), p)
    got = O.decode(xp.to_host_storage(lat), wl.dtype)
    check_close(got, want, LAT_TOL[wl.dtype], "lat")


def test_init_argmax(case):
    wl, d, dev, p = case
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
    xp.xp_init_argmax(dev.head.handle, dev.base, dev.sn, dev.sb, dev.anchor, wl.N, blk, win, dev.ws)
    base = O.decode(d["base"], wl.dtype)
    want = O.init_blk(base, d["anchor"])
    # both sides compare the same stored values: exact, ties to the lowest id included
    assert np.array_equal(blk.cpu().numpy(), want)
    assert np.array_equal(win.cpu().numpy().astype(np.float64), base.max(-1).reshape(-1))


def _random_lat(wl, seed=11):
    return I.random_lat(wl, seed)


def _readout_check(wl, d, dev, p, base_ptr, sn, sb, lat_np):
    lat = xp.to_device(lat_np, wl.dtype)
    blk = dev.blk_in.clone()
    win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
    xp.xp_readout_argmax(dev.head.handle, lat, base_ptr, sn, sb, wl.N, blk, win, dev.ws)
    s = O.readout(O.decode(lat_np, wl.dtype), p.w2, O.decode(d["base"], wl.dtype))
    ids, vals, margin = O.argmax_lowest(s)
    got = blk.cpu().numpy()
    assert np.array_equal(got[:, 0], d["blk"][:, 0])          # slot 0 untouched
    excused = check_rows(got[:, 1:], ids, margin, "readout")
    same = got[:, 1:].reshape(-1) == ids.reshape(-1)
    check_close(win.cpu().numpy()[same], vals.reshape(-1)[same], LAT_TOL[wl.dtype], "win")
    return excused


def test_readout_argmax(case):
    wl, d, dev, p = case
    _readout_check(wl, d, dev, p, dev.base, dev.sn, dev.sb, _random_lat(wl))


def test_readout_argmax_twice_same_workspace(case):
    # the argmax partials and tickets are reset by the last CTA of each tile
    wl, d, dev, p = case
    lat_np = _random_lat(wl, seed=12)
    _readout_check(wl, d, dev, p, dev.base, dev.sn, dev.sb, lat_np)
    _readout_check(wl, d, dev, p, dev.base, dev.sn, dev.sb, lat_np)


def test_readout_strided_full_block_layout(case):
    # base given as [N, B, V] with an unused slot-0 row: draft rows start one row in
    wl, d, dev, p = case
    full = torch.zeros(wl.N, wl.B, wl.V, dtype=xp.torch_dtype(wl.dtype), device="cuda")
    full[:, 1:, :] = dev.base
    view = full[:, 1:, :]
    _readout_check(wl, d, dev, p, view.data_ptr(), wl.B * wl.V, wl.V, _random_lat(wl, 13))


def test_readout_zero_w2_is_init(case):
    # a zero latent makes the readout the plain base argmax
    wl, d, dev, p = case
    lat = np.zeros((wl.N, wl.B - 1, wl.r), np.uint16 if wl.dtype == "bf16" else np.float32)
    blk = dev.blk_in.clone()
    xp.xp_readout_argmax(dev.head.handle, xp.to_device(lat, wl.dtype), dev.base, dev.sn, dev.sb,
                         wl.N, blk, None, dev.ws)
    want = O.argmax_lowest(O.decode(d["base"], wl.dtype))[0]
    assert np.array_equal(blk.cpu().numpy()[:, 1:], want)


@pytest.mark.parametrize("C", [1, 37, 512])
def test_topc_gather(case, C):
    wl, d, dev, p = case
    C = min(C, wl.V)
    dt = xp.torch_dtype(wl.dtype)
    cand = torch.empty(wl.N, wl.B - 1, C, dtype=torch.int64, device="cuda")
    base_c = torch.empty(wl.N, wl.B - 1, C, dtype=dt, device="cuda")
    w2c = torch.empty(wl.N, wl.B - 1, C, wl.r, dtype=dt, device="cuda")
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_topc_gather(dev.head.handle, dev.base, dev.sn, dev.sb, wl.N, C, cand, base_c, w2c, blk)
    base = O.decode(d["base"], wl.dtype)
    want_cand, want_bc = O.topc_select(base, C)
    assert np.array_equal(cand.cpu().numpy(), want_cand)
    assert np.array_equal(O.decode(xp.to_host_storage(base_c), wl.dtype), want_bc)
    assert np.array_equal(xp.to_host_storage(w2c), d["w2"][want_cand])
    assert np.array_equal(blk.cpu().numpy()[:, 1:], O.argmax_lowest(base)[0])
    assert (blk.cpu().numpy()[:, 0] == -1).all()


@pytest.mark.parametrize("materialise", [True, False])
def test_topc_readout(case, materialise):
    wl, d, dev, p = case
    C = min(64, wl.V)
    dt = xp.torch_dtype(wl.dtype)
    base = O.decode(d["base"], wl.dtype)
    cand_np, bc_np = O.topc_select(base, C)
    cand = torch.from_numpy(cand_np).cuda()
    base_c = xp.to_device(O.encode(bc_np, wl.dtype), wl.dtype)
    w2c = xp.to_device(d["w2"][cand_np], wl.dtype) if materialise else None
    lat_np = _random_lat(wl, 14)
    blk = dev.blk_in.clone()
    win = torch.empty(wl.rows, dtype=torch.float32, device="cuda")
    xp.xp_topc_readout_argmax(dev.head.handle, xp.to_device(lat_np, wl.dtype), base_c, cand, w2c,
                              wl.N, C, blk, win)
    s_c = O.topc_scores(O.decode(lat_np, wl.dtype), p.w2, cand_np, bc_np)
    ids, vals, margin = O.topc_argmax(s_c, cand_np)
    got = blk.cpu().numpy()
    check_rows(got[:, 1:], ids, margin, "topc readout")
    same = got[:, 1:].reshape(-1) == ids.reshape(-1)
    check_close(win.cpu().numpy()[same], vals.reshape(-1)[same], LAT_TOL[wl.dtype], "topc win")


def test_jacobi_refine_full_vocab(case):
    wl, d, dev, p = case
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, wl.K, 0, blk, dev.ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want, margins = O.jacobi_refine(O.decode(d["base"], wl.dtype), O.decode(d["h_full"], wl.dtype),
                                    d["anchor"], d["am1"], wl.K, p)
    check_blocks(blk.cpu().numpy(), want, margins, "jacobi")


def test_jacobi_refine_topc(case):
    wl, d, dev, p = case
    C = min(96, wl.V)
    ws = dev.head.workspace(wl.N, C)
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, wl.K, C, blk, ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want, margins = O.jacobi_refine_topc(O.decode(d["base"], wl.dtype),
                                         O.decode(d["h_full"], wl.dtype), d["anchor"], d["am1"],
                                         wl.K, C, p)
    check_blocks(blk.cpu().numpy(), want, margins, "jacobi topc")


def test_topc_with_C_equal_V_matches_full_vocab(case):
    wl, d, dev, p = case
    # rows x C > V here, so the passes read the candidates' w2 rows by id from w2 and
    # the workspace holds only cand and base_c (rows x V ids and values)
    ws = dev.head.workspace(wl.N, wl.V)
    a = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    b = a.clone()
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, wl.K, wl.V, a, ws)
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, wl.K, 0, b, ws)
    want, margins = O.jacobi_refine(O.decode(d["base"], wl.dtype), O.decode(d["h_full"], wl.dtype),
                                    d["anchor"], d["am1"], wl.K, p)
    check_blocks(a.cpu().numpy(), want, margins, "topc C=V")
    check_blocks(b.cpu().numpy(), want, margins, "full")


def test_bad_token_is_flagged_and_clamped(case):
    wl, d, dev, p = case
    blk_np = d["blk"].copy()
    blk_np[0, 1] = wl.V + 5          # read by slot 2 of block 0
    blk_np[-1, 0] = -3               # read by slot 1 of the last block
    blk = torch.from_numpy(blk_np).cuda()
    xh_np = I.random_xh(wl, seed=8)
    lat = torch.empty(wl.N, wl.B - 1, wl.r, dtype=xp.torch_dtype(wl.dtype), device="cuda")
    xp.xp_latent_pass(dev.head.handle, blk, dev.am1, torch.from_numpy(xh_np).cuda(), wl.N, lat)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_EBADTOKEN
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK            # read clears the flag
    clamped = blk_np.copy()
    clamped[0, 1] = wl.V - 1
    clamped[-1, 0] = 0
    want = O.latent(clamped, d["am1"], xh_np.astype(np.float64), p)
    check_close(O.decode(xp.to_host_storage(lat), wl.dtype), want, LAT_TOL[wl.dtype], "clamped lat")


def test_capacity_and_validation(case):
    wl, d, dev, p = case
    blk = dev.blk_in.clone()
    with pytest.raises(xp.XPError) as e:
        xp.xp_readout_argmax(dev.head.handle, dev.base, dev.base, dev.sn, dev.sb, wl.N + 1, blk,
                             None, dev.ws)
    assert e.value.code == xp.XP_ECAPACITY
    with pytest.raises(xp.XPError) as e:
        xp.xp_topc_gather(dev.head.handle, dev.base, dev.sn, dev.sb, wl.N, wl.V + 1, blk, blk,
                          None, None)
    assert e.value.code == xp.XP_EINVAL
    # zero blocks is a no-op
    xp.xp_readout_argmax(dev.head.handle, dev.base, dev.base, dev.sn, dev.sb, 0, blk, None, dev.ws)


def test_latent_persistent_many_groups():
    # more row groups than co-resident clusters: every cluster walks several groups
    wl = I.workload("batched-decode", V=4096, hidden=64, N=300, K=1)
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    xh_np = I.random_xh(wl, seed=5)
    lat = torch.empty(wl.N, wl.B - 1, wl.r, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):                       # twice: the second call reuses warm state
        xp.xp_latent_pass(dev.head.handle, dev.blk_in, dev.am1, torch.from_numpy(xh_np).cuda(),
                          wl.N, lat)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want = O.latent(d["blk"], d["am1"], xh_np.astype(np.float64), p)
    check_close(O.decode(xp.to_host_storage(lat), "bf16"), want, LAT_TOL["bf16"], "lat")
    dev.close()


def test_fp16_range_flag():
    # the tensor-core latent exchanges fp16: a weight or a latent value past its range
    # saturates and is reported, never silently turned into inf
    wl = I.workload("batched-decode", V=4096, hidden=64, N=4, K=1)
    d = I.make_inputs(wl)
    d["w_gate"] = d["w_gate"].copy()
    d["w_gate"][3, 5] = I.f32_to_bf16_bits(np.float32([1.0e6]))[0]
    dev = Dev(d, wl)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_ERANGE
    dev.close()
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    xh_np = I.random_xh(wl, seed=3)
    xh_np[1, 2, 7] = 1.0e6
    lat = torch.empty(wl.N, wl.B - 1, wl.r, dtype=torch.bfloat16, device="cuda")
    xp.xp_latent_pass(dev.head.handle, dev.blk_in, dev.am1, torch.from_numpy(xh_np).cuda(), wl.N,
                      lat)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_ERANGE
    dev.close()


@pytest.mark.parametrize("B,N", [(3, 37), (32, 5), (7, 41)])
def test_latent_group_shapes(B, N):
    # blocks per row group of the cluster latent: 10 (generic path), 1 and 4 / 6
    wl = I.workload("batched-decode", V=4096, hidden=64, B=B, N=N, K=2)
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    xh_np = I.random_xh(wl, seed=11)
    lat = torch.empty(wl.N, wl.B - 1, wl.r, dtype=torch.bfloat16, device="cuda")
    xp.xp_latent_pass(dev.head.handle, dev.blk_in, dev.am1, torch.from_numpy(xh_np).cuda(), wl.N,
                      lat)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want = O.latent(d["blk"], d["am1"], xh_np.astype(np.float64), p)
    check_close(O.decode(xp.to_host_storage(lat), "bf16"), want, LAT_TOL["bf16"], "lat")
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, wl.K, 0, blk, dev.ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    want_blk, margins = O.jacobi_refine(O.decode(d["base"], "bf16"), O.decode(d["h_full"], "bf16"),
                                        d["anchor"], d["am1"], wl.K, p)
    check_blocks(blk.cpu().numpy(), want_blk, margins, f"jacobi B={B}")
    dev.close()
