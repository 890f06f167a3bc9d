"""Pins of the fp64 CPU oracle against facts that do not come from the oracle itself.

Each test checks the oracle against a worked example written by hand
(tests/golden), a closed form, a special case that reduces the pass to
something checkable by eye, an invariant the pages state, or brute force on
tiny inputs.  Chosen so that a dropped term, a wrong index or sign, or a
transposed operand anywhere in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest

from conftest import load_golden
from oracle import xp_oracle as O
from jacobi_speculative_decode_gb300 import inputs as I


def _params(**kw):
    return O.Params(**{k: np.asarray(v, np.float64) for k, v in kw.items()})


def _rand_params(rng, V, hid, r, H, B, mix_scale=0.1):
    g = lambda *s: rng.standard_normal(s)
    raw = mix_scale * g(r, B, B)
    return O.Params(g(V, r) / math.sqrt(r), g(r, hid) / math.sqrt(hid),
                    g(r, hid) / math.sqrt(hid), g(r, 3 * r) / math.sqrt(3 * r),
                    O.fold(raw), g(H, r) / math.sqrt(r), g(H, r) / math.sqrt(r),
                    g(r, H) / math.sqrt(H), g(V, r) / math.sqrt(r))


# ---------------------------------------------------------------- storage ---

def test_bf16_encode_known_bit_patterns():
    # bf16 = top 16 bits of IEEE binary32; 8 significant bits; ties to even.
    cases = {1.0: 0x3F80, -2.5: 0xC020, 0.0: 0x0000, 0.15625: 0x3E20,
             1.0 + 2 ** -8: 0x3F80,                 # midpoint -> even (down)
             1.0 + 3 * 2 ** -8: 0x3F82,             # midpoint -> even (up)
             1.0 + 2 ** -8 + 2 ** -30: 0x3F81,      # just above midpoint: no double rounding
             3.0 + 2 ** -7: 0x4040,                 # spacing at 3 is 2^-6: midpoint -> even
             65280.0: 0x477F}
    x = np.array(list(cases), np.float64)
    got = O.encode(x, "bf16")
    assert [int(v) for v in got] == list(cases.values())


def test_bf16_decode_known_bit_patterns():
    bits = np.array([0x3F80, 0xC020, 0x0000, 0x8000, 0x3E20, 0x477F, 0x3F81], np.uint16)
    want = [1.0, -2.5, 0.0, -0.0, 0.15625, 65280.0, 1.0 + 2 ** -7]
    assert O.decode(bits, "bf16").tolist() == want


def test_f32_roundtrip_is_exact():
    x = np.array([1.0, 1 / 3, -7.25e-3], np.float64)
    assert O.decode(O.encode(x, "f32"), "f32").tolist() == np.float32(x).astype(np.float64).tolist()


# ------------------------------------------------------------------- fold ---

def test_fold_golden():
    g = load_golden("fold_b3.json")
    assert O.fold(np.array(g["raw"])).tolist() == g["folded"]
    assert O.fold(np.zeros((1, 3, 3))).tolist() == g["raw_zero_folded"]


def test_fold_index_by_index():
    rng = np.random.default_rng(1)
    raw = rng.standard_normal((5, 6, 6))
    f = O.fold(raw)
    for c in range(5):
        for b in range(6):
            for j in range(6):
                want = raw[c, b, j] + 1.0 if j == b else (raw[c, b, j] if j < b else 0.0)
                assert f[c, b, j] == want


def test_fold_stored_bf16_rounds_once():
    # the diagonal 1 + raw is rounded once from the exact sum
    raw_vals = np.array([2 ** -8, 3 * 2 ** -8, -2 ** -9, -2 ** -8, -3 * 2 ** -9, 0.1015625],
                        np.float64)
    raw = np.zeros((len(raw_vals), 1, 1))
    raw[:, 0, 0] = raw_vals
    stored = O.fold_stored(O.encode(raw, "bf16"), "bf16")
    got = O.decode(stored, "bf16")[:, 0, 0]
    # hand-rounded: spacing is 2^-7 above 1 and 2^-8 below it; midpoints go to the even pattern
    want = [1.0, 1.0 + 2 ** -6, 1.0, 1.0 - 2 ** -8, 1.0 - 2 ** -7, 1.1015625]
    assert got.tolist() == want


# -------------------------------------------------------- the whole pass ---

def test_pass_golden():
    g = load_golden("pass_tiny.json")
    p = _params(w1=g["w1"], down_h=g["down_h"], down_g=g["down_g"], in_proj=g["in_proj"],
                mix=O.fold(np.array(g["raw_mix"])), w_gate=g["w_gate"], w_up=g["w_up"],
                w_down=g["w_down"], w2=g["w2"])
    h = np.array(g["h_full"])
    xh = O.xh_from_cache(O.hidden_cache(h, p.down_h, p.down_g), p.in_proj)
    np.testing.assert_allclose(xh, g["expect_xh"], rtol=0, atol=1e-12)
    blk = np.array(g["blk"], np.int64)
    am1 = np.array(g["am1"], np.int64)
    lat = O.latent(blk, am1, xh, p)
    np.testing.assert_allclose(lat, g["expect_lat"], rtol=0, atol=1e-12)
    s = O.readout(lat, p.w2, np.array(g["base"]))
    np.testing.assert_allclose(s, g["expect_logits"], rtol=0, atol=1e-12)
    new_blk, _, _, _ = O.full_pass(blk, am1, xh, np.array(g["base"]), p)
    assert new_blk.tolist() == g["expect_blk_after_pass"]


# ----------------------------------------------------------- hidden cache ---

def test_hidden_cache_identity_projections_give_h():
    # hidden = r, down_h = I, down_g = 0, in_proj[:, :2r] = [I | 0]  =>  xh = h
    rng = np.random.default_rng(2)
    N, B, r = 3, 5, 4
    h = rng.standard_normal((N, B, r))
    W = np.concatenate([np.eye(r), np.zeros((r, r)), rng.standard_normal((r, r))], 1)
    xh = O.xh_from_cache(O.hidden_cache(h, np.eye(r), np.zeros((r, r))), W)
    np.testing.assert_allclose(xh, h, rtol=0, atol=1e-14)


def test_hidden_cache_mean_half_is_block_average():
    # down_h = 0, down_g = I, in_proj[:, :2r] = [0 | I]  =>  xh[n, b] = average of h[n, :]
    rng = np.random.default_rng(3)
    N, B, r = 3, 5, 4
    h = rng.standard_normal((N, B, r))
    W = np.concatenate([np.zeros((r, r)), np.eye(r), np.zeros((r, r))], 1)
    xh = O.xh_from_cache(O.hidden_cache(h, np.zeros((r, r)), np.eye(r)), W)
    for n in range(N):
        avg = [sum(h[n, b, c] for b in range(B)) / B for c in range(r)]
        for b in range(B):
            np.testing.assert_allclose(xh[n, b], avg, rtol=0, atol=1e-14)


def test_hidden_cache_constant_block_equal_halves():
    # h constant over a block's slots, down_g = down_h and in_proj[:, :r] = in_proj[:, r:2r]
    # => the two halves coincide and xh = 2 * in_proj[:, :r] down_h h
    rng = np.random.default_rng(4)
    N, B, hid, r = 2, 4, 6, 3
    h = np.repeat(rng.standard_normal((N, 1, hid)), B, axis=1)
    D = rng.standard_normal((r, hid))
    A = rng.standard_normal((r, r))
    W = np.concatenate([A, A, rng.standard_normal((r, r))], 1)
    xh = O.xh_from_cache(O.hidden_cache(h, D, D), W)
    for n in range(N):
        want = 2 * A @ (D @ h[n, 0])
        for b in range(B):
            np.testing.assert_allclose(xh[n, b], want, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------- latent ---

def _plain_head(V, r, H, B, rng):
    """Identity mixer, zero MLP, zero hidden part: lat is the embedding projection."""
    return O.Params(rng.standard_normal((V, r)), np.zeros((r, 1)), np.zeros((r, 1)),
                    np.concatenate([np.zeros((r, 2 * r)), rng.standard_normal((r, r))], 1),
                    O.fold(np.zeros((r, B, B))), np.zeros((H, r)), np.zeros((H, r)),
                    np.zeros((r, H)), rng.standard_normal((V, r)))


def test_latent_identity_mix_zero_mlp_is_in_proj_output():
    rng = np.random.default_rng(5)
    V, r, H, B, N = 11, 4, 6, 5, 3
    p = _plain_head(V, r, H, B, rng)
    xh = rng.standard_normal((N, B, r))
    blk = rng.integers(0, V, (N, B))
    am1 = rng.integers(0, V, N)
    lat = O.latent(blk, am1, xh, p)
    Wl = p.in_proj[:, 2 * r:]
    for n in range(N):
        for b in range(1, B):          # output index b-1 is slot b, which embeds blk[n, b-1]
            want = xh[n, b] + Wl @ p.w1[blk[n, b - 1]]
            np.testing.assert_allclose(lat[n, b - 1], want, rtol=0, atol=1e-13)


def test_latent_slot0_reads_am1_through_the_mixer():
    # mix slot 1 <- slot 0 with weight 1 on every channel; W_lat = I, xh = 0, zero MLP:
    # lat[slot 1] = w1[blk[n, 0]] + w1[am1[n]]
    rng = np.random.default_rng(6)
    V, r, H, B, N = 9, 3, 2, 3, 2
    raw = np.zeros((r, B, B))
    raw[:, 1, 0] = 1.0
    p = O.Params(rng.standard_normal((V, r)), np.zeros((r, 1)), np.zeros((r, 1)),
                 np.concatenate([np.zeros((r, 2 * r)), np.eye(r)], 1), O.fold(raw),
                 np.zeros((H, r)), np.zeros((H, r)), np.zeros((r, H)), np.zeros((V, r)))
    blk = np.array([[4, 7, 1], [0, 2, 8]])
    am1 = np.array([5, 3])
    lat = O.latent(blk, am1, np.zeros((N, B, r)), p)
    for n in range(N):
        np.testing.assert_allclose(lat[n, 0], p.w1[blk[n, 0]] + p.w1[am1[n]], atol=1e-14)
        np.testing.assert_allclose(lat[n, 1], p.w1[blk[n, 1]], atol=1e-14)


def test_latent_mixer_orientation_channel_out_in():
    # one entry raw[c=1, b=2, j=0] = m: only channel 1 of slot 2 picks up m * x[slot 0]
    rng = np.random.default_rng(7)
    V, r, H, B, N = 6, 3, 2, 4, 1
    p0 = _plain_head(V, r, H, B, rng)
    raw = np.zeros((r, B, B))
    raw[1, 2, 0] = 0.75
    p = p0._replace(mix=O.fold(raw))
    xh = rng.standard_normal((N, B, r))
    blk = rng.integers(0, V, (N, B))
    am1 = rng.integers(0, V, N)
    a = O.latent(blk, am1, xh, p0)
    b = O.latent(blk, am1, xh, p)
    x0 = xh[0, 0] + p.in_proj[:, 2 * r:] @ p.w1[am1[0]]
    d = b - a
    want = np.zeros_like(d)
    want[0, 1, 1] = 0.75 * x0[1]        # output index 1 = slot 2
    np.testing.assert_allclose(d, want, atol=1e-13)


def test_silu_values():
    z = np.array([0.0, 1.0, -1.0, 40.0, -40.0, 2.0])
    s = O.silu(z)
    assert s[0] == 0.0
    assert abs(s[1] - 1.0 / (1.0 + 1.0 / math.e)) < 1e-15        # sigmoid(1) = e/(1+e)
    assert abs((s[1] - s[2]) - 1.0) < 1e-15                       # silu(z) - silu(-z) = z
    assert abs(s[3] - 40.0) < 1e-12 and abs(s[4]) < 1e-15
    assert abs(s[5] - 2.0 * math.e ** 2 / (1.0 + math.e ** 2)) < 1e-15


def test_latent_mlp_plumbing_diagonal():
    # H = r, W_gate = diag(a), W_up = diag(b), W_down = I:
    # lat_c = u_c + silu(a_c u_c) * (b_c u_c), channel by channel (gate inside silu, up outside)
    rng = np.random.default_rng(8)
    V, r, B, N = 7, 4, 3, 2
    p0 = _plain_head(V, r, r, B, rng)
    a = np.array([1.0, -2.0, 0.5, 3.0])
    bb = np.array([2.0, 1.0, -1.0, 0.25])
    p = p0._replace(w_gate=np.diag(a), w_up=np.diag(bb), w_down=np.eye(r))
    xh = rng.standard_normal((N, B, r))
    blk = rng.integers(0, V, (N, B))
    am1 = rng.integers(0, V, N)
    u = O.latent(blk, am1, xh, p0)               # identity mixer: u = in_proj output
    lat = O.latent(blk, am1, xh, p)
    for n in range(N):
        for s in range(B - 1):
            for c in range(r):
                uc = u[n, s, c]
                z = a[c] * uc
                want = uc + z / (1.0 + math.exp(-z)) * (bb[c] * uc)
                assert abs(lat[n, s, c] - want) < 1e-12


def test_latent_causality():
    # changing blk[n, k] leaves the latent of slots <= k unchanged (slot b embeds blk[b-1])
    rng = np.random.default_rng(9)
    V, hid, r, H, B, N = 13, 5, 6, 7, 6, 2
    p = _rand_params(rng, V, hid, r, H, B, mix_scale=0.5)
    xh = rng.standard_normal((N, B, r))
    blk = rng.integers(0, V, (N, B))
    am1 = rng.integers(0, V, N)
    base_lat = O.latent(blk, am1, xh, p)
    for k in range(B - 1):
        b2 = blk.copy()
        b2[0, k] = (b2[0, k] + 1) % V
        lat = O.latent(b2, am1, xh, p)
        # output index s is slot s+1; slots <= k unchanged, slot k+1 changed
        np.testing.assert_array_equal(lat[0, :k], base_lat[0, :k])
        assert not np.allclose(lat[0, k], base_lat[0, k])
        np.testing.assert_array_equal(lat[1], base_lat[1])


# ---------------------------------------------------------- readout+argmax --

def test_argmax_golden_ties_and_signed_zero():
    g = load_golden("topc_ties.json")
    ids, win, margin = O.argmax_lowest(np.array([g["argmax_row"]]))
    assert int(ids[0]) == g["argmax_expect"] and margin[0] == 0.0


def test_readout_zero_w2_is_base_argmax():
    rng = np.random.default_rng(10)
    N, Bm1, V, r = 2, 3, 50, 4
    base = rng.standard_normal((N, Bm1, V))
    lat = rng.standard_normal((N, Bm1, r))
    ids, _, _ = O.argmax_lowest(O.readout(lat, np.zeros((V, r)), base))
    for n in range(N):
        for b in range(Bm1):
            row = base[n, b].tolist()
            assert ids[n, b] == row.index(max(row))


def test_readout_brute_force_small_vocab():
    rng = np.random.default_rng(11)
    N, Bm1, V, r = 2, 2, 37, 3
    base = rng.standard_normal((N, Bm1, V))
    lat = rng.standard_normal((N, Bm1, r))
    w2 = rng.standard_normal((V, r))
    s = O.readout(lat, w2, base)
    ids, win, margin = O.argmax_lowest(s)
    for n in range(N):
        for b in range(Bm1):
            vals = [base[n, b, v] + sum(w2[v, c] * lat[n, b, c] for c in range(r)) for v in range(V)]
            for v in range(V):
                assert abs(vals[v] - s[n, b, v]) < 1e-12
            best = max(vals)
            first = vals.index(best)
            second = max(x for i, x in enumerate(vals) if i != first)
            assert ids[n, b] == first
            assert abs(win[n, b] - best) < 1e-12 and abs(margin[n, b] - (best - second)) < 1e-12


# ------------------------------------------------------------------ top-C ---

def test_topc_golden_ties():
    g = load_golden("topc_ties.json")
    row = np.array([[g["base_row"]]])
    for case in g["cases"]:
        cand, base_c = O.topc_select(row, case["C"])
        assert cand[0, 0].tolist() == case["cand"]
        assert base_c[0, 0].tolist() == [g["base_row"][i] for i in case["cand"]]


def test_topc_winner_ties_to_lowest_vocab_id_not_position():
    s_c = np.array([[[2.0, 5.0, 5.0, 1.0]]])
    cand = np.array([[[9, 7, 3, 1]]])        # unsorted candidates: winner must be id 3
    ids, win, margin = O.topc_argmax(s_c, cand)
    assert ids[0, 0] == 3 and win[0, 0] == 5.0 and margin[0, 0] == 0.0


def test_topc_full_vocab_equals_full_pass():
    rng = np.random.default_rng(12)
    V, hid, r, H, B, N = 40, 6, 5, 7, 4, 3
    p = _rand_params(rng, V, hid, r, H, B)
    xh = rng.standard_normal((N, B, r))
    base = 3 * rng.standard_normal((N, B - 1, V))
    blk = rng.integers(0, V, (N, B))
    am1 = rng.integers(0, V, N)
    cand, base_c = O.topc_select(base, V)
    a = O.full_pass(blk, am1, xh, base, p)
    b = O.topc_pass(blk, am1, xh, cand, base_c, p)
    assert np.array_equal(a[0], b[0])
    np.testing.assert_allclose(a[2], b[2], atol=1e-12)


def test_topc_one_candidate_is_base_argmax():
    rng = np.random.default_rng(13)
    base = rng.standard_normal((2, 3, 30))
    cand, base_c = O.topc_select(base, 1)
    assert np.array_equal(cand[..., 0], O.argmax_lowest(base)[0])


def test_topc_select_brute_force():
    rng = np.random.default_rng(14)
    base = np.round(rng.standard_normal((1, 2, 25)) * 2) / 2      # many exact ties
    for C in (1, 3, 7, 25):
        cand, _ = O.topc_select(base, C)
        for b in range(2):
            row = base[0, b].tolist()
            ranked = sorted(range(25), key=lambda i: (-row[i], i))
            assert cand[0, b].tolist() == sorted(ranked[:C])


# ----------------------------------------------------------------- Jacobi ---

@pytest.mark.parametrize("seed,V,hid,r,H,B,N", [(20, 31, 5, 4, 6, 4, 2), (21, 23, 3, 3, 4, 5, 2),
                                                 (22, 17, 4, 2, 3, 6, 1)])
def test_jacobi_reaches_sequential_greedy(seed, V, hid, r, H, B, N):
    rng = np.random.default_rng(seed)
    p = _rand_params(rng, V, hid, r, H, B, mix_scale=0.4)
    h = rng.standard_normal((N, B, hid))
    # weak base so the refiner decides most slots
    base = 0.3 * rng.standard_normal((N, B - 1, V))
    anchor = rng.integers(0, V, N)
    am1 = rng.integers(0, V, N)
    seq = O.sequential_greedy(base, h, anchor, am1, p)
    xh = O.xh_from_cache(O.hidden_cache(h, p.down_h, p.down_g), p.in_proj)
    blk = O.init_blk(base, anchor)
    for k in range(1, B):
        blk = O.full_pass(blk, am1, xh, base, p)[0]
        # after pass k, slots 0..k agree with the sequential decode (settled prefix)
        assert np.array_equal(blk[:, : k + 1], seq[:, : k + 1])
    assert np.array_equal(blk, seq)
    again = O.full_pass(blk, am1, xh, base, p)[0]          # a fixed point
    assert np.array_equal(again, blk)
    full, _ = O.jacobi_refine(base, h, anchor, am1, B - 1, p)
    assert np.array_equal(full, seq)


def test_jacobi_tiny_workload_matches_sequential_greedy():
    wl = I.workload("tiny-fp32")
    d = I.make_inputs(wl)
    p = O.params_from_inputs(d, "f32")
    h, base = O.decode(d["h_full"], "f32"), O.decode(d["base"], "f32")
    seq = O.sequential_greedy(base, h, d["anchor"], d["am1"], p)
    blk, _ = O.jacobi_refine(base, h, d["anchor"], d["am1"], wl.B - 1, p)
    assert np.array_equal(blk, seq)


def test_zero_passes_is_init():
    rng = np.random.default_rng(15)
    p = _rand_params(rng, 20, 4, 3, 5, 4)
    base = rng.standard_normal((2, 3, 20))
    anchor = np.array([3, 11])
    blk, margins = O.jacobi_refine(base, rng.standard_normal((2, 4, 4)), anchor, np.array([0, 1]), 0, p)
    assert blk[:, 0].tolist() == [3, 11]
    assert np.array_equal(blk[:, 1:], np.argmax(base, -1)) and len(margins) == 1


# ------------------------------------------------- top-C Jacobi and params ---

def _brute_topc(base, C):
    """The C best ids of every row by (value descending, id ascending), by sorting lists."""
    N, Bm1, V = base.shape
    keep = np.zeros(base.shape, bool)
    for n in range(N):
        for b in range(Bm1):
            row = base[n, b].tolist()
            for i in sorted(range(V), key=lambda i: (-row[i], i))[:C]:
                keep[n, b, i] = True
    return keep


@pytest.mark.parametrize("seed,V,hid,r,H,B,N", [(40, 31, 5, 4, 6, 4, 2), (41, 23, 3, 3, 4, 5, 2),
                                                 (42, 17, 4, 2, 3, 6, 1)])
def test_topc_jacobi_equals_masked_sequential_greedy(seed, V, hid, r, H, B, N):
    # qwen3_xpress page, top-C branch of jacobi_refine_greedy: scoring only a row's C
    # best base candidates is full scoring with every other id pushed out of reach.  So
    # after B-1 passes the top-C refinement must equal the pure-Python slot-by-slot
    # greedy decode run on a base whose non-candidates are -1e30 (candidates chosen by
    # sorting each row).  Catches candidates taken from the wrong row or slice of base,
    # or chosen by the wrong order; C = V is the exact full-vocabulary case.
    rng = np.random.default_rng(seed)
    p = _rand_params(rng, V, hid, r, H, B, mix_scale=0.4)
    h = rng.standard_normal((N, B, hid))
    base = np.round(0.6 * rng.standard_normal((N, B - 1, V)) * 8) / 8     # ties included
    anchor = rng.integers(0, V, N)
    am1 = rng.integers(0, V, N)
    for C in (1, 2, 5, V // 2, V):
        masked = np.where(_brute_topc(base, C), base, -1e30)
        want = O.sequential_greedy(masked, h, anchor, am1, p)
        got, margins = O.jacobi_refine_topc(base, h, anchor, am1, B - 1, C, p)
        assert np.array_equal(got, want), C
        assert len(margins) == B


def test_topc_jacobi_full_vocab_on_tiny_workload():
    # C = V on the tiny-fp32 workload: the same blocks as the sequential greedy decode
    wl = I.workload("tiny-fp32")
    d = I.make_inputs(wl)
    p = O.params_from_inputs(d, "f32")
    h, base = O.decode(d["h_full"], "f32"), O.decode(d["base"], "f32")
    seq = O.sequential_greedy(base, h, d["anchor"], d["am1"], p)
    got, _ = O.jacobi_refine_topc(base, h, d["anchor"], d["am1"], wl.B - 1, wl.V, p)
    assert np.array_equal(got, seq)


@pytest.mark.parametrize("K", [0, 1, 3])
def test_topc_jacobi_one_candidate_keeps_the_base_argmax(K):
    # with one candidate per row every pass can only pick that row's best base id
    rng = np.random.default_rng(43)
    V, hid, r, H, B, N = 19, 4, 3, 5, 5, 3
    p = _rand_params(rng, V, hid, r, H, B)
    base = np.round(rng.standard_normal((N, B - 1, V)) * 4) / 4
    anchor = np.array([2, 7, 11])
    got, _ = O.jacobi_refine_topc(base, rng.standard_normal((N, B, hid)), anchor,
                                  rng.integers(0, V, N), K, 1, p)
    want = [[int(anchor[n])] + [max(range(V), key=lambda v: (base[n, b, v], -v))
                                for b in range(B - 1)] for n in range(N)]
    assert got.tolist() == want


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_params_from_inputs_maps_every_key_and_folds_once(dtype):
    # qwen3_xpress page, XPressRefinerHead.__init__ (parameter names and shapes) and
    # fold_from_raw_: every generated array lands in its own field, widened exactly,
    # and the raw mixer is folded exactly once.  Each array holds one distinct value
    # that bf16 represents exactly, so a swapped key shows up as a wrong value.
    V, hid, r, H, B = 6, 5, 4, 3, 3
    shapes = {"w1": (V, r), "down_h": (r, hid), "down_g": (r, hid), "in_proj": (r, 3 * r),
              "w_gate": (H, r), "w_up": (H, r), "w_down": (r, H), "w2": (V, r)}
    values = {"w1": 0.5, "down_h": -1.5, "down_g": 2.25, "in_proj": -0.375, "w_gate": 3.0,
              "w_up": -0.0625, "w_down": 1.75, "w2": -2.5}
    # bf16 bit patterns written by hand: sign | exponent | 7 fraction bits
    bits = {0.5: 0x3F00, -1.5: 0xBFC0, 2.25: 0x4010, -0.375: 0xBEC0, 3.0: 0x4040,
            -0.0625: 0xBD80, 1.75: 0x3FE0, -2.5: 0xC020, 0.25: 0x3E80}
    def stored(v, shape):
        if dtype == "bf16":
            return np.full(shape, bits[v], np.uint16)
        return np.full(shape, v, np.float32)
    inp = {k: stored(values[k], s) for k, s in shapes.items()}
    inp["raw_mix"] = stored(0.25, (r, B, B))
    p = O.params_from_inputs(inp, dtype)
    for k, v in values.items():
        arr = getattr(p, k)
        assert arr.shape == shapes[k] and arr.dtype == np.float64, k
        assert (arr == v).all(), (k, np.unique(arr))
    # folded once: 0.25 below the diagonal, 1.25 on it, 0 above (a second fold would
    # give 2.25 on the diagonal; no fold would leave 0.25 above it)
    want = np.array([[1.25, 0.0, 0.0], [0.25, 1.25, 0.0], [0.25, 0.25, 1.25]])
    assert p.mix.shape == (r, B, B)
    for c in range(r):
        assert p.mix[c].tolist() == want.tolist()
