"""The seeded input generator: determinism and the stated distributions/structure."""
import numpy as np

from jacobi_speculative_decode_gb300 import inputs as I


def test_deterministic():
    wl = I.workload("batched-decode", V=2048, hidden=64, r=64, H=64, N=4)
    a, b = I.make_inputs(wl), I.make_inputs(wl)
    for k in ("h_full", "w1", "w2", "base", "raw_mix", "anchor", "am1", "blk"):
        assert np.array_equal(a[k], b[k]), k


def test_chunked_draws_equal_one_draw():
    r1 = np.random.default_rng(5)
    one = r1.standard_normal(1000, dtype=np.float32)
    r2 = np.random.default_rng(5)
    parts = np.concatenate([r2.standard_normal(n, dtype=np.float32) for n in (1, 400, 599)])
    assert np.array_equal(one, parts)


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5], np.float32)
    assert I.f32_to_bf16_bits(x).tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020]


def test_scales():
    wl = I.workload("single-request", V=8192, hidden=1024)
    d = I.make_inputs(wl)
    f = lambda k: I.bf16_bits_to_f32(d[k]).astype(np.float64)
    assert abs(f("w2").std() * 16 - 1) < 0.02            # N(0, 1/256)
    assert abs(f("down_h").std() * 32 - 1) < 0.02        # N(0, 1/1024)
    assert abs(f("in_proj").std() * np.sqrt(768) - 1) < 0.02
    assert abs(f("raw_mix").std() / 0.1 - 1) < 0.05
    base = f("base").reshape(wl.rows, wl.V)
    assert (base.max(axis=1) > 8).all()                   # planted peaks
    assert 0 <= d["anchor"].min() and d["anchor"].max() < wl.V and d["blk"].dtype == np.int64


def test_near_ties_and_peaks():
    wl = I.workload("batched-decode", V=4096, hidden=64, N=32)
    d = I.make_inputs(wl)
    m = d["meta"]
    base = I.bf16_bits_to_f32(d["base"]).reshape(wl.rows, wl.V).astype(np.float64)
    assert len(m["peak_rows"]) == wl.rows // 2 and len(m["tie_rows"]) == wl.rows * 5 // 100
    for row, (v1, v2) in zip(m["tie_rows"], m["tie_ids"]):
        srt = np.sort(base[row])
        assert base[row, v1] == srt[-1] and base[row, v2] == srt[-2]
        assert 0 <= srt[-1] - srt[-2] <= 0.0625 + 1e-9


def test_zipf_rows_are_permuted_ranks():
    wl = I.workload("topc", V=4096, hidden=64, N=2, topc=64)
    d = I.make_inputs(wl)
    m = d["meta"]
    assert m["alpha"] >= 4.0
    for row in range(wl.rows):
        pi = (m["zipf_a"][row] * np.arange(wl.V) + m["zipf_b"][row]) % wl.V
        assert len(np.unique(pi)) == wl.V
