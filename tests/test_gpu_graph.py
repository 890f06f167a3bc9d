"""A refine step captured into a CUDA graph and replayed (qwen3_xpress page: the refiner
runs inside captured CUDA graphs).  The calls make no host synchronisation and keep their
workspace addresses, so a captured step must replay to the same blk as a direct call,
every time, and that blk must follow the oracle."""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from oracle import xp_oracle as O
from parity import Dev, check_blocks

pytestmark = pytest.mark.gpu

SHAPES = [
    I.workload("batched-decode", V=5000, hidden=256, N=32, K=4),     # 4 row tiles: clusters
    I.workload("single-request", V=4104, hidden=256, B=5, N=40, K=3, base_kind="peaks_half_ties"),
]
IDS = ["B16-N32", "B5-N40"]


@pytest.mark.parametrize("wl", SHAPES, ids=IDS)
def test_captured_refine_replays_the_direct_call(wl):
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)

    def step(out):
        xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor,
                            dev.am1, wl.N, wl.K, 0, out, dev.ws)

    direct = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    step(direct)                                  # also warms every launch-time query
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    captured = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(captured)
    for _ in range(2):
        captured.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
        assert torch.equal(captured, direct)
    want, margins = O.jacobi_refine(O.decode(d["base"], wl.dtype), O.decode(d["h_full"], wl.dtype),
                                    d["anchor"], d["am1"], wl.K, p)
    check_blocks(captured.cpu().numpy(), want, margins, "graph replay")
    del g
    dev.close()
