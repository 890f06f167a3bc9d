"""The multi-rank host logic on CPU (gloo, world size 2): block sharding, gathering,
and the max-over-ranks timer.  Blocks are independent, so the sharded refinement
must equal the whole-batch one."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from jacobi_speculative_decode_gb300 import shard


def test_block_range_partitions():
    for n in (0, 1, 5, 32, 33):
        for world in (1, 2, 3, 8):
            spans = [shard.block_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(h - l for l, h in spans) - min(h - l for l, h in spans) <= 1
    with pytest.raises(ValueError):
        shard.block_range(4, 2, 2)
    assert shard.rank_seed(5, 0) == 5 and shard.rank_seed(5, 1) != shard.rank_seed(5, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    from jacobi_speculative_decode_gb300 import inputs as I
    from oracle import xp_oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = I.workload("tiny-fp32", N=5)
    d = I.make_inputs(wl)
    p = O.params_from_inputs(d, "f32")
    lo, hi = shard.block_range(wl.N, rank, world)
    base = O.decode(d["base"], "f32")[lo:hi]
    h = O.decode(d["h_full"], "f32")[lo:hi]
    blk, _ = O.jacobi_refine(base, h, d["anchor"][lo:hi], d["am1"][lo:hi], wl.K, p)
    parts = [None] * world
    dist.all_gather_object(parts, (lo, blk))
    slowest = shard.max_over_ranks(1.0 + rank)
    if rank == 0:
        out.put((parts, slowest))
    dist.destroy_process_group()


def test_sharded_refinement_equals_whole_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    parts, slowest = q.get(timeout=120)
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    from jacobi_speculative_decode_gb300 import inputs as I
    from oracle import xp_oracle as O
    wl = I.workload("tiny-fp32", N=5)
    d = I.make_inputs(wl)
    p = O.params_from_inputs(d, "f32")
    whole, _ = O.jacobi_refine(O.decode(d["base"], "f32"), O.decode(d["h_full"], "f32"),
                               d["anchor"], d["am1"], wl.K, p)
    got = np.concatenate([b for _, b in sorted(parts, key=lambda t: t[0])])
    assert np.array_equal(got, whole)
    assert slowest == 2.0
