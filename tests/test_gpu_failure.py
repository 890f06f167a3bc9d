"""The kernels' failure path, exercised without a GPU fault.

Every mbarrier wait in the library is bounded in time: when it runs out it sets
XP_ETIMEOUT in the head's error word, raises its CTA's abort flag and returns, so
the kernel ends and the host reads the error.  xp_selftest_wait_timeout launches
one wait that nothing ever completes; afterwards the context must still run the
refinement correctly.
"""
import numpy as np
import pytest
import torch

from jacobi_speculative_decode_gb300 import inputs as I
from jacobi_speculative_decode_gb300 import xp
from oracle import xp_oracle as O
from parity import Dev, check_blocks

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_survives():
    wl = I.workload("batched-decode", V=5000, hidden=512, N=20, K=4)
    d = I.make_inputs(wl)
    dev = Dev(d, wl)
    p = O.params_from_inputs(d, wl.dtype)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    xp.xp_selftest_wait_timeout(dev.head.handle)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_ETIMEOUT
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK          # read and cleared
    # the same context still refines correctly (tensor-core kernels, their own waits)
    blk = torch.full((wl.N, wl.B), -1, dtype=torch.int64, device="cuda")
    xp.xp_jacobi_refine(dev.head.handle, dev.base, dev.sn, dev.sb, dev.h, dev.anchor, dev.am1,
                        wl.N, wl.K, 0, blk, dev.ws)
    assert xp.xp_get_error(dev.head.handle) == xp.XP_OK
    base = O.decode(d["base"], wl.dtype)
    h = O.decode(d["h_full"], wl.dtype)
    want, margins = O.jacobi_refine(base, h, d["anchor"], d["am1"], wl.K, p)
    check_blocks(blk.cpu().numpy(), want, margins, "after a timed-out wait")
    dev.close()
