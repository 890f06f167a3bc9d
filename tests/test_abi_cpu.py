"""The C-ABI library on a machine without a GPU: it loads, exports every symbol that
include/xp.h declares, and its host-side validation answers without touching a device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from jacobi_speculative_decode_gb300 import build as B
from jacobi_speculative_decode_gb300 import xp


@pytest.fixture(scope="module")
def lib():
    B.build()
    return xp.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "xp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(xp_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("xp_hidden_cache", "xp_latent_pass", "xp_readout_argmax", "xp_topc_gather",
                 "xp_topc_readout_argmax", "xp_jacobi_refine", "xp_init_argmax", "xp_fold_mix"):
        assert want in names


def test_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(_declared()) == sorted(xp.exported_symbols())


def test_status_strings(lib):
    for code in range(9):
        assert xp.status_str(code) and xp.status_str(code) != "unknown status"


def _w(**kw):
    base = dict(V=151936, hidden=4096, r=256, H=512, B=16, max_N=32, dtype=xp.XP_BF16)
    base.update(kw)
    return xp.make_weights(**base)


def test_sizes(lib):
    w = _w()
    es = 2
    prep = xp.xp_head_prep_bytes(w)
    # every prepared copy is present: w1 + w2 + down_h + down_g + in_proj + mix + MLP,
    # plus the [b][j][channel] copy of the mixer, the fp32 projected embedding table and
    # the folded hidden-cache projection [2r, hidden] as two bf16 planes (hi, lo) and
    # the fp16 copies of the SwiGLU input weights
    floor = es * (2 * 151936 * 256 + 2 * 256 * 4096 + 3 * 256 * 256 + 256 * 16 * 16 + 3 * 512 * 256)
    floor += es * 256 * 16 * 16 + 4 * 151936 * 256 + 2 * es * 512 * 4096
    floor += 2 * 2 * 512 * 256      # fp16 copies of w_gate and w_up
    assert floor <= prep <= floor + 64 * 1024
    ws0 = xp.xp_workspace_bytes(w, 32, 0)
    ws1 = xp.xp_workspace_bytes(w, 32, 512)
    rows = 32 * 15
    # 480 rows x 512 candidates > V: cand and base_c only, the passes read w2 rows by id
    assert rows * 512 * (8 + 2) <= ws1 - ws0 < rows * 512 * (8 + 2) + 4 * 1024
    # one block x 16 candidates <= V: the step copies the candidates' w2 rows as well
    ws2 = xp.xp_workspace_bytes(w, 1, 16)
    assert ws2 - xp.xp_workspace_bytes(w, 1, 0) >= 15 * 16 * (8 + 2 + 256 * 2)
    assert xp.xp_head_prep_bytes(_w(B=1)) == 0            # B >= 2
    assert xp.xp_workspace_bytes(_w(dtype=7), 1, 0) == 0   # unknown dtype


def test_validation_without_device(lib):
    L = lib
    # no head -> XP_ENOTPREPARED, before any CUDA call
    assert L.xp_latent_pass(None, 1, 1, 1, 1, 1, None) == xp.XP_ENOTPREPARED
    assert L.xp_readout_argmax(None, 1, 1, 0, 0, 1, 1, None, 1, 1 << 20, None) == xp.XP_ENOTPREPARED
    assert L.xp_jacobi_refine(None, 1, 0, 0, 1, 1, 1, 1, 1, 0, 1, 1, 1 << 20, None) == \
        xp.XP_ENOTPREPARED
    assert L.xp_hidden_cache(None, 1, 1, 1, 1, 1 << 20, None) == xp.XP_ENOTPREPARED
    assert L.xp_init_argmax(None, 1, 0, 0, 1, 1, 1, None, 1, 1 << 20, None) == xp.XP_ENOTPREPARED
    assert L.xp_get_error(None, None) == xp.XP_ENOTPREPARED
    assert L.xp_refine_logits(None, 1, None, 0, 0, 1, 1, 4096, None) == xp.XP_ENOTPREPARED
    assert L.xp_selftest_wait_timeout(None, None) == xp.XP_ENOTPREPARED
    assert L.xp_readout_argmax_noalloc(None, 1, 1, 0, 0, 1, 1, None, None) == xp.XP_ENOTPREPARED
    # null pointers / bad shapes -> XP_EINVAL
    w = _w()
    out = ctypes.c_void_p()
    assert L.xp_head_create(ctypes.byref(w), None, 0, None, ctypes.byref(out)) == xp.XP_EINVAL
    assert L.xp_fold_mix(None, None, 4, 4, 0, None) == xp.XP_EINVAL
    assert L.xp_fold_mix(1, 1, 4, 4, 9, None) == xp.XP_EINVAL
    assert L.xp_workspace_init(None, 16, None) == xp.XP_EINVAL
    assert L.xp_head_create(None, 1, 1, None, ctypes.byref(out)) == xp.XP_EINVAL


def _header_prototypes():
    """name -> list of parameter declarations, from include/xp.h (comments removed)."""
    src = open(os.path.join(ROOT, "include", "xp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(xp_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", src):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        protos[m.group(1)] = params
    return protos


def _ctype_class(decl):
    """The ctypes kind a C parameter declaration marshals to (pointer, int64, size, int)."""
    d = " ".join(decl.split())
    if "*" in d:
        return "ptr"
    if "cudaStream_t" in d:
        return "ptr"
    if d.startswith("int64_t") or d.startswith("const int64_t"):
        return "i64"
    if d.startswith("size_t"):
        return "size"
    return "int"


def test_binding_signatures_match_the_header():
    # every ctypes argument list has the header's arity and the same kind per position,
    # so a binding cannot silently drop, add or narrow an argument
    protos = _header_prototypes()
    kinds = {ctypes.c_void_p: "ptr", ctypes.c_int64: "i64", ctypes.c_size_t: "size",
             ctypes.c_int: "int"}
    for name, (_, args) in xp._SIGS.items():
        assert name in protos, name
        want = [_ctype_class(d) for d in protos[name]]
        got = [kinds.get(a, "ptr") for a in args]   # struct pointers marshal as pointers
        assert got == want, f"{name}: binding {got} != header {want}"
