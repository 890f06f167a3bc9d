"""Thin ctypes binding of libxp.so (the C ABI in include/xp.h), same names as the C calls.

Argument marshalling only: tensors become raw pointers, ``None`` becomes NULL,
the stream defaults to torch's current stream.  Every step of the pass runs in
the library's CUDA kernels; there is no Python or CPU fallback -- a missing
library or device raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libxp.so")

XP_BF16, XP_F32 = 0, 1
XP_PASSES_AUTO, XP_PASSES_PERSISTENT, XP_PASSES_PER_STAGE = 0, 1, 2
STATUS = {0: "XP_OK", 1: "XP_EINVAL", 2: "XP_ECAPACITY", 3: "XP_ENOTPREPARED", 4: "XP_ECUDA",
          5: "XP_EBADTOKEN", 6: "XP_ETIMEOUT", 7: "XP_EUNSUPPORTED", 8: "XP_ERANGE"}
XP_OK, XP_EINVAL, XP_ECAPACITY, XP_ENOTPREPARED, XP_ECUDA, XP_EBADTOKEN, XP_ETIMEOUT, \
    XP_EUNSUPPORTED, XP_ERANGE = range(9)


class XPError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({status_str(code)})")
        self.code = code


class xp_weights(ctypes.Structure):
    _fields_ = [("V", ctypes.c_int), ("hidden", ctypes.c_int), ("r", ctypes.c_int),
                ("H", ctypes.c_int), ("B", ctypes.c_int), ("max_N", ctypes.c_int),
                ("dtype", ctypes.c_int),
                ("w1", ctypes.c_void_p), ("down_h", ctypes.c_void_p), ("down_g", ctypes.c_void_p),
                ("in_proj", ctypes.c_void_p), ("mix_L", ctypes.c_void_p),
                ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("w2", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_S = ctypes.c_size_t
_SIGS = {
    "xp_head_prep_bytes": (_S, [ctypes.POINTER(xp_weights)]),
    "xp_workspace_bytes": (_S, [ctypes.POINTER(xp_weights), _I, _I]),
    "xp_workspace_init": (_I, [_P, _S, _P]),
    "xp_head_create": (_I, [ctypes.POINTER(xp_weights), _P, _S, _P, ctypes.POINTER(_P)]),
    "xp_head_refill": (_I, [_P, ctypes.POINTER(xp_weights), _P]),
    "xp_head_destroy": (None, [_P]),
    "xp_fold_mix": (_I, [_P, _P, _I, _I, _I, _P]),
    "xp_hidden_cache": (_I, [_P, _P, _I, _P, _P, _S, _P]),
    "xp_latent_pass": (_I, [_P, _P, _P, _P, _I, _P, _P]),
    "xp_readout_argmax": (_I, [_P, _P, _P, _I64, _I64, _I, _P, _P, _P, _S, _P]),
    "xp_readout_argmax_noalloc": (_I, [_P, _P, _P, _I64, _I64, _I, _P, _P, _P]),
    "xp_refine_logits": (_I, [_P, _P, _P, _I64, _I64, _I, _P, _I64, _P]),
    "xp_selftest_wait_timeout": (_I, [_P, _P]),
    "xp_init_argmax": (_I, [_P, _P, _I64, _I64, _P, _I, _P, _P, _P, _S, _P]),
    "xp_topc_gather": (_I, [_P, _P, _I64, _I64, _I, _I, _P, _P, _P, _P, _P]),
    "xp_topc_readout_argmax": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _P, _P]),
    "xp_jacobi_refine": (_I, [_P, _P, _I64, _I64, _P, _P, _P, _I, _I, _I, _P, _P, _S, _P]),
    "xp_jacobi_passes": (_I, [_P, _P, _I64, _I64, _P, _P, _I, _I, _P, _P, _S, _P]),
    "xp_set_pass_mode": (_I, [_P, _I]),
    "xp_passes_persistent": (_I, [_P, _P, _I64, _I64, _I]),
    "xp_set_readout_pairs": (_I, [_P, _I]),
    "xp_readout_pairs": (_I, [_P, _I]),
    "xp_get_error": (_I, [_P, _P]),
    "xp_readout_kernel_name": (ctypes.c_char_p, [_P]),
    "xp_profile_timeline": (_I, [_P, _P, _S, _I, ctypes.POINTER(_S)]),
    "xp_status_str": (ctypes.c_char_p, [_I]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libxp.so once (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "jacobi_speculative_decode_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            raise RuntimeError("no CUDA device: libxp has no CPU path")
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(x):
    """Size in bytes of a buffer given as a tensor (0 for None)."""
    if x is None:
        return 0
    return x.numel() * x.element_size()


def _check(name, code):
    if code != XP_OK:
        raise XPError(name, code)


def status_str(code: int) -> str:
    return lib().xp_status_str(code).decode()


# ------------------------------------------------------------------ sizing ---

def make_weights(V, hidden, r, H, B, max_N, dtype, w1=None, down_h=None, down_g=None,
                 in_proj=None, mix_L=None, w_gate=None, w_up=None, w_down=None, w2=None):
    return xp_weights(V, hidden, r, H, B, max_N, dtype, _ptr(w1), _ptr(down_h), _ptr(down_g),
                      _ptr(in_proj), _ptr(mix_L), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                      _ptr(w2))


def xp_head_prep_bytes(w: xp_weights) -> int:
    return lib().xp_head_prep_bytes(ctypes.byref(w))


def xp_workspace_bytes(w: xp_weights, N: int, topc: int = 0) -> int:
    return lib().xp_workspace_bytes(ctypes.byref(w), N, topc)


# ------------------------------------------------------------------- calls ---

def xp_workspace_init(ws, stream=None):
    _check("xp_workspace_init", lib().xp_workspace_init(_ptr(ws), ws.numel() * ws.element_size(),
                                                        _stream(stream)))


def xp_head_create(w: xp_weights, prep, stream=None):
    out = ctypes.c_void_p()
    _check("xp_head_create", lib().xp_head_create(ctypes.byref(w), _ptr(prep),
                                                  prep.numel() * prep.element_size(),
                                                  _stream(stream), ctypes.byref(out)))
    return out.value


def xp_head_refill(head, w: xp_weights, stream=None):
    _check("xp_head_refill", lib().xp_head_refill(head, ctypes.byref(w), _stream(stream)))


def xp_head_destroy(head):
    lib().xp_head_destroy(head)


def xp_fold_mix(raw, mix, r, B, dtype, stream=None):
    _check("xp_fold_mix", lib().xp_fold_mix(_ptr(raw), _ptr(mix), r, B, dtype, _stream(stream)))


def xp_hidden_cache(head, h_full, N, xh, ws, stream=None):
    _check("xp_hidden_cache", lib().xp_hidden_cache(head, _ptr(h_full), N, _ptr(xh), _ptr(ws),
                                                    _nbytes(ws), _stream(stream)))


def xp_latent_pass(head, blk, am1, xh, N, lat, stream=None):
    _check("xp_latent_pass", lib().xp_latent_pass(head, _ptr(blk), _ptr(am1), _ptr(xh), N,
                                                  _ptr(lat), _stream(stream)))


def xp_readout_argmax(head, lat, base, stride_n, stride_b, N, blk, win_val, ws, stream=None):
    _check("xp_readout_argmax", lib().xp_readout_argmax(
        head, _ptr(lat), _ptr(base), stride_n, stride_b, N, _ptr(blk), _ptr(win_val), _ptr(ws),
        _nbytes(ws), _stream(stream)))


def xp_readout_argmax_noalloc(head, lat, base, stride_n, stride_b, N, blk, win_val, stream=None):
    """xp_readout_argmax without a workspace, for callers that cannot allocate device memory."""
    _check("xp_readout_argmax_noalloc", lib().xp_readout_argmax_noalloc(
        head, _ptr(lat), _ptr(base), stride_n, stride_b, N, _ptr(blk), _ptr(win_val),
        _stream(stream)))


def xp_selftest_wait_timeout(head, stream=None):
    """Launch one wait that can only end by its time limit (sets XP_ETIMEOUT)."""
    _check("xp_selftest_wait_timeout", lib().xp_selftest_wait_timeout(head, _stream(stream)))


def xp_refine_logits(head, lat, base, stride_n, stride_b, N, out, ld_out, stream=None):
    """Draft rows' fp32 logits base + lat.w2 (the bias alone when base is None)."""
    _check("xp_refine_logits", lib().xp_refine_logits(
        head, _ptr(lat), _ptr(base), stride_n, stride_b, N, _ptr(out), ld_out, _stream(stream)))


def xp_init_argmax(head, base, stride_n, stride_b, anchor, N, blk, win_val, ws, stream=None):
    _check("xp_init_argmax", lib().xp_init_argmax(
        head, _ptr(base), stride_n, stride_b, _ptr(anchor), N, _ptr(blk), _ptr(win_val),
        _ptr(ws), _nbytes(ws), _stream(stream)))


def xp_topc_gather(head, base, stride_n, stride_b, N, C, cand, base_c, w2c, blk, stream=None):
    _check("xp_topc_gather", lib().xp_topc_gather(
        head, _ptr(base), stride_n, stride_b, N, C, _ptr(cand), _ptr(base_c), _ptr(w2c),
        _ptr(blk), _stream(stream)))


def xp_topc_readout_argmax(head, lat, base_c, cand, w2c, N, C, blk, win_val, stream=None):
    _check("xp_topc_readout_argmax", lib().xp_topc_readout_argmax(
        head, _ptr(lat), _ptr(base_c), _ptr(cand), _ptr(w2c), N, C, _ptr(blk), _ptr(win_val),
        _stream(stream)))


def xp_jacobi_refine(head, base, stride_n, stride_b, h_full, anchor, am1, N, K, topc, blk, ws,
                     stream=None):
    _check("xp_jacobi_refine", lib().xp_jacobi_refine(
        head, _ptr(base), stride_n, stride_b, _ptr(h_full), _ptr(anchor), _ptr(am1), N, K, topc,
        _ptr(blk), _ptr(ws), _nbytes(ws), _stream(stream)))


def xp_jacobi_passes(head, base, stride_n, stride_b, xh, am1, N, K, blk, ws, stream=None):
    """K passes on an initialised blk (refined in place), given the hidden cache xh."""
    _check("xp_jacobi_passes", lib().xp_jacobi_passes(
        head, _ptr(base), stride_n, stride_b, _ptr(xh), _ptr(am1), N, K, _ptr(blk), _ptr(ws),
        _nbytes(ws), _stream(stream)))


def xp_set_pass_mode(head, mode: int):
    _check("xp_set_pass_mode", lib().xp_set_pass_mode(head, mode))


def xp_passes_persistent(head, base, stride_n, stride_b, N) -> bool:
    return bool(lib().xp_passes_persistent(head, _ptr(base), stride_n, stride_b, N))


def xp_set_readout_pairs(head, on: bool):
    _check("xp_set_readout_pairs", lib().xp_set_readout_pairs(head, int(on)))


def xp_readout_pairs(head, N) -> bool:
    return bool(lib().xp_readout_pairs(head, N))


def xp_get_error(head, stream=None) -> int:
    """Synchronise the stream, read and clear the device error word; returns the status code."""
    return lib().xp_get_error(head, _stream(stream))


def xp_profile_timeline(head, buf, K: int) -> int:
    """Record the persistent refine's per-CTA phase stamps into buf (None: stop); returns
    the bytes K passes need."""
    needed = ctypes.c_size_t()
    _check("xp_profile_timeline", lib().xp_profile_timeline(head, _ptr(buf), _nbytes(buf), K,
                                                            ctypes.byref(needed)))
    return needed.value


def xp_readout_kernel_name(head) -> str:
    return lib().xp_readout_kernel_name(head).decode()


# ------------------------------------------------------ torch conveniences ---

def torch_dtype(dtype: str):
    import torch
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def to_device(a: np.ndarray, dtype: str, device="cuda"):
    """Storage array from the generator (bf16 as uint16 bits) -> device tensor, bit for bit."""
    import torch
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def to_host_storage(t) -> np.ndarray:
    """Device tensor -> numpy storage form (bf16 as uint16 bits)."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


class Head:
    """Owns a head's prepared device memory (a torch buffer) and its handle."""

    def __init__(self, shape: dict, weights: dict, dtype: str, max_N: int, stream=None):
        import torch
        self.dtype = dtype
        self.code = XP_BF16 if dtype == "bf16" else XP_F32
        self.shape = dict(shape, max_N=max_N)
        self.V, self.hidden, self.r, self.H, self.B = (shape[k] for k in ("V", "hidden", "r", "H", "B"))
        self.max_N = max_N
        w = make_weights(self.V, self.hidden, self.r, self.H, self.B, max_N, self.code, **weights)
        self.prep = torch.empty(xp_head_prep_bytes(w), dtype=torch.uint8, device="cuda")
        self.handle = xp_head_create(w, self.prep, stream)

    def weights_struct(self, **weights) -> xp_weights:
        return make_weights(self.V, self.hidden, self.r, self.H, self.B, self.max_N, self.code,
                            **weights)

    def workspace(self, N: int, topc: int = 0):
        import torch
        w = self.weights_struct()
        return torch.zeros(xp_workspace_bytes(w, N, topc), dtype=torch.uint8, device="cuda")

    def close(self):
        if self.handle:
            xp_head_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def head_from_inputs(inp: dict, wl, max_N: int | None = None, stream=None):
    """Device head from generator output: raw mixer folded on the GPU by xp_fold_mix.

    Returns (Head, dict of the device weight tensors used).
    """
    import torch
    d = wl.dtype
    t = {k: to_device(inp[k], d) for k in ("w1", "down_h", "down_g", "in_proj", "raw_mix",
                                            "w_gate", "w_up", "w_down", "w2")}
    code = XP_BF16 if d == "bf16" else XP_F32
    mix = torch.empty_like(t["raw_mix"])
    xp_fold_mix(t["raw_mix"], mix, wl.r, wl.B, code, stream)
    t["mix_L"] = mix
    shape = dict(V=wl.V, hidden=wl.hidden, r=wl.r, H=wl.H, B=wl.B)
    weights = {k: t[k] for k in ("w1", "down_h", "down_g", "in_proj", "mix_L", "w_gate", "w_up",
                                 "w_down", "w2")}
    head = Head(shape, weights, d, max_N or wl.N, stream)
    return head, t
