"""Deterministic causal grouped-query flash attention on sm_103a (GB300).

Thin Python binding over the C-ABI library ``libdetattn.so`` (declared in
``include/detattn.h``).  This module only marshals arguments: every step of
the forward and backward runs in the library's CUDA kernels.  PyTorch is used
for device memory and the current stream.  There is no CPU fallback: if the
library is missing or the device is not sm_103, calls raise.

Layouts: q, o, dout, dq are bf16 [B, T, Hq, D]; k, v, dk, dv are bf16
[B, T, Hkv, D]; lse is fp32 [B, Hq, T] (natural log).
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

from .build import LIB as _LIB_PATH, build  # noqa: F401

__all__ = ["attn_fwd", "attn_bwd", "attn_bwd_delta", "attn_bwd_dkdv", "attn_bwd_dq",
           "workspace_bytes", "check_status", "set_wait_limit_ns", "selftest_wait_timeout",
           "set_dkdv_split", "new_workspace", "rowstats_view", "last_error", "lib",
           "DetAttnError", "STATUS", "header_symbols", "build"]

STATUS = {0: "DETATTN_OK", -1: "DETATTN_ERR_NULL", -2: "DETATTN_ERR_ALIGN",
          -3: "DETATTN_ERR_SHAPE", -4: "DETATTN_ERR_HEADDIM", -5: "DETATTN_ERR_SCALE",
          -6: "DETATTN_ERR_CUDA", -7: "DETATTN_ERR_DEVICE_TIMEOUT", -8: "DETATTN_ERR_ARCH",
          -9: "DETATTN_ERR_WORKSPACE"}

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "detattn.h")


class DetAttnError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}: {msg}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library with argument types set (raises if not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is not built; call deterministic_attention_gb300.build()")
    L = ctypes.CDLL(_LIB_PATH)
    vp, fp, i, f, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd.argtypes = [vp, vp, vp, vp, fp, i, i, i, i, i, f, i, vp]
    L.attn_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
    L.attn_bwd_workspace_bytes.restype = sz
    L.attn_bwd.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, vp]
    L.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    L.attn_bwd_noalloc.restype = i
    L.attn_bwd_delta.argtypes = [vp, vp, fp, vp, sz, i, i, i, i, vp]
    L.attn_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, sz, vp, vp, i, i, i, i, i, f, i, vp]
    L.attn_bwd_dq.argtypes = [vp, vp, vp, vp, vp, sz, vp, i, i, i, i, i, f, i, vp]
    L.detattn_check_status.argtypes = [vp]
    L.detattn_diag_exp2.argtypes = [vp, vp, vp, vp, i, vp]
    L.detattn_diag_exp2.restype = i
    L.detattn_diag_qtile_deal.argtypes = [i, i, i, i, i, i, vp, i]
    L.detattn_diag_qtile_deal.restype = i
    L.detattn_diag_dkdv_split.argtypes = [i, i, i, i, i, i, vp, i, vp, vp]
    L.detattn_diag_dkdv_split.restype = i
    L.detattn_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, vp]
    L.detattn_selftest_wait_timeout.restype = i
    L.detattn_set_dkdv_split.argtypes = [i]
    L.detattn_set_dkdv_split.restype = i
    L.detattn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    L.detattn_set_wait_limit_ns.restype = None
    L.detattn_last_error.argtypes = []
    L.detattn_last_error.restype = ctypes.c_char_p
    L.detattn_version.argtypes = []
    for name in ("attn_fwd", "attn_bwd", "attn_bwd_delta", "attn_bwd_dkdv", "attn_bwd_dq",
                 "detattn_check_status", "detattn_version"):
        getattr(L, name).restype = i
    _lib = L
    return L


def header_symbols() -> list[str]:
    """Function names declared in include/detattn.h."""
    text = open(HEADER).read()
    return re.findall(r"^\s*(?:int|size_t|void|const char\*)\s+(\w+)\s*\(", text, re.M)


def last_error() -> str:
    return lib().detattn_last_error().decode()


def _check(rc: int, where: str):
    if rc != 0:
        raise DetAttnError(rc, where, last_error())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, name, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be 4-D [B, T, H, D]")
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    return B, T, Hq, Hkv, D


def _scale(scale, D):
    return float(1.0 / math.sqrt(D) if scale is None else scale)


def attn_fwd(q, k, v, scale=None, causal=True, out=None, lse=None):
    """Forward: returns (o bf16 [B,T,Hq,D], lse fp32 [B,Hq,T])."""
    B, T, Hq, Hkv, D = _dims(q, k)
    bf = torch.bfloat16
    _need(q, "q", bf, (B, T, Hq, D))
    _need(k, "k", bf, (B, T, Hkv, D))
    _need(v, "v", bf, (B, T, Hkv, D))
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "o", bf, (B, T, Hq, D))
    _need(l, "lse", torch.float32, (B, Hq, T))
    rc = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, T, Hq, Hkv, D,
                        _scale(scale, D), int(bool(causal)), _stream())
    _check(rc, "attn_fwd")
    return o, l


def workspace_bytes(B, T, Hq, Hkv, D) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, T, Hq, Hkv, D))


def attn_bwd(q, k, v, o, lse, dout, scale=None, causal=True, dq=None, dk=None, dv=None,
             workspace=None):
    """Backward: returns (dq, dk, dv), bf16, in the layouts of q, k, v."""
    B, T, Hq, Hkv, D = _dims(q, k)
    bf = torch.bfloat16
    for t, n, s in ((q, "q", (B, T, Hq, D)), (k, "k", (B, T, Hkv, D)), (v, "v", (B, T, Hkv, D)),
                    (o, "o", (B, T, Hq, D)), (dout, "dout", (B, T, Hq, D))):
        _need(t, n, bf, s)
    _need(lse, "lse", torch.float32, (B, Hq, T))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need(dq, "dq", bf, (B, T, Hq, D))
    _need(dk, "dk", bf, (B, T, Hkv, D))
    _need(dv, "dv", bf, (B, T, Hkv, D))
    if workspace is None:
        workspace = new_workspace(B, T, Hq, Hkv, D, q.device)
    rc = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                        _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, T, Hq, Hkv, D,
                        _scale(scale, D), int(bool(causal)), _stream())
    _check(rc, "attn_bwd")
    return dq, dk, dv


def new_workspace(B, T, Hq, Hkv, D, device="cuda"):
    """A device workspace of attn_bwd_workspace_bytes (uint8)."""
    return torch.empty((max(16, workspace_bytes(B, T, Hq, Hkv, D)),), dtype=torch.uint8,
                       device=device)


def rowstats_view(workspace, B, T, Hq):
    """The workspace's row statistics as fp32 [B, Hq, Tp, 2]:
    [..., 0] = -LSE*log2(e), [..., 1] = -Delta (see include/detattn.h)."""
    Tp = (T + 127) // 128 * 128
    return workspace[: B * Hq * Tp * 8].view(torch.float32).view(B, Hq, Tp, 2)


def attn_bwd_delta(o, dout, lse, workspace):
    """Backward step 1: row statistics (from o, dout, lse) into `workspace`."""
    B, T, Hq, D = o.shape
    _need(o, "o", torch.bfloat16, (B, T, Hq, D))
    _need(dout, "dout", torch.bfloat16, (B, T, Hq, D))
    _need(lse, "lse", torch.float32, (B, Hq, T))
    _check(lib().attn_bwd_delta(_ptr(o), _ptr(dout), _ptr(lse), _ptr(workspace), workspace.numel(),
                                B, T, Hq, D, _stream()), "attn_bwd_delta")
    return workspace


def attn_bwd_dkdv(q, k, v, dout, workspace, scale=None, causal=True, dk=None, dv=None):
    """Backward step 2: dk, dv from the row statistics in `workspace`."""
    B, T, Hq, Hkv, D = _dims(q, k)
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().attn_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(workspace),
                               workspace.numel(), _ptr(dk), _ptr(dv), B, T, Hq, Hkv, D,
                               _scale(scale, D), int(bool(causal)), _stream()), "attn_bwd_dkdv")
    return dk, dv


def attn_bwd_dq(q, k, v, dout, workspace, scale=None, causal=True, dq=None):
    """Backward step 3: dq from the row statistics in `workspace`."""
    B, T, Hq, Hkv, D = _dims(q, k)
    dq = torch.empty_like(q) if dq is None else dq
    _check(lib().attn_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(workspace),
                             workspace.numel(), _ptr(dq), B, T, Hq, Hkv, D, _scale(scale, D),
                             int(bool(causal)), _stream()), "attn_bwd_dq")
    return dq


def check_status():
    """Synchronises the current stream and raises if a kernel timed out."""
    _check(lib().detattn_check_status(_stream()), "detattn_check_status")


def diag_qtile_deal(D, B, T, Hq, causal, sms):
    """(number of pipelines, numpy int32 pipeline of each unit) of the static
    query-tile deal; host-only, no GPU needed."""
    import numpy as np
    n = B * Hq * -(-T // 128) if B > 0 and T > 0 else 0
    out = np.empty(max(1, n), dtype=np.int32)
    rc = lib().detattn_diag_qtile_deal(D, B, T, Hq, int(bool(causal)), sms,
                                       ctypes.c_void_p(out.ctypes.data), n)
    if rc < 0:
        raise DetAttnError(rc, "detattn_diag_qtile_deal", last_error())
    return rc, out[:n]


def diag_dkdv_split(B, T, Hq, Hkv, D, causal, resident, blocks_per_key_tile=0):
    """(C, NG) the dK/dV step would choose on a device holding resident[i]
    clusters of 2**i blocks (i = 0..3); host-only, no GPU needed."""
    import numpy as np
    res = np.zeros(4, dtype=np.int32)
    res[:len(resident)] = resident
    c, ng = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().detattn_diag_dkdv_split(B, T, Hq, Hkv, D, int(bool(causal)),
                                       ctypes.c_void_p(res.ctypes.data), blocks_per_key_tile,
                                       ctypes.byref(c), ctypes.byref(ng))
    if rc < 0:
        raise DetAttnError(rc, "detattn_diag_dkdv_split", last_error())
    return c.value, ng.value


def diag_exp2(x):
    """(poly, poly pair form, special-function unit) 2^x of a float32 CUDA tensor."""
    _need(x, "x", torch.float32, tuple(x.shape))
    ys = [torch.empty_like(x) for _ in range(3)]
    _check(lib().detattn_diag_exp2(_ptr(x), _ptr(ys[0]), _ptr(ys[1]), _ptr(ys[2]), x.numel(),
                                   _stream()), "detattn_diag_exp2")
    return tuple(ys)


def selftest_wait_timeout(limit_ns: int = 50_000_000):
    """Runs the device-side bounded-wait self-test (see include/detattn.h)."""
    _check(lib().detattn_selftest_wait_timeout(int(limit_ns), _stream()),
           "detattn_selftest_wait_timeout")


def set_dkdv_split(blocks_per_key_tile: int):
    """Forces the dK/dV split (1, 2, 4, 8) or restores automatic (0)."""
    _check(lib().detattn_set_dkdv_split(int(blocks_per_key_tile)), "detattn_set_dkdv_split")


def set_wait_limit_ns(ns: int):
    lib().detattn_set_wait_limit_ns(int(ns))
