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
           "set_dkdv_split", "set_dkdv_deal", "new_workspace", "rowstats_view", "last_error", "lib",
           "DetAttnError", "STATUS", "header_symbols", "build", "embed_grad",
           "embed_grad_workspace_bytes", "attn_fwd_varlen", "attn_bwd_varlen",
           "varlen_workspace_bytes", "layer_gemm", "layer_workspace_bytes", "LayerState",
           "layer_train_step", "ds_workspace_bytes", "set_bwd_dq_mode"]

STATUS = {0: "DETATTN_OK", -1: "DETATTN_ERR_NULL", -2: "DETATTN_ERR_ALIGN",
          -3: "DETATTN_ERR_SHAPE", -4: "DETATTN_ERR_HEADDIM", -5: "DETATTN_ERR_SCALE",
          -6: "DETATTN_ERR_CUDA", -7: "DETATTN_ERR_DEVICE_TIMEOUT", -8: "DETATTN_ERR_ARCH",
          -9: "DETATTN_ERR_WORKSPACE", -10: "DETATTN_ERR_INDEX"}

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
    L.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, fp, vp, vp, i, i, i, i, f, i, vp]
    L.attn_fwd_varlen.restype = i
    L.attn_bwd_varlen_workspace_bytes.argtypes = [vp, vp, i, i, i, i]
    L.attn_bwd_varlen_workspace_bytes.restype = sz
    L.attn_bwd_varlen.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, vp, sz, vp, vp, i, i, i, i, f,
                                  i, vp]
    L.attn_bwd_varlen.restype = i
    L.attn_bwd_ds_workspace_bytes.argtypes = [i, i, i, i, i, i]
    L.attn_bwd_ds_workspace_bytes.restype = sz
    L.detattn_set_bwd_dq_mode.argtypes = [i]
    L.detattn_set_bwd_dq_mode.restype = i
    L.layer_gemm.argtypes = [vp, i, i, vp, i, i, vp, i, i, i, i, i, f, vp]
    L.layer_gemm.restype = i
    L.layer_workspace_bytes.argtypes = [i, i, i, i, i, i]
    L.layer_workspace_bytes.restype = sz
    L.layer_train_step.argtypes = [vp] * 15 + [sz] + [i] * 7 + [f] * 5 + [vp]
    L.layer_train_step.restype = i
    L.embed_grad_workspace_bytes.argtypes = [i, i, i]
    L.embed_grad_workspace_bytes.restype = sz
    L.embed_grad.argtypes = [vp, vp, vp, vp, sz, i, i, i, vp]
    L.embed_grad.restype = i
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
    L.detattn_diag_dkdv_list.argtypes = [i, i, i, i, i, i, i, i, vp, vp, i]
    L.detattn_diag_dkdv_list.restype = i
    L.detattn_set_dkdv_deal.argtypes = [i]
    L.detattn_set_dkdv_deal.restype = i
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


def ds_workspace_bytes(B, T, Hq, Hkv, D, causal=True) -> int:
    return int(lib().attn_bwd_ds_workspace_bytes(B, T, Hq, Hkv, D, int(bool(causal))))


def new_workspace(B, T, Hq, Hkv, D, device="cuda", stored_ds=False, causal=True):
    """A device workspace (uint8) of attn_bwd_workspace_bytes, or with
    stored_ds of attn_bwd_ds_workspace_bytes (the stored-dS backward)."""
    n = ds_workspace_bytes(B, T, Hq, Hkv, D, causal) if stored_ds else 0
    if n == 0:
        n = workspace_bytes(B, T, Hq, Hkv, D)
    return torch.empty((max(16, n),), dtype=torch.uint8, device=device)


def set_bwd_dq_mode(mode: int):
    """0 (default): the dQ step recomputes S and dP; 1: stored-dS backward
    whenever the workspace holds it (new_workspace(..., stored_ds=True))."""
    _check(lib().detattn_set_bwd_dq_mode(int(mode)), "detattn_set_bwd_dq_mode")


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


def _host_cu(cu):
    """Offsets as a contiguous host int32 array (kept alive by the caller)."""
    import numpy as np
    if isinstance(cu, torch.Tensor):
        cu = cu.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(cu, dtype=np.int32).reshape(-1))


def varlen_workspace_bytes(cu_q, cu_k, Hq, Hkv, D) -> int:
    cq, ck = _host_cu(cu_q), _host_cu(cu_k)
    return int(lib().attn_bwd_varlen_workspace_bytes(ctypes.c_void_p(cq.ctypes.data),
                                                     ctypes.c_void_p(ck.ctypes.data),
                                                     cq.size - 1, Hq, Hkv, D))


def attn_fwd_varlen(q, k, v, cu_q, cu_k, scale=None, causal=True, out=None, lse=None):
    """Packed variable-length forward: q [total_q, Hq, D], k, v [total_k, Hkv,
    D]; sequence s is query rows cu_q[s]..cu_q[s+1]-1 and key rows
    cu_k[s]..cu_k[s+1]-1 (cu_q, cu_k on the host).  Returns o [total_q, Hq,
    D] and lse fp32 [Hq, total_q] (-inf for rows that see no key)."""
    Nq, Hq, D = q.shape
    Nk, Hkv = k.shape[0], k.shape[1]
    bf = torch.bfloat16
    _need(q, "q", bf, (Nq, Hq, D))
    _need(k, "k", bf, (Nk, Hkv, D))
    _need(v, "v", bf, (Nk, Hkv, D))
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((Hq, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(o, "o", bf, (Nq, Hq, D))
    _need(l, "lse", torch.float32, (Hq, Nq))
    cq, ck = _host_cu(cu_q), _host_cu(cu_k)
    rc = lib().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l),
                               ctypes.c_void_p(cq.ctypes.data), ctypes.c_void_p(ck.ctypes.data),
                               cq.size - 1, Hq, Hkv, D, _scale(scale, D), int(bool(causal)),
                               _stream())
    _check(rc, "attn_fwd_varlen")
    return o, l


def attn_bwd_varlen(q, k, v, o, lse, dout, cu_q, cu_k, scale=None, causal=True, dq=None,
                    dk=None, dv=None, workspace=None):
    """Packed variable-length backward: (dq, dk, dv) in the layouts of q, k, v."""
    Nq, Hq, D = q.shape
    Nk, Hkv = k.shape[0], k.shape[1]
    bf = torch.bfloat16
    for t, n, shp in ((q, "q", (Nq, Hq, D)), (k, "k", (Nk, Hkv, D)), (v, "v", (Nk, Hkv, D)),
                      (o, "o", (Nq, Hq, D)), (dout, "dout", (Nq, Hq, D))):
        _need(t, n, bf, shp)
    _need(lse, "lse", torch.float32, (Hq, Nq))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    cq, ck = _host_cu(cu_q), _host_cu(cu_k)
    if workspace is None:
        workspace = torch.empty((max(16, varlen_workspace_bytes(cq, ck, Hq, Hkv, D)),),
                                dtype=torch.uint8, device=q.device)
    rc = lib().attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                               _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
                               ctypes.c_void_p(cq.ctypes.data), ctypes.c_void_p(ck.ctypes.data),
                               cq.size - 1, Hq, Hkv, D, _scale(scale, D), int(bool(causal)),
                               _stream())
    _check(rc, "attn_bwd_varlen")
    return dq, dk, dv


def layer_gemm(a, b, a_mn_major=False, b_mn_major=True, out=None, out_fp32=False, alpha=1.0):
    """C = alpha A B on the tensor cores (bf16 in, fp32 accumulation).  a is
    [M, K] (or, with a_mn_major, stored transposed as [K, M]); b is [K, N]
    with b_mn_major (the default, row-major B) or stored transposed [N, K]."""
    M, K = (a.shape[1], a.shape[0]) if a_mn_major else tuple(a.shape)
    N = b.shape[1] if b_mn_major else b.shape[0]
    if (b.shape[0] if b_mn_major else b.shape[1]) != K:
        raise ValueError(f"inner dimensions differ: a {tuple(a.shape)}, b {tuple(b.shape)}")
    _need(a, "a", torch.bfloat16, tuple(a.shape))
    _need(b, "b", torch.bfloat16, tuple(b.shape))
    dt = torch.float32 if out_fp32 else torch.bfloat16
    c = torch.empty((M, N), dtype=dt, device=a.device) if out is None else out
    _need(c, "c", dt, (M, N))
    _check(lib().layer_gemm(_ptr(a), int(a_mn_major), a.shape[1], _ptr(b), int(b_mn_major),
                            b.shape[1], _ptr(c), int(out_fp32), N, M, N, K, float(alpha),
                            _stream()), "layer_gemm")
    return c


def layer_workspace_bytes(B, T, d, Hq, Hkv, D) -> int:
    return int(lib().layer_workspace_bytes(B, T, d, Hq, Hkv, D))


class LayerState:
    """Device state of one attention layer under AdamW: fp32 master weights
    w_qkv [d, (Hq + 2 Hkv) D] (= [Wq | Wk | Wv]) and w_o [Hq D, d], their
    moments, bf16 copies, gradient buffers and the step workspace."""

    def __init__(self, wq, wk, wv, wo, B, T, Hq, Hkv, D, device="cuda"):
        d = wq.shape[0]
        self.dims = (B, T, d, Hq, Hkv, D)
        f32 = dict(dtype=torch.float32, device=device)
        self.w_qkv = torch.cat([wq, wk, wv], dim=1).to(**f32).contiguous()
        self.w_o = wo.to(**f32).contiguous()
        self.m_qkv, self.v_qkv = torch.zeros_like(self.w_qkv), torch.zeros_like(self.w_qkv)
        self.m_o, self.v_o = torch.zeros_like(self.w_o), torch.zeros_like(self.w_o)
        self.w_qkv_bf16 = self.w_qkv.to(torch.bfloat16)
        self.w_o_bf16 = self.w_o.to(torch.bfloat16)
        self.g_qkv, self.g_o = torch.empty_like(self.w_qkv), torch.empty_like(self.w_o)
        self.y = torch.empty((B, T, d), dtype=torch.bfloat16, device=device)
        self.dx = torch.empty((B, T, d), dtype=torch.bfloat16, device=device)
        self.workspace = torch.empty((layer_workspace_bytes(*self.dims),), dtype=torch.uint8,
                                     device=device)
        self.step = 0


def layer_train_step(state, x, dy, lr=3e-4, weight_decay=0.1, beta1=0.9, beta2=0.999, eps=1e-8,
                     with_dx=True):
    """One training step of the layer on (x, dy), then AdamW; returns
    (g_qkv, g_o) of this step (the state's buffers)."""
    B, T, d, Hq, Hkv, D = state.dims
    _need(x, "x", torch.bfloat16, (B, T, d))
    _need(dy, "dy", torch.bfloat16, (B, T, d))
    state.step += 1
    s = state
    _check(lib().layer_train_step(_ptr(x), _ptr(dy), _ptr(s.w_qkv), _ptr(s.w_o), _ptr(s.m_qkv),
                                  _ptr(s.v_qkv), _ptr(s.m_o), _ptr(s.v_o), _ptr(s.w_qkv_bf16),
                                  _ptr(s.w_o_bf16), _ptr(s.g_qkv), _ptr(s.g_o), _ptr(s.y),
                                  _ptr(s.dx) if with_dx else None, _ptr(s.workspace),
                                  s.workspace.numel(), B, T, d, Hq, Hkv, D, s.step, float(lr),
                                  float(weight_decay), float(beta1), float(beta2), float(eps),
                                  _stream()), "layer_train_step")
    return s.g_qkv, s.g_o


def embed_grad_workspace_bytes(N, V, E) -> int:
    return int(lib().embed_grad_workspace_bytes(N, V, E))


def embed_grad(ids, dy, V, dw=None, workspace=None):
    """Deterministic embedding-lookup gradient: dw fp32 [V, E] with
    dw[v] = sum of dy[t] over tokens t with ids[t] == v (include/detattn.h)."""
    if ids.dim() != 1 or dy.dim() != 2:
        raise ValueError("ids must be [N] and dy [N, E]")
    N, E = dy.shape
    _need(ids, "ids", torch.int32, (N,))
    _need(dy, "dy", torch.bfloat16, (N, E))
    dw = torch.empty((V, E), dtype=torch.float32, device=dy.device) if dw is None else dw
    _need(dw, "dw", torch.float32, (V, E))
    if workspace is None:
        workspace = torch.empty((max(16, embed_grad_workspace_bytes(N, V, E)),), dtype=torch.uint8,
                                device=dy.device)
    _check(lib().embed_grad(_ptr(ids), _ptr(dy), _ptr(dw), _ptr(workspace), workspace.numel(), N,
                            V, E, _stream()), "embed_grad")
    return dw


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


def diag_dkdv_list(B, T, Hq, Hkv, causal, c, ng, force=False):
    """The listed deal of the 64-dim dK/dV step's key tiles over ng clusters
    of c blocks: a list, per block, of (tile, shared) pairs, or None where
    the plain walk is used (see include/detattn.h); host-only."""
    import numpy as np
    nb = ng * c
    start = np.zeros(nb + 1, dtype=np.int32)
    cap = 4096
    entry = np.zeros(cap, dtype=np.int32)
    rc = lib().detattn_diag_dkdv_list(B, T, Hq, Hkv, int(bool(causal)), c, ng, int(bool(force)),
                                      ctypes.c_void_p(start.ctypes.data),
                                      ctypes.c_void_p(entry.ctypes.data), cap)
    if rc < 0:
        raise DetAttnError(rc, "detattn_diag_dkdv_list", last_error())
    if rc == 0:
        return None
    return [[(int(e) >> 1, bool(e & 1)) for e in entry[start[i]:start[i + 1]]] for i in range(nb)]


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


def set_dkdv_deal(mode: int):
    """dK/dV key-tile deal at D = 64: 0 automatic, 1 plain walk, 2 listed deal."""
    _check(lib().detattn_set_dkdv_deal(int(mode)), "detattn_set_dkdv_deal")


def set_wait_limit_ns(ns: int):
    lib().detattn_set_wait_limit_ns(int(ns))
