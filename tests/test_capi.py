"""The C-ABI boundary without a GPU: the library builds and loads, exports
every function include/detattn.h declares, and rejects invalid arguments with
the documented status codes before any CUDA call (so no device is needed)."""
import ctypes
import math

import pytest

import deterministic_attention_gb300 as da


@pytest.fixture(scope="module")
def L():
    da.build()
    return da.lib()


def test_exports_every_declared_symbol(L):
    names = da.header_symbols()
    assert set(names) >= {"attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_bwd_delta",
                          "attn_bwd_dkdv", "attn_bwd_dq", "detattn_check_status",
                          "detattn_set_wait_limit_ns", "detattn_last_error", "detattn_version"}
    for n in names:
        assert hasattr(L, n), n


def test_dkdv_split_knob_validates(L):
    for ok in (0, 1, 2, 4, 8):
        assert L.detattn_set_dkdv_split(ok) == 0
    for bad in (-1, 3, 16):
        assert L.detattn_set_dkdv_split(bad) == -3
    assert L.detattn_set_dkdv_split(0) == 0


def test_version(L):
    assert L.detattn_version() == 10000


P = ctypes.c_void_p(0x10000)       # 16-byte aligned stand-in pointer (never dereferenced)
BAD = ctypes.c_void_p(0x10008)     # misaligned


def _fwd(L, q=P, k=P, v=P, o=P, lse=P, B=1, T=128, Hq=2, Hkv=1, D=64, scale=0.125, causal=1):
    return L.attn_fwd(q, k, v, o, lse, B, T, Hq, Hkv, D, scale, causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(lse=None), -1),
    (dict(v=BAD), -2), (dict(o=BAD), -2),
    (dict(B=-1), -3), (dict(T=-5), -3), (dict(Hq=3, Hkv=2), -3), (dict(Hkv=0), -3),
    (dict(D=96), -4), (dict(D=32), -4), (dict(D=256), -4),
    (dict(scale=0.0), -5), (dict(scale=-1.0), -5), (dict(scale=math.inf), -5),
    (dict(scale=math.nan), -5), (dict(causal=2), -5),
])
def test_fwd_rejects(L, kw, code):
    assert _fwd(L, **kw) == code
    assert da.last_error() != ""


def test_empty_problem_is_ok_without_device(L):
    assert _fwd(L, q=None, k=None, v=None, o=None, lse=None, B=0) == 0
    assert _fwd(L, T=0, q=None) == 0


def test_workspace_bytes(L):
    # Row statistics rounded up to 256 bytes, then 256 bytes for the dQ step's
    # tile counter.
    assert L.attn_bwd_workspace_bytes(4, 1024, 12, 4, 64) == 4 * 12 * 1024 * 8 + 256
    assert L.attn_bwd_workspace_bytes(1, 3, 1, 1, 64) == 128 * 8 + 256
    assert L.attn_bwd_workspace_bytes(2, 129, 3, 1, 128) == 2 * 3 * 256 * 8 + 256
    assert L.attn_bwd_workspace_bytes(1, 1, 1, 1, 64) == 1024 + 256
    assert L.attn_bwd_workspace_bytes(1, 3, 3, 2, 64) == 0
    assert L.attn_bwd_workspace_bytes(0, 3, 2, 1, 64) == 0


def test_bwd_rejects(L):
    args = [P] * 10
    def call(ws=P, wsb=1 << 20, **kw):
        a = dict(B=1, T=128, Hq=2, Hkv=1, D=64, scale=0.125, causal=1)
        a.update(kw)
        v = list(args)
        v[9] = ws
        return L.attn_bwd(*v, wsb, a["B"], a["T"], a["Hq"], a["Hkv"], a["D"], a["scale"],
                          a["causal"], None)
    assert call(ws=None) == -9
    assert call(wsb=100) == -9
    assert call(ws=BAD) == -2
    assert call(D=80) == -4
    assert call(Hq=5, Hkv=2) == -3
    assert L.attn_bwd_dq(P, P, P, P, P, 1 << 20, None, 1, 128, 2, 1, 64, 0.125, 1, None) == -1
    assert L.attn_bwd_dq(P, P, P, P, P, 100, P, 1, 128, 2, 1, 64, 0.125, 1, None) == -9
    assert L.attn_bwd_dkdv(P, P, P, P, P, 1 << 20, P, BAD, 1, 128, 2, 1, 64, 0.125, 1, None) == -2
    assert L.attn_bwd_dkdv(P, P, P, P, None, 1 << 20, P, P, 1, 128, 2, 1, 64, 0.125, 1, None) == -9
    assert L.attn_bwd_delta(P, P, None, P, 1 << 20, 1, 128, 2, 64, None) == -1
    assert L.attn_bwd_delta(P, P, P, BAD, 1 << 20, 1, 128, 2, 64, None) == -2


def test_python_binding_refuses_cpu_tensors(L):
    import torch
    q = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        da.attn_fwd(q, q[:, :, :1], q[:, :, :1])
