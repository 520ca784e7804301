"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (its row statistics live in an array built into the library).

Collected last on purpose: the GPU tests compare it, through the C ABI, with
attn_bwd (which takes a caller workspace) on two calls in a row, and must pass
both alone in a fresh process and after every other test.  Both entry points
run the same kernels on the same row statistics, and the dQ step gives the
same bits under its static deal (the one the built-in scratch uses) as under
its dynamic one, so the results must be equal bit for bit.
"""
import ctypes
import math
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import deterministic_attention_gb300 as da
from deterministic_attention_gb300.inputs import make_inputs
from helpers import assert_bwd_close, to_np, widen

MAX_PAIRS = 1 << 20  # B * Hq * Tp the built-in scratch holds
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_rejects_problems_beyond_the_builtin_scratch():
    """Sizes past the built-in array fail with DETATTN_ERR_WORKSPACE before
    any CUDA call (so this runs without a GPU)."""
    da.build()
    L = da.lib()
    P = ctypes.c_void_p(0x10000)
    # B * Hq * Tp = 2 * 32 * 16384 = 1,048,576 pairs fits; one more batch does not.
    rc = L.attn_bwd_noalloc(P, P, P, P, P, P, P, P, P, 3, 16384, 32, 8, 128, 0.1, 1, None)
    assert rc == -9
    assert "built-in scratch" in da.last_error()
    # T = 129 pads to 256 positions: twice the limit, refused.
    rc = L.attn_bwd_noalloc(P, P, P, P, P, P, P, P, P, 64, 129, 128, 16, 64, 0.1, 1, None)
    assert rc == -9
    assert L.attn_bwd_noalloc(P, P, P, P, P, P, P, P, P, 1, 8, 3, 2, 64, 0.1, 1, None) == -3


def _noalloc(q, k, v, o, lse, do, scale, causal=True):
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = da.lib().attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), _p(dq), _p(dk),
                                   _p(dv), B, T, Hq, Hkv, D, scale, int(causal), stream)
    assert rc == 0, da.last_error()
    torch.cuda.synchronize()
    da.check_status()
    return dq, dk, dv


def _equal_twice(B, T, Hq, Hkv, D, seed, causal=True):
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = (t.cuda() for t in make_inputs(B, T, Hq, Hkv, D, seed=seed, dout_std=0.2))
    o, lse = da.attn_fwd(q, k, v, scale=scale, causal=causal)
    ref = da.attn_bwd(q, k, v, o, lse, do, scale=scale, causal=causal)
    torch.cuda.synchronize()
    for call in range(2):
        got = _noalloc(q, k, v, o, lse, do, scale, causal)
        for name, x, r in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.equal(x, r), f"call {call}: {name} differs from attn_bwd's bits"
    return (q, k, v, do), got


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_twice():
    """D = 64, ragged T: equal to attn_bwd bit for bit on two calls in a row,
    and within the backward tolerance of the fp64 oracle."""
    import oracle
    B, T, Hq, Hkv, D = 2, 700, 6, 2, 64
    (q, k, v, do), (dq, dk, dv) = _equal_twice(B, T, Hq, Hkv, D, seed=99)
    qf, kf, vf, dof = (widen(t.cpu()) for t in (q, k, v, do))
    dq_r, dk_r, dv_r, _, _ = oracle.attn_bwd(qf, kf, vf, dof, 1.0 / math.sqrt(D), True)
    assert_bwd_close([("dQ", to_np(dq.cpu()), dq_r), ("dK", to_np(dk.cpu()), dk_r),
                      ("dV", to_np(dv.cpu()), dv_r)], "noalloc vs oracle")


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_d128():
    _equal_twice(1, 300, 4, 2, 128, seed=98)


@pytest.mark.gpu
def test_noalloc_at_the_scratch_limit():
    """B * Hq * Tp exactly 1,048,576 (64 * 128 * 128, T = 120 padded to 128):
    every pair of the built-in array is in use, still bit-equal."""
    B, T, Hq, Hkv = 64, 120, 128, 16
    assert B * Hq * ((T + 127) // 128 * 128) == MAX_PAIRS
    _equal_twice(B, T, Hq, Hkv, 64, seed=97)


_RESET_SCRIPT = textwrap.dedent(r"""
    # Device memory through the driver API only: a device reset would leave
    # torch's own CUDA state dangling, so torch is used on the CPU alone.
    import ctypes, math, sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    from deterministic_attention_gb300.build import LIB
    from deterministic_attention_gb300.inputs import make_inputs

    cu = ctypes.CDLL("libcuda.so.1")
    L = ctypes.CDLL(LIB)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd.argtypes = [vp] * 5 + [i] * 5 + [f, i, vp]
    L.attn_bwd.argtypes = [vp] * 10 + [sz] + [i] * 5 + [f, i, vp]
    L.attn_bwd_noalloc.argtypes = [vp] * 9 + [i] * 5 + [f, i, vp]
    L.attn_bwd_workspace_bytes.argtypes = [i] * 5
    L.attn_bwd_workspace_bytes.restype = sz
    L.detattn_check_status.argtypes = [vp]
    L.detattn_last_error.restype = ctypes.c_char_p

    def ck(rc, what):
        assert rc == 0, f"{{what}}: {{rc}} {{L.detattn_last_error().decode()}}"

    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int(0)
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")

    def make_current():
        ctx = ctypes.c_void_p()
        ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(ctx), dev), "retain")
        ck(cu.cuCtxSetCurrent(ctx), "set current")

    B, T, Hq, Hkv, D = 1, 333, 4, 2, 64
    scale = 1.0 / math.sqrt(D)
    host = [t.contiguous().view(torch.int16).numpy()
            for t in make_inputs(B, T, Hq, Hkv, D, seed=96, dout_std=0.2)]

    def alloc(nbytes):
        p = ctypes.c_uint64()
        ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(max(nbytes, 16))), "cuMemAlloc")
        return p.value

    def run():
        bufs = []
        def dev_of(a):
            p = alloc(a.nbytes)
            ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(p), a.ctypes.data_as(vp), ctypes.c_size_t(a.nbytes)), "HtoD")
            bufs.append(p)
            return p
        q, k, v, do = (dev_of(a) for a in host)
        nq, nk = host[0].nbytes, host[1].nbytes
        o, lse = alloc(nq), alloc(B * Hq * T * 4)
        outs = [alloc(n) for n in (nq, nk, nk, nq, nk, nk)]
        wsb = L.attn_bwd_workspace_bytes(B, T, Hq, Hkv, D)
        ws = alloc(wsb)
        bufs += [o, lse, ws] + outs
        ck(L.attn_fwd(q, k, v, o, lse, B, T, Hq, Hkv, D, scale, 1, None), "attn_fwd")
        ck(L.attn_bwd(q, k, v, o, lse, do, outs[0], outs[1], outs[2], ws, wsb, B, T, Hq, Hkv, D,
                      scale, 1, None), "attn_bwd")
        ck(L.attn_bwd_noalloc(q, k, v, o, lse, do, outs[3], outs[4], outs[5], B, T, Hq, Hkv, D,
                              scale, 1, None), "attn_bwd_noalloc")
        ck(cu.cuCtxSynchronize(), "sync")
        ck(L.detattn_check_status(None), "status")
        res = []
        for p, n in zip(outs, (nq, nk, nk, nq, nk, nk)):
            a = np.empty(n, dtype=np.uint8)
            ck(cu.cuMemcpyDtoH_v2(a.ctypes.data_as(vp), ctypes.c_uint64(p), ctypes.c_size_t(n)), "DtoH")
            res.append(a)
        for p in bufs:
            ck(cu.cuMemFree_v2(ctypes.c_uint64(p)), "cuMemFree")
        for a, b in zip(res[:3], res[3:]):
            assert np.array_equal(a, b), "noalloc differs from attn_bwd"
        return res

    make_current()
    before = run()
    ck(cu.cuDevicePrimaryCtxReset_v2(dev), "primary context reset")
    make_current()
    after = run()
    for a, b in zip(before, after):
        assert np.array_equal(a, b), "results changed across the device reset"
    print("reset ok")
""")


@pytest.mark.gpu
def test_noalloc_after_device_reset():
    """After a device reset the library's module (and its built-in array) is
    loaded again in a new context: the entry point must look the array's
    address up again instead of writing through the old one.  Runs in its own
    process, which holds device memory through the driver API only (the reset
    discards every device allocation and torch's CUDA state with them)."""
    code = _RESET_SCRIPT.format(root=ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "reset ok" in r.stdout, r.stdout + r.stderr
