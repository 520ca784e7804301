"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (its row statistics live in an array built into the library).

Collected last on purpose: the GPU test compares it, through the C ABI, with
attn_bwd (which takes a caller workspace) on two calls in a row, and must pass
both alone in a fresh process and after every other test.
"""
import ctypes
import math

import pytest
import torch

import deterministic_attention_gb300 as da
from deterministic_attention_gb300.inputs import make_inputs
from helpers import TOL_BWD_REL, rel_l2, to_np

MAX_PAIRS = 1 << 20  # B * Hq * Tp the built-in scratch holds


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
    assert L.attn_bwd_noalloc(P, P, P, P, P, P, P, P, P, 1, 8, 3, 2, 64, 0.1, 1, None) == -3


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_twice():
    B, T, Hq, Hkv, D = 2, 700, 6, 2, 64
    scale = 1.0 / math.sqrt(D)
    q, k, v, do = (t.cuda() for t in make_inputs(B, T, Hq, Hkv, D, seed=99, dout_std=0.2))
    o, lse = da.attn_fwd(q, k, v, scale=scale)
    ref = da.attn_bwd(q, k, v, o, lse, do, scale=scale)
    torch.cuda.synchronize()
    L = da.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in ref)
        rc = L.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), _p(dq), _p(dk),
                                _p(dv), B, T, Hq, Hkv, D, scale, 1, stream)
        assert rc == 0, da.last_error()
        torch.cuda.synchronize()
        da.check_status()
        for name, x, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert torch.isfinite(x.float()).all(), f"call {call}: non-finite {name}"
            err = rel_l2(to_np(x.cpu()), to_np(r.cpu()))
            assert err <= TOL_BWD_REL, f"call {call}: {name} rel-L2 {err:.3g}"
