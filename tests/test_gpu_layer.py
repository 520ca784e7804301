"""GPU parity of the training micro-loop's kernels (layer_gemm, the rotary
split/merge and AdamW inside layer_train_step) against the fp64 oracle
(numpy products and oracle.layer), and SHA-256 identity of the weight
gradients at every step.

Tolerances, from the arithmetic:
* layer_gemm with fp32 output sums K products of bf16 numbers (exact in
  fp32) in fp32: relative error about sqrt(K) 2^-24, so rel-L2 <= 1e-5; a
  bf16 output adds one rounding (2^-9): rel-L2 <= 4e-3.
* The layer step rounds its intermediates to bf16 (QKV, rotated Q and K, O,
  dO, the joined projection gradient) and runs the attention kernels, whose
  own bar is rel-L2 <= 1e-2 for dQ, dK, dV: the weight gradients and dX are
  held to rel-L2 <= 1e-2, Y to 5e-3.
* After N AdamW steps the fp32 master weights are compared with the oracle's
  fp64 ones.  AdamW divides each gradient element by its own running
  magnitude, so an element whose gradient lies within the bf16 noise can take
  the opposite step (2 lr apart); the test bounds the rel-L2 of the weights
  (<= 1e-2) and of their total update (<= 0.25).
"""
import hashlib
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import deterministic_attention_gb300 as da
from deterministic_attention_gb300.inputs import LAYER_PAGE3, make_layer_inputs
from helpers import rel_l2, to_np, widen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


@pytest.mark.gpu
@pytest.mark.parametrize("a_mn,b_mn", [(False, True), (False, False), (True, True), (True, False)])
@pytest.mark.parametrize("out_fp32", [False, True])
def test_gemm_matches_fp64_product(a_mn, b_mn, out_fp32):
    M, N, K = 384, 256, 640
    a = _bf16((K, M) if a_mn else (M, K), 1)
    b = _bf16((K, N) if b_mn else (N, K), 2)
    ref = (widen(a).T if a_mn else widen(a)) @ (widen(b) if b_mn else widen(b).T)
    c = da.layer_gemm(a.cuda(), b.cuda(), a_mn_major=a_mn, b_mn_major=b_mn, out_fp32=out_fp32,
                      alpha=0.5)
    c2 = da.layer_gemm(a.cuda(), b.cuda(), a_mn_major=a_mn, b_mn_major=b_mn, out_fp32=out_fp32,
                       alpha=0.5)
    torch.cuda.synchronize()
    da.check_status()
    assert torch.equal(c, c2)
    err = rel_l2(to_np(c.cpu()), 0.5 * ref)
    assert err <= (1e-5 if out_fp32 else 4e-3), err


def _oracle_grads(x, wq, wk, wv, wo, dy, Hq, Hkv, D):
    from oracle import layer
    f = lambda t: widen(t) if t.dtype == torch.bfloat16 else t.double().numpy()
    y, _ = layer.layer_forward(f(x), f(wq), f(wk), f(wv), f(wo), Hq, Hkv, D)
    dx, dwq, dwk, dwv, dwo = layer.layer_backward(f(x), f(wq), f(wk), f(wv), f(wo), f(dy), Hq, Hkv, D)
    return y, dx, np.concatenate([dwq, dwk, dwv], axis=1), dwo


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(2, 256, 256, 4, 2, 64), (1, 384, 256, 2, 1, 128)])
def test_layer_step_gradients_match_oracle(shape):
    B, T, d, Hq, Hkv, D = shape
    x, wq, wk, wv, wo, dy = make_layer_inputs(B, T, d, Hq, Hkv, D, seed=31)
    st = da.LayerState(wq, wk, wv, wo, B, T, Hq, Hkv, D)
    g_qkv, g_o = da.layer_train_step(st, x.cuda(), dy.cuda())
    torch.cuda.synchronize()
    da.check_status()
    y_r, dx_r, gqkv_r, go_r = _oracle_grads(x, wq, wk, wv, wo, dy, Hq, Hkv, D)
    assert rel_l2(to_np(st.y.cpu()), y_r) <= 5e-3
    for name, got, ref in (("g_qkv", g_qkv, gqkv_r), ("g_o", g_o, go_r), ("dX", st.dx, dx_r)):
        err = rel_l2(to_np(got.cpu()), ref)
        assert err <= 1e-2, f"{name} rel-L2 {err:.3g}"


def _digest(t):
    return hashlib.sha256(t.contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()


def _page3_loop(n_steps):
    """The page-3 layer for n_steps with inputs drawn per step (seed 7 + t);
    returns per-step gradient digests, the last step's state and inputs."""
    w = LAYER_PAGE3
    B, T, d, Hq, Hkv, D = (w[k] for k in ("B", "T", "d", "Hq", "Hkv", "D"))
    _, wq, wk, wv, wo, _ = make_layer_inputs(B, T, d, Hq, Hkv, D, seed=w["seed"])
    st = da.LayerState(wq, wk, wv, wo, B, T, Hq, Hkv, D)
    digests, steps = [], []
    for t in range(n_steps):
        x, _, _, _, _, dy = make_layer_inputs(B, T, d, Hq, Hkv, D, seed=w["seed"] + 1 + t)
        g_qkv, g_o = da.layer_train_step(st, x.cuda(), dy.cuda())
        torch.cuda.synchronize()
        digests.append((_digest(g_qkv[:, :Hq * D]), _digest(g_qkv[:, Hq * D:(Hq + Hkv) * D]),
                        _digest(g_qkv[:, (Hq + Hkv) * D:]), _digest(g_o)))
        steps.append((x, dy))
    da.check_status()
    return digests, st, (wq, wk, wv, wo), steps


@pytest.mark.gpu
def test_layer_loop_page3_matches_oracle_and_repeats():
    """Three steps at the page-3 layer shape: the four weight gradients are
    bit-identical at every step across two runs, step 1's gradients match the
    oracle, and the weights after three AdamW steps match oracle.layer's
    train_steps."""
    from oracle import layer
    w = LAYER_PAGE3
    Hq, Hkv, D = w["Hq"], w["Hkv"], w["D"]
    n = 3
    d1, st, w0, steps = _page3_loop(n)
    d2, _, _, _ = _page3_loop(n)
    assert d1 == d2, "weight gradients differ between two runs"
    f = widen
    w_fin, grads = layer.train_steps([f(t) for t in w0], [f(x) for x, _ in steps],
                                     [f(dy) for _, dy in steps], Hq, Hkv, D)
    gqkv_r = np.concatenate(grads[-1][:3], axis=1)
    # The last step's gradients at nearly the same weights.
    assert rel_l2(to_np(st.g_qkv.cpu()), gqkv_r) <= 1e-2
    assert rel_l2(to_np(st.g_o.cpu()), grads[-1][3]) <= 1e-2
    wqkv_r = np.concatenate(w_fin[:3], axis=1)
    wqkv0 = np.concatenate([f(t) for t in w0[:3]], axis=1)
    for got, ref, start in ((st.w_qkv, wqkv_r, wqkv0), (st.w_o, w_fin[3], f(w0[3]))):
        g = to_np(got.cpu())
        # An element can move at most about 2 N lr further one way than the
        # other (opposite AdamW steps); measured: 1.1e-3 on the weights and
        # 2.4 % of the update's norm.  Held to about ten times that.
        assert rel_l2(g, ref) <= 1e-2
        assert rel_l2(g - start, ref - start) <= 0.25


@pytest.mark.gpu
def test_layer_loop_second_process_reproduces_digests():
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); sys.path.insert(0, {os.path.join(ROOT, 'tests')!r});"
            "import test_gpu_layer as t; d, *_ = t._page3_loop(2); print(repr(d))")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d_here, *_ = _page3_loop(2)
    assert r.stdout.strip().splitlines()[-1] == repr(d_here)
