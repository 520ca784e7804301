"""Pins of the fp64 one-layer oracle (QKV projection, rotary positions,
causal GQA attention, output projection) to facts other than itself: rotary
positions are rotations with known angles whose scores depend only on
relative position, central finite differences of the layer's loss, and
PyTorch fp64 autograd over an independent formulation (rotary positions as
complex multiplication, attention by scaled_dot_product_attention)."""
import math

import numpy as np
import pytest
import torch

from oracle import layer


def _rand(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_rope_is_a_rotation():
    x = _rand(1, 2, 9, 3, 8)
    y = layer.rope(x)
    # Each (i, i + D/2) pair keeps its length; the transpose undoes it; t = 0 is fixed.
    n = lambda a: a[..., :4] ** 2 + a[..., 4:] ** 2
    np.testing.assert_allclose(n(y), n(x), rtol=1e-13)
    np.testing.assert_allclose(layer.rope(y, inverse=True), x, rtol=1e-13, atol=1e-14)
    assert np.array_equal(y[:, 0], x[:, 0])


def test_rope_known_angles():
    """D = 4: pair 0 turns by t radians, pair 1 by t / 100 (base^(-1/2))."""
    T = 6
    x = np.zeros((1, T, 1, 4))
    x[..., 0] = 1.0  # pair 0 = (1, 0)
    x[..., 3] = 1.0  # pair 1 = (0, 1)
    y = layer.rope(x)
    t = np.arange(T)
    np.testing.assert_allclose(y[0, :, 0, 0], np.cos(t), atol=1e-15)
    np.testing.assert_allclose(y[0, :, 0, 2], np.sin(t), atol=1e-15)
    np.testing.assert_allclose(y[0, :, 0, 1], -np.sin(t / 100.0), atol=1e-15)
    np.testing.assert_allclose(y[0, :, 0, 3], np.cos(t / 100.0), atol=1e-15)


def test_rope_scores_depend_on_relative_position():
    """<rope(q) at t1, rope(k) at t2> depends only on t1 - t2."""
    D, T = 16, 12
    q, k = _rand(2, D), _rand(3, D)
    xq = np.broadcast_to(q, (1, T, 1, D)).copy()
    xk = np.broadcast_to(k, (1, T, 1, D)).copy()
    rq, rk = layer.rope(xq)[0, :, 0], layer.rope(xk)[0, :, 0]
    for delta in (0, 1, 5):
        s = [float(rq[t + delta] @ rk[t]) for t in range(T - delta)]
        np.testing.assert_allclose(s, s[0], rtol=1e-12, atol=1e-12)


def _layer_case(seed, B, T, d, Hq, Hkv, D):
    x = _rand(seed, B, T, d)
    wq = _rand(seed + 1, d, Hq * D, scale=0.3)
    wk = _rand(seed + 2, d, Hkv * D, scale=0.3)
    wv = _rand(seed + 3, d, Hkv * D, scale=0.3)
    wo = _rand(seed + 4, Hq * D, d, scale=0.3)
    dy = _rand(seed + 5, B, T, d)
    return x, wq, wk, wv, wo, dy


def test_layer_finite_differences():
    """Central differences of L = sum(dY * Y) in every entry of X and of the
    four weights match the closed-form backward."""
    B, T, d, Hq, Hkv, D = 1, 4, 5, 2, 1, 4
    x, wq, wk, wv, wo, dy = _layer_case(10, B, T, d, Hq, Hkv, D)
    grads = layer.layer_backward(x, wq, wk, wv, wo, dy, Hq, Hkv, D)
    args = [x, wq, wk, wv, wo]

    def loss(a):
        y, _ = layer.layer_forward(*a, Hq, Hkv, D)
        return float(np.sum(dy * y))

    h = 1e-6
    for i, (arg, g) in enumerate(zip(args, grads)):
        fd = np.zeros_like(arg)
        for idx in np.ndindex(arg.shape):
            ap, am = [a.copy() for a in args], [a.copy() for a in args]
            ap[i][idx] += h
            am[i][idx] -= h
            fd[idx] = (loss(ap) - loss(am)) / (2 * h)
        assert np.max(np.abs(fd - g)) <= 1e-6 * max(1.0, np.max(np.abs(g))), i


def _torch_layer(x, wq, wk, wv, wo, dy, Hq, Hkv, D):
    """The layer in torch fp64 with rotary positions as complex rotations."""
    tt = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    X, Wq, Wk, Wv, Wo = (tt(a) for a in (x, wq, wk, wv, wo))
    B, T, d = x.shape
    G = Hq // Hkv

    def rot(m, H):
        m = m.reshape(B, T, H, D)
        z = torch.complex(m[..., : D // 2], m[..., D // 2:])
        i = torch.arange(D // 2, dtype=torch.float64)
        theta = torch.arange(T, dtype=torch.float64)[:, None] * 10000.0 ** (-2.0 * i / D)
        z = z * torch.polar(torch.ones_like(theta), theta)[None, :, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    q = rot(X @ Wq, Hq).permute(0, 2, 1, 3)
    k = rot(X @ Wk, Hkv).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    v = (X @ Wv).reshape(B, T, Hkv, D).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                         scale=1.0 / math.sqrt(D))
    y = o.permute(0, 2, 1, 3).reshape(B, T, Hq * D) @ Wo
    y.backward(torch.tensor(dy, dtype=torch.float64))
    return y.detach().numpy(), [a.grad.numpy() for a in (X, Wq, Wk, Wv, Wo)]


@pytest.mark.parametrize("shape", [(2, 9, 12, 4, 2, 8), (1, 17, 10, 3, 3, 4)])
def test_layer_matches_torch_autograd(shape):
    B, T, d, Hq, Hkv, D = shape
    x, wq, wk, wv, wo, dy = _layer_case(20, B, T, d, Hq, Hkv, D)
    y_t, grads_t = _torch_layer(x, wq, wk, wv, wo, dy, Hq, Hkv, D)
    y, _ = layer.layer_forward(x, wq, wk, wv, wo, Hq, Hkv, D)
    grads = layer.layer_backward(x, wq, wk, wv, wo, dy, Hq, Hkv, D)
    rel = lambda a, b: float(np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b))))
    assert rel(y, y_t) <= 1e-12
    for name, g, g_t in zip(("dX", "dWq", "dWk", "dWv", "dWo"), grads, grads_t):
        assert rel(g, g_t) <= 1e-12, name


def test_adamw_matches_torch():
    """Five AdamW steps on random gradients equal torch.optim.AdamW in fp64
    (same defaults: betas 0.9, 0.999, eps 1e-8; lr 3e-4, weight decay 0.1)."""
    w0, gs = _rand(40, 6, 5), [_rand(41 + i, 6, 5) for i in range(5)]
    p = torch.tensor(w0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([p], lr=3e-4, weight_decay=0.1)
    w, m, v = w0, np.zeros_like(w0), np.zeros_like(w0)
    for t, g in enumerate(gs, start=1):
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        w, m, v = layer.adamw_step(w, g, m, v, t)
        np.testing.assert_allclose(w, p.detach().numpy(), rtol=1e-15, atol=1e-15)


def test_adamw_first_step_closed_form():
    """At t = 1 the corrected moments are g and g^2, so each weight moves by
    lr * g / (|g| + eps) after its decay."""
    w0, g = _rand(50, 4, 3), _rand(51, 4, 3)
    w, _, _ = layer.adamw_step(w0, g, np.zeros_like(g), np.zeros_like(g), 1)
    np.testing.assert_allclose(w, w0 * (1 - 3e-4 * 0.1) - 3e-4 * g / (np.abs(g) + 1e-8),
                               rtol=1e-14)


def test_train_steps_is_the_composition():
    """Two micro-loop steps equal gradient, update, gradient, update done by
    hand; with lr = 0 the weights stay and both steps' gradients are equal."""
    B, T, d, Hq, Hkv, D = 1, 6, 8, 4, 2, 4
    x, wq, wk, wv, wo, dy = _layer_case(60, B, T, d, Hq, Hkv, D)
    x2, dy2 = _rand(70, B, T, d), _rand(71, B, T, d)
    w, grads = layer.train_steps([wq, wk, wv, wo], [x, x2], [dy, dy2], Hq, Hkv, D)
    ws = [wq, wk, wv, wo]
    ms = [np.zeros_like(a) for a in ws]
    vs = [np.zeros_like(a) for a in ws]
    for t, (xx, dd) in enumerate(((x, dy), (x2, dy2)), start=1):
        g = layer.layer_backward(xx, *ws, dd, Hq, Hkv, D)[1:]
        for a, b in zip(g, grads[t - 1]):
            assert np.array_equal(a, b)
        for i in range(4):
            ws[i], ms[i], vs[i] = layer.adamw_step(ws[i], g[i], ms[i], vs[i], t)
    for a, b in zip(w, ws):
        assert np.array_equal(a, b)
    w0, g0 = layer.train_steps([wq, wk, wv, wo], [x, x], [dy, dy], Hq, Hkv, D, lr=0.0)
    assert all(np.array_equal(a, b) for a, b in zip(w0, [wq, wk, wv, wo]))
    assert all(np.array_equal(a, b) for a, b in zip(g0[0], g0[1]))


# Planted mistakes in a copy of oracle/layer.py: (name, text, replacement,
# occurrences).  Each must make at least one pin above fail.
_LAYER_MUTANTS = [
    ("rope_inverse_not_inverted", "    if inverse:\n        s = -s\n", "", 1),
    ("rope_base_1000", "ROPE_BASE = 10000.0", "ROPE_BASE = 1000.0", 1),
    ("rope_second_half_sign", "x2 * c + x1 * s", "x2 * c - x1 * s", 1),
    ("rope_positions_from_1", "np.arange(T, dtype=np.float64)[:, None] * inv",
     "(np.arange(T, dtype=np.float64)[:, None] + 1) * inv", 1),
    ("fwd_scale_1_over_D", "o, lse = attn_fwd(q, k, v, 1.0 / np.sqrt(D), causal)",
     "o, lse = attn_fwd(q, k, v, 1.0 / D, causal)", 1),
    ("dwv_from_dk", "xf.T @ dvf", "xf.T @ dk", 1),
    ("dx_without_v_term", " + dvf @ wv.T", "", 1),
    ("dk_rotated_forward", "dk = rope(dkr, inverse=True)", "dk = rope(dkr, inverse=False)", 1),
    ("adamw_no_bias_correction", "mhat = m / (1.0 - b1 ** t)", "mhat = m", 1),
    ("adamw_no_weight_decay", "    w = w * (1.0 - lr * wd)\n", "", 1),
]

_LAYER_PINS = [
    ("rotation", test_rope_is_a_rotation, ()),
    ("angles", test_rope_known_angles, ()),
    ("relative", test_rope_scores_depend_on_relative_position, ()),
    ("fd", test_layer_finite_differences, ()),
    ("torch_a", test_layer_matches_torch_autograd, ((2, 9, 12, 4, 2, 8),)),
    ("torch_b", test_layer_matches_torch_autograd, ((1, 17, 10, 3, 3, 4),)),
    ("adamw_torch", test_adamw_matches_torch, ()),
    ("adamw_first", test_adamw_first_step_closed_form, ()),
    ("loop", test_train_steps_is_the_composition, ()),
]


@pytest.mark.parametrize("name,old,new,count",
                         [pytest.param(*m, id=m[0])
                          for m in [("unchanged", None, None, 0)] + _LAYER_MUTANTS])
def test_layer_pins_catch_planted_mistakes(name, old, new, count, tmp_path, monkeypatch):
    import importlib.util
    import sys
    src = open(layer.__file__).read()
    if old is not None:
        assert src.count(old) == count, name
        src = src.replace(old, new)
    src = src.replace("from . import attn_bwd, attn_fwd", "from oracle import attn_bwd, attn_fwd")
    path = tmp_path / f"layer_{name}.py"
    path.write_text(src)
    spec = importlib.util.spec_from_file_location(f"layer_{name}", path)
    mutant = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mutant)
    monkeypatch.setattr(sys.modules[__name__], "layer", mutant)
    caught = []
    for pin, fn, args in _LAYER_PINS:
        try:
            fn(*args)
        except AssertionError:
            caught.append(pin)
    if old is None:
        assert caught == [], f"the unchanged source fails {caught}"
    else:
        assert caught, f"no pin catches the planted mistake {name}"
