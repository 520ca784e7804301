"""fp64 oracle of one attention layer of a training step: QKV projection,
rotary positions, causal grouped-query attention, output projection, and
their closed-form backward.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only the test suite
and the benchmark's CPU legs may use it.

What it computes (RustingBrain vs PyTorch/TensorFlow page, "The setup": a
decoder-only model of d_model 768 with 12 query heads sharing 4 KV heads of
head_dim 64 and rotary positions).  For X [B, T, d]:

    Q = rope(X Wq),  K = rope(X Wk),  V = X Wv      (heads split from the last axis)
    O = attention(Q, K, V)                           (the attention oracle, causal)
    Y = O Wo                                         (heads joined on the last axis)

with Wq [d, Hq*D], Wk, Wv [d, Hkv*D], Wo [Hq*D, d].  Given dY, the backward
is

    dWo = O^T dY,   dO = dY Wo^T
    dQr, dKr, dV = attention backward at (Q, K, V, dO)
    dQ = rope^T(dQr),  dK = rope^T(dKr)             (rope is a rotation: its transpose inverts it)
    dWq = X^T dQ,  dWk = X^T dK,  dWv = X^T dV,  dX = dQ Wq^T + dK Wk^T + dV Wv^T

with every product over the flattened (b, t) rows.  The pages do not say
which components rope pairs; this takes the rotate-half form: component i of
a head's first half and component i of its second half turn together by
angle t * base^(-2i/D), base 10000.

Matrix products use numpy (a library step); the attention is the C oracle.

The training micro-loop around the layer updates its four weights with AdamW
(oxide-train README: the trainer's step ends in AdamW, run with LR 3e-4 and
weight decay 0.1).  The pages give neither betas nor epsilon; the reading
takes 0.9, 0.999 and 1e-8, with decoupled weight decay:

    m = b1 m + (1 - b1) g,   v = b2 v + (1 - b2) g^2
    w = w - lr (m / (1 - b1^t) / (sqrt(v / (1 - b2^t)) + eps) + wd w)
"""
from __future__ import annotations

import numpy as np

from . import attn_bwd, attn_fwd

ROPE_BASE = 10000.0


def rope_angles(T: int, D: int, base: float = ROPE_BASE) -> np.ndarray:
    """[T, D/2] angles t * base^(-2i/D)."""
    inv = base ** (-np.arange(0, D // 2, dtype=np.float64) * 2.0 / D)
    return np.arange(T, dtype=np.float64)[:, None] * inv[None, :]


def rope(x: np.ndarray, base: float = ROPE_BASE, inverse: bool = False) -> np.ndarray:
    """Rotate-half rotary positions on x [B, T, H, D]; inverse=True applies
    the transpose (the rotation by minus the angle)."""
    B, T, H, D = x.shape
    ang = rope_angles(T, D, base)
    c, s = np.cos(ang)[None, :, None, :], np.sin(ang)[None, :, None, :]
    if inverse:
        s = -s
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def _heads(m: np.ndarray, B: int, T: int, D: int) -> np.ndarray:
    return m.reshape(B, T, -1, D)


def layer_forward(x, wq, wk, wv, wo, Hq: int, Hkv: int, D: int, causal: bool = True):
    """Y [B, T, d] and the intermediates the backward needs."""
    x, wq, wk, wv, wo = (np.asarray(a, dtype=np.float64) for a in (x, wq, wk, wv, wo))
    B, T, d = x.shape
    xf = x.reshape(B * T, d)
    q = rope(_heads(xf @ wq, B, T, D))
    k = rope(_heads(xf @ wk, B, T, D))
    v = _heads(xf @ wv, B, T, D)
    o, lse = attn_fwd(q, k, v, 1.0 / np.sqrt(D), causal)
    y = (o.reshape(B * T, Hq * D) @ wo).reshape(B, T, -1)
    return y, {"q": q, "k": k, "v": v, "o": o, "lse": lse}


def layer_backward(x, wq, wk, wv, wo, dy, Hq: int, Hkv: int, D: int, causal: bool = True):
    """(dX, dWq, dWk, dWv, dWo) for the upstream gradient dy [B, T, d]."""
    x, wq, wk, wv, wo, dy = (np.asarray(a, dtype=np.float64) for a in (x, wq, wk, wv, wo, dy))
    B, T, d = x.shape
    _, c = layer_forward(x, wq, wk, wv, wo, Hq, Hkv, D, causal)
    xf, dyf = x.reshape(B * T, d), dy.reshape(B * T, d)
    of = c["o"].reshape(B * T, Hq * D)
    dwo = of.T @ dyf
    do = _heads(dyf @ wo.T, B, T, D)
    dqr, dkr, dv, _, _ = attn_bwd(c["q"], c["k"], c["v"], do, 1.0 / np.sqrt(D), causal)
    dq = rope(dqr, inverse=True).reshape(B * T, Hq * D)
    dk = rope(dkr, inverse=True).reshape(B * T, Hkv * D)
    dvf = dv.reshape(B * T, Hkv * D)
    dwq, dwk, dwv = xf.T @ dq, xf.T @ dk, xf.T @ dvf
    dx = (dq @ wq.T + dk @ wk.T + dvf @ wv.T).reshape(B, T, d)
    return dx, dwq, dwk, dwv, dwo


def adamw_step(w, g, m, v, t: int, lr: float = 3e-4, wd: float = 0.1, b1: float = 0.9,
               b2: float = 0.999, eps: float = 1e-8):
    """One AdamW update of step t (1-based): returns (w, m, v), new arrays."""
    w, g, m, v = (np.asarray(a, dtype=np.float64) for a in (w, g, m, v))
    w = w * (1.0 - lr * wd)
    m = b1 * m + (1.0 - b1) * g
    v = b2 * v + (1.0 - b2) * g * g
    mhat = m / (1.0 - b1 ** t)
    vhat = v / (1.0 - b2 ** t)
    return w - lr * mhat / (np.sqrt(vhat) + eps), m, v


def train_steps(weights, xs, dys, Hq: int, Hkv: int, D: int, causal: bool = True,
                lr: float = 3e-4, wd: float = 0.1):
    """The micro-loop: for each (x, dy) in turn, the layer's weight gradients
    at the current weights, then one AdamW update of (Wq, Wk, Wv, Wo).
    Returns the final weights and every step's gradients."""
    w = [np.asarray(a, dtype=np.float64) for a in weights]
    m = [np.zeros_like(a) for a in w]
    v = [np.zeros_like(a) for a in w]
    grads = []
    for t, (x, dy) in enumerate(zip(xs, dys), start=1):
        g = layer_backward(x, *w, dy, Hq, Hkv, D, causal)[1:]
        grads.append(g)
        for i in range(4):
            w[i], m[i], v[i] = adamw_step(w[i], g[i], m[i], v[i], t, lr, wd)
    return w, grads
