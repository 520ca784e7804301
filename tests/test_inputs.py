"""The seeded input generators (CPU only): the fixed-length recipe and the
packed variable-length one share a draw order, lengths cover their total, and
the varlen oracle runs on what the generator draws."""
import numpy as np
import pytest
import torch

import oracle
from deterministic_attention_gb300.inputs import (VARLEN_PAGE3, WORKLOADS, bf16_bits,
                                                  make_inputs, make_varlen_inputs,
                                                  varlen_lengths, varlen_page3_inputs)


def test_fixed_length_recipe_is_seeded_and_bf16():
    a = make_inputs(2, 33, 4, 2, 8, seed=9, dout_std=0.1, k_peak_frac=0.1)
    b = make_inputs(2, 33, 4, 2, 8, seed=9, dout_std=0.1, k_peak_frac=0.1)
    assert all(x.dtype == torch.bfloat16 and torch.equal(x, y) for x, y in zip(a, b))
    c = make_inputs(2, 33, 4, 2, 8, seed=10, dout_std=0.1, k_peak_frac=0.1)
    assert not torch.equal(a[0], c[0])
    # dO drawn with sigma 0.1: its spread is an order of magnitude below Q's.
    assert 0.05 < float(a[3].float().std()) < 0.2 < 0.5 < float(a[0].float().std())


def test_peaked_keys_are_doubled_exactly():
    base = make_inputs(1, 200, 2, 1, 8, seed=3)
    peak = make_inputs(1, 200, 2, 1, 8, seed=3, k_peak_frac=0.01)
    doubled = [t for t in range(200) if not torch.equal(base[1][0, t], peak[1][0, t])]
    assert len(doubled) == 2  # ceil(0.01 * 200)
    for t in doubled:
        assert torch.equal(peak[1][0, t].float(), 2 * base[1][0, t].float())


@pytest.mark.parametrize("total,lo,hi", [(4096, 64, 1024), (1000, 1, 7), (5, 10, 20), (0, 1, 2)])
def test_varlen_lengths_cover_the_total(total, lo, hi):
    n = varlen_lengths(total, lo, hi, seed=1)
    assert sum(n) == total and all(1 <= x <= hi for x in n)
    assert all(x >= lo for x in n[:-1])
    assert n == varlen_lengths(total, lo, hi, seed=1)


def test_varlen_lengths_validate():
    for lo, hi in ((0, 5), (6, 5)):
        with pytest.raises(ValueError):
            varlen_lengths(10, lo, hi, seed=0)


def test_packed_recipe_matches_the_fixed_length_one():
    """B sequences of length T draw exactly the [B, T] recipe's values."""
    a = make_inputs(3, 11, 4, 2, 8, seed=7, dout_std=0.1)
    q, k, v, do, cu_q, cu_k = make_varlen_inputs([11] * 3, [11] * 3, 4, 2, 8, seed=7, dout_std=0.1)
    for x, y in zip(a, (q, k, v, do)):
        assert torch.equal(x.reshape(y.shape), y)
    assert cu_q.tolist() == [0, 11, 22, 33] and cu_q.dtype == torch.int32


def test_varlen_page3_workload():
    q, k, v, do, cu_q, cu_k = varlen_page3_inputs()
    w = VARLEN_PAGE3
    assert q.shape == (w["total"], w["Hq"], w["D"]) and k.shape == (w["total"], w["Hkv"], w["D"])
    lens = np.diff(cu_q.numpy())
    assert torch.equal(cu_q, cu_k) and lens.sum() == 4096 and lens.max() <= 1024
    assert (lens[:-1] >= 64).all()


def test_varlen_oracle_on_generated_inputs():
    """The generator's bf16 values, widened exactly, feed the varlen oracle;
    each sequence of the pack matches the fixed-length oracle on it alone."""
    tqs = [17, 5, 40]
    q, k, v, do, cu_q, cu_k = make_varlen_inputs(tqs, tqs, 6, 2, 16, seed=12, dout_std=0.1)
    f = lambda t: oracle.bf16_bits_to_f64(bf16_bits(t)).reshape(tuple(t.shape))
    q, k, v, do = (f(t) for t in (q, k, v, do))
    o, lse = oracle.attn_fwd_varlen(q, k, v, cu_q.numpy(), cu_k.numpy(), 0.25, True)
    for s in range(len(tqs)):
        sl = slice(int(cu_q[s]), int(cu_q[s + 1]))
        o1, lse1 = oracle.attn_fwd(q[sl][None], k[sl][None], v[sl][None], 0.25, True)
        assert np.array_equal(o[sl], o1[0]) and np.array_equal(lse[:, sl], lse1[0])


def test_named_workloads_are_the_documented_shapes():
    shapes = {n: w.shape for n, w in WORKLOADS.items()}
    assert shapes == {"tiny": (1, 128, 2, 1, 64), "small": (1, 512, 12, 4, 64),
                      "page3": (4, 1024, 12, 4, 64), "wide": (32, 1024, 24, 24, 64),
                      "long": (1, 8192, 32, 8, 128)}


def test_visible_pairs_count_the_mask():
    """The closed-form pair count equals a count of the bottom-right causal
    mask (and of the full matrix) for every tq, tk < 12."""
    from deterministic_attention_gb300.inputs import varlen_fwd_flops, visible_pairs
    for tq in range(12):
        for tk in range(12):
            i, j = np.arange(tq)[:, None], np.arange(tk)[None, :]
            assert visible_pairs(tq, tk, True) == int((j <= i + (tk - tq)).sum()), (tq, tk)
            assert visible_pairs(tq, tk, False) == tq * tk
    # tq = tk = T, causal: 2 Hq T^2 D plus the diagonal's 2 Hq T D.
    T, Hq, D = 1024, 12, 64
    assert varlen_fwd_flops([T], [T], Hq, D, True) == 2 * Hq * T * T * D + 2 * Hq * T * D


@pytest.mark.parametrize("dist", ["uniform", "zipf"])
def test_embed_grad_inputs(dist):
    from deterministic_attention_gb300.inputs import make_embed_grad_inputs
    ids, dy = make_embed_grad_inputs(5000, 300, 7, seed=3, dist=dist)
    ids2, dy2 = make_embed_grad_inputs(5000, 300, 7, seed=3, dist=dist)
    assert torch.equal(ids, ids2) and torch.equal(dy, dy2)
    assert ids.dtype == torch.int32 and dy.dtype == torch.bfloat16 and dy.shape == (5000, 7)
    assert int(ids.min()) >= 0 and int(ids.max()) < 300
    counts = torch.bincount(ids.long(), minlength=300)
    if dist == "zipf":
        # Id 0 takes the largest share, far above the uniform 1/300.
        assert int(counts.argmax()) == 0 and counts[0] > 5000 / 30
    else:
        assert counts.max() < 5000 / 300 * 3


def test_embed_grad_oracle_on_generated_inputs():
    """The oracle on the generator's ids and exactly widened bf16 rows matches
    the one-hot product."""
    from deterministic_attention_gb300.inputs import make_embed_grad_inputs
    ids, dy = make_embed_grad_inputs(2000, 120, 9, seed=4, dist="zipf")
    dyf = oracle.bf16_bits_to_f64(bf16_bits(dy)).reshape(tuple(dy.shape))
    dw = oracle.embed_grad(ids.numpy(), dyf, 120)
    onehot = np.zeros((2000, 120))
    onehot[np.arange(2000), ids.numpy()] = 1.0
    ref = onehot.T @ dyf
    assert np.max(np.abs(dw - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_layer_inputs_and_the_layer_oracle():
    """The layer recipe's shapes and spreads, and the layer oracle on its
    exactly widened bf16 values (a small copy of the page-3 layer)."""
    from deterministic_attention_gb300.inputs import make_layer_inputs
    from oracle import layer
    B, T, d, Hq, Hkv, D = 2, 40, 48, 6, 2, 8
    t = make_layer_inputs(B, T, d, Hq, Hkv, D, seed=3)
    assert [tuple(a.shape) for a in t] == [(B, T, d), (d, Hq * D), (d, Hkv * D), (d, Hkv * D),
                                           (Hq * D, d), (B, T, d)]
    assert all(a.dtype == torch.bfloat16 for a in t)
    assert 0.01 < float(t[1].float().std()) < 0.03 and 0.05 < float(t[5].float().std()) < 0.2
    f = lambda a: oracle.bf16_bits_to_f64(bf16_bits(a)).reshape(tuple(a.shape))
    x, wq, wk, wv, wo, dy = (f(a) for a in t)
    y, _ = layer.layer_forward(x, wq, wk, wv, wo, Hq, Hkv, D)
    grads = layer.layer_backward(x, wq, wk, wv, wo, dy, Hq, Hkv, D)
    assert y.shape == (B, T, d) and all(np.all(np.isfinite(g)) for g in grads)
    assert [g.shape for g in grads] == [x.shape, wq.shape, wk.shape, wv.shape, wo.shape]
