"""Pins of the fp64 oracle to facts other than itself.

The pages print no worked attention example (no inputs with outputs), so the
oracle is pinned by: central finite differences of its own loss, closed forms
(a hand-derived two-token case, uniform attention, T = 1, constant V),
invariants (softmax rows sum to one, causality, GQA as repeated-KV MHA) and a
library special case (PyTorch's fp64 CPU scaled_dot_product_attention with
autograd).  Each test names the kind of mistake it is there to catch.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _case(seed, B, T, Hq, Hkv, D):
    rng = np.random.default_rng(seed)
    return (_rand(rng, B, T, Hq, D), _rand(rng, B, T, Hkv, D), _rand(rng, B, T, Hkv, D),
            _rand(rng, B, T, Hq, D))


def _rel(a, b, floor=1e-300):
    """max |a - b| relative to max |b| (or to `floor` when b is all ~0)."""
    return float(np.max(np.abs(a - b)) / max(floor, np.max(np.abs(b))))


# ------------------------------------------------------------ closed forms
def test_hand_derived_two_tokens():
    """T=2, D=1, scale=1, q=(1,2), k=(1,-1), v=(3,5), dO=(0.5,-1.5).

    Row 0 sees only key 0: LSE_0 = 1, O_0 = 3.  Row 1 has scores (2, -2):
    with p = 1/(1+e^4) = P_11, LSE_1 = ln(e^2 + e^-2), O_1 = 3 + 2p.
    Backward: dS_00 = 0, dS_10 = P_10 P_11 dO_1 (v_0 - v_1) = 3p(1-p) = -dS_11,
    so dQ = (0, 6p(1-p)), dK = (6p(1-p), -6p(1-p)),
    dV = (0.5 - 1.5(1-p), -1.5p).  Catches sign, transposition and masking
    mistakes in every formula of the backward.
    """
    q = np.array([1.0, 2.0]).reshape(1, 2, 1, 1)
    k = np.array([1.0, -1.0]).reshape(1, 2, 1, 1)
    v = np.array([3.0, 5.0]).reshape(1, 2, 1, 1)
    do = np.array([0.5, -1.5]).reshape(1, 2, 1, 1)
    p = 1.0 / (1.0 + math.exp(4.0))
    o, lse = oracle.attn_fwd(q, k, v, 1.0, True)
    np.testing.assert_allclose(o.reshape(-1), [3.0, 3.0 + 2.0 * p], rtol=1e-15, atol=0)
    np.testing.assert_allclose(lse.reshape(-1), [1.0, math.log(math.exp(2) + math.exp(-2))],
                               rtol=1e-15)
    dq, dk, dv, delta, worst = oracle.attn_bwd(q, k, v, do, 1.0, True)
    s = 6.0 * p * (1.0 - p)
    np.testing.assert_allclose(dq.reshape(-1), [0.0, s], rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(dk.reshape(-1), [s, -s], rtol=1e-13)
    np.testing.assert_allclose(dv.reshape(-1), [0.5 - 1.5 * (1.0 - p), -1.5 * p], rtol=1e-14)
    np.testing.assert_allclose(delta.reshape(-1), [0.5 * 3.0, -1.5 * (3.0 + 2.0 * p)], rtol=1e-15)
    assert worst < 1e-14


def test_uniform_attention_when_q_is_zero():
    """Q = 0 makes every visible score 0: P_ij = 1/(i+1), LSE_i = ln(i+1),
    O_i = mean(V_0..V_i).  Catches an off-by-one in the causal range."""
    B, T, Hq, Hkv, D = 2, 9, 4, 2, 5
    _, k, v, _ = _case(1, B, T, Hq, Hkv, D)
    q = np.zeros((B, T, Hq, D))
    o, lse = oracle.attn_fwd(q, k, v, 0.3, True)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            for i in range(T):
                assert abs(lse[b, h, i] - math.log(i + 1)) < 1e-14
                ref = v[b, : i + 1, g, :].mean(axis=0)
                np.testing.assert_allclose(o[b, i, h], ref, rtol=1e-13, atol=1e-14)
    p = oracle.attn_probs(q, k, 1, 3, 0.3, True)
    for i in range(T):
        np.testing.assert_allclose(p[i, : i + 1], 1.0 / (i + 1), rtol=1e-14)


def test_single_token():
    """T = 1: O = V_0 and LSE = scale * q.k_0 (a one-term softmax)."""
    q, k, v, _ = _case(2, 3, 1, 6, 3, 7)
    o, lse = oracle.attn_fwd(q, k, v, 0.4, True)
    for b in range(3):
        for h in range(6):
            g = h // 2
            np.testing.assert_allclose(o[b, 0, h], v[b, 0, g], rtol=1e-15)
            assert abs(lse[b, h, 0] - 0.4 * float(q[b, 0, h] @ k[b, 0, g])) < 1e-14


def test_constant_v_rows():
    """Every V row equal to v: O_i = v; then D_i = dO_i.v = dP_ij for every j,
    so dS = 0 and dQ = dK = 0.  Catches a wrong D_i or a missing P factor."""
    B, T, Hq, Hkv, D = 1, 11, 3, 1, 6
    q, k, _, do = _case(3, B, T, Hq, Hkv, D)
    vrow = np.linspace(-1.0, 2.0, D)
    v = np.broadcast_to(vrow, (B, T, Hkv, D)).copy()
    o, _ = oracle.attn_fwd(q, k, v, 0.5, True)
    np.testing.assert_allclose(o, np.broadcast_to(vrow, o.shape), rtol=1e-15, atol=1e-15)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, 0.5, True)
    assert np.max(np.abs(dq)) < 1e-14
    assert np.max(np.abs(dk)) < 1e-14
    assert np.max(np.abs(dv)) > 0.1


# ------------------------------------------------------------ invariants
@pytest.mark.parametrize("causal", [True, False])
def test_softmax_rows_sum_to_one_and_mask(causal):
    q, k, _, _ = _case(4, 2, 13, 4, 2, 8)
    for b in range(2):
        for h in range(4):
            p = oracle.attn_probs(q, k, b, h, 0.35, causal)
            assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-12
            assert np.all(p >= 0)
            if causal:
                assert np.all(p[np.triu_indices(13, 1)] == 0.0)
            else:
                assert np.all(p > 0)


def test_causality_is_exact():
    """Perturbing keys/values after position i leaves O_i and LSE_i
    bit-identical.  Catches a mask that lets a later key leak in."""
    B, T, Hq, Hkv, D = 2, 17, 4, 2, 8
    q, k, v, _ = _case(5, B, T, Hq, Hkv, D)
    o, lse = oracle.attn_fwd(q, k, v, 0.25, True)
    for i0 in (0, 5, 16):
        k2, v2 = k.copy(), v.copy()
        rng = np.random.default_rng(i0)
        k2[:, i0 + 1:] += rng.standard_normal(k2[:, i0 + 1:].shape) * 3
        v2[:, i0 + 1:] -= rng.standard_normal(v2[:, i0 + 1:].shape) * 3
        o2, lse2 = oracle.attn_fwd(q, k2, v2, 0.25, True)
        assert np.array_equal(o2[:, : i0 + 1], o[:, : i0 + 1])
        assert np.array_equal(lse2[:, :, : i0 + 1], lse[:, :, : i0 + 1])
        if i0 < T - 1:
            assert not np.array_equal(o2[:, i0 + 1:], o[:, i0 + 1:])


@pytest.mark.parametrize("G", [2, 3])
def test_gqa_is_repeated_kv_mha(G):
    """GQA with group size G equals MHA with each KV head repeated G times
    (query head h reads KV head h // G); dK/dV are the sums of the MHA
    gradients over the group.  Catches a wrong head mapping (e.g. h % Hkv)."""
    B, T, Hkv, D = 2, 10, 2, 4
    Hq = Hkv * G
    q, k, v, do = _case(6 + G, B, T, Hq, Hkv, D)
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    o, lse = oracle.attn_fwd(q, k, v, 0.6, True)
    o_m, lse_m = oracle.attn_fwd(q, kr, vr, 0.6, True)
    assert np.array_equal(o, o_m) and np.array_equal(lse, lse_m)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, 0.6, True)
    dq_m, dk_m, dv_m, _, _ = oracle.attn_bwd(q, kr, vr, do, 0.6, True)
    np.testing.assert_allclose(dq, dq_m, rtol=1e-13, atol=1e-15)
    dk_sum = dk_m.reshape(B, T, Hkv, G, D).sum(axis=3)
    dv_sum = dv_m.reshape(B, T, Hkv, G, D).sum(axis=3)
    assert _rel(dk, dk_sum) <= 1e-13
    assert _rel(dv, dv_sum) <= 1e-13


def test_rowdot_is_the_backward_delta():
    """The standalone rowsum of dO * O equals the D_i the backward forms."""
    q, k, v, do = _case(14, 2, 21, 4, 2, 8)
    o, _ = oracle.attn_fwd(q, k, v, 0.3, True)
    *_, delta, _ = oracle.attn_bwd(q, k, v, do, 0.3, True)
    np.testing.assert_allclose(oracle.rowdot(o, do), delta, rtol=1e-13, atol=1e-15)


def test_delta_forms_agree():
    """D_i = dO_i.O_i equals sum_j P_ij dP_ij (softmax Jacobian identity)."""
    q, k, v, do = _case(9, 2, 33, 6, 2, 16)
    *_, worst = oracle.attn_bwd(q, k, v, do, 0.25, True)
    assert worst <= 1e-12


# ------------------------------------------------------------ finite differences
@pytest.mark.parametrize("causal", [True, False])
def test_finite_differences(causal):
    """Central differences of L = sum(dO * O) with h = 1e-6 in every entry of
    Q, K and V match the closed-form dQ, dK, dV.  Catches any dropped term,
    wrong sign or missing scale in the backward."""
    B, T, Hq, Hkv, D = 1, 5, 2, 1, 3
    q, k, v, do = _case(10, B, T, Hq, Hkv, D)
    scale = 0.7
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, scale, causal)

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd(q_, k_, v_, scale, causal)
        return float(np.sum(do * o))

    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (loss(**{kk + "_": vv for kk, vv in args_p.items()}) -
                       loss(**{kk + "_": vv for kk, vv in args_m.items()})) / (2 * h)
        assert np.max(np.abs(fd - grad)) <= 1e-6 * max(1.0, np.max(np.abs(grad))), name


# ------------------------------------------------------------ library special case
def _torch_ref(q, k, v, do, scale, causal):
    G = q.shape[2] // k.shape[2]
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64).permute(0, 2, 1, 3).contiguous()
                  .requires_grad_(True) for x in (q, k, v))
    kr = tk.repeat_interleave(G, dim=1)
    vr = tv.repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(tq, kr, vr, is_causal=causal,
                                                         scale=scale)
    tdo = torch.tensor(do, dtype=torch.float64).permute(0, 2, 1, 3)
    o.backward(tdo)
    s = (tq @ kr.transpose(-1, -2)) * scale
    if causal:
        T = q.shape[1]
        s = s.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    f = lambda t: t.detach().permute(0, 2, 1, 3).numpy()
    return f(o), lse.detach().numpy(), f(tq.grad), f(tk.grad), f(tv.grad)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(2, 37, 6, 2, 16), (1, 64, 4, 4, 32), (1, 1, 2, 1, 8)])
def test_matches_torch_sdpa_fp64(shape, causal):
    B, T, Hq, Hkv, D = shape
    q, k, v, do = _case(11, *shape)
    scale = 1.0 / math.sqrt(D)
    o_r, lse_r, dq_r, dk_r, dv_r = _torch_ref(q, k, v, do, scale, causal)
    o, lse = oracle.attn_fwd(q, k, v, scale, causal)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, scale, causal)
    # With T = 1 the exact dQ and dK are 0 (one-term softmax); torch leaves
    # ~1e-17 of rounding there, so the relative measure gets a floor of 1.
    assert _rel(o, o_r) <= 1e-12
    assert _rel(lse, lse_r) <= 1e-12
    assert _rel(dq, dq_r, floor=1.0) <= 1e-12
    assert _rel(dk, dk_r, floor=1.0) <= 1e-12
    assert _rel(dv, dv_r) <= 1e-12


# ------------------------------------------------------------ sampled rows, determinism
def test_sampled_rows_match_full_oracle():
    B, T, Hq, Hkv, D = 2, 40, 6, 2, 8
    q, k, v, do = _case(12, B, T, Hq, Hkv, D)
    for causal in (True, False):
        o, lse = oracle.attn_fwd(q, k, v, 0.3, causal)
        dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, 0.3, causal)
        # Heads 1 and 4 are where the group mapping h // G differs from h % Hkv.
        rows = [(0, 0, 0), (1, 5, 39), (0, 3, 17), (1, 2, 1), (0, 1, 22), (1, 4, 30)]
        o_r, lse_r, dq_r = oracle.attn_rows(q, k, v, do, rows, 0.3, causal)
        for s, (b, h, i) in enumerate(rows):
            assert np.array_equal(o_r[s], o[b, i, h])
            assert lse_r[s] == lse[b, h, i]
            np.testing.assert_allclose(dq_r[s], dq[b, i, h], rtol=1e-12, atol=1e-15)
        js = [0, 7, 39]
        for b, g in ((1, 1), (0, 0)):
            dk_r, dv_r = oracle.kv_rows(q, k, v, do, b, g, js, 0.3, causal)
            for s, j in enumerate(js):
                np.testing.assert_allclose(dk_r[s], dk[b, j, g], rtol=1e-12, atol=1e-15)
                np.testing.assert_allclose(dv_r[s], dv[b, j, g], rtol=1e-12, atol=1e-15)


def test_oracle_is_deterministic():
    q, k, v, do = _case(13, 2, 50, 4, 2, 8)
    a = oracle.attn_bwd(q, k, v, do, 0.3, True)
    b = oracle.attn_bwd(q, k, v, do, 0.3, True)
    for x, y in zip(a[:4], b[:4]):
        assert x.tobytes() == y.tobytes()


def _fixture_module():
    import importlib.util
    import os
    golden = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location(
        "make_oracle_fixture", os.path.join(golden, "make_oracle_fixture.py"))
    fx = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(fx)
    return fx, golden


@pytest.mark.parametrize("which", ["fixed", "varlen"])
def test_oracle_reproduces_its_fixture(which):
    """The stored outputs of tests/golden/make_oracle_fixture.py (written by
    the oracle alone) are reproduced; tolerance for libm differences between
    hosts only (-inf entries must match exactly)."""
    import os
    fx, golden = _fixture_module()
    name, outputs = ((fx.NAME, fx.outputs) if which == "fixed"
                     else (fx.VARLEN_NAME, fx.varlen_outputs))
    stored = {}
    with open(os.path.join(golden, name)) as f:
        for line in f:
            if line.startswith("#"):
                continue
            causal, tensor, *vals = line.split()
            stored[(int(causal.split("=")[1]), tensor)] = np.array([float(x) for x in vals])
    assert len(stored) == 10
    for causal in (1, 0):
        for tensor, x in outputs(bool(causal)).items():
            ref = stored[(causal, tensor)]
            assert ref.size == x.size, (causal, tensor)
            np.testing.assert_allclose(x.reshape(-1), ref, rtol=1e-13, atol=1e-15,
                                       err_msg=f"causal={causal} {tensor}")


def test_bf16_widening_is_exact():
    vals = torch.tensor([0.0, -0.0, 1.0, -2.5, 3.140625, 1e-30, 65280.0, float("inf")],
                        dtype=torch.bfloat16)
    bits = vals.view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_bits_to_f64(bits)
    np.testing.assert_array_equal(got, vals.to(torch.float64).numpy())


# ------------------------------------------------------------ packed variable-length batches
def _packed(seed, tqs, tks, Hq, Hkv, D):
    rng = np.random.default_rng(seed)
    cu_q, cu_k = np.concatenate([[0], np.cumsum(tqs)]), np.concatenate([[0], np.cumsum(tks)])
    return (_rand(rng, cu_q[-1], Hq, D), _rand(rng, cu_k[-1], Hkv, D), _rand(rng, cu_k[-1], Hkv, D),
            _rand(rng, cu_q[-1], Hq, D), cu_q, cu_k)


def test_varlen_equal_lengths_is_the_batched_oracle():
    """B sequences of one length T, packed, give the fixed-length oracle's
    bytes (same operations in the same order).  Catches a wrong packed offset
    or LSE layout."""
    B, T, Hq, Hkv, D = 3, 11, 6, 2, 5
    q, k, v, do = _case(20, B, T, Hq, Hkv, D)
    cu = np.arange(B + 1) * T
    pk = lambda x: x.reshape(B * T, x.shape[2], D)
    lse_layout = lambda x: x.transpose(1, 0, 2).reshape(x.shape[1], B * T)
    for causal in (True, False):
        o, lse = oracle.attn_fwd(q, k, v, 0.4, causal)
        ov, lsev = oracle.attn_fwd_varlen(pk(q), pk(k), pk(v), cu, cu, 0.4, causal)
        assert np.array_equal(pk(o), ov) and np.array_equal(lse_layout(lse), lsev)
        dq, dk, dv, delta, _ = oracle.attn_bwd(q, k, v, do, 0.4, causal)
        dqv, dkv, dvv, deltav, _ = oracle.attn_bwd_varlen(pk(q), pk(k), pk(v), pk(do), cu, cu, 0.4,
                                                          causal)
        assert np.array_equal(pk(dq), dqv) and np.array_equal(pk(dk), dkv)
        assert np.array_equal(pk(dv), dvv) and np.array_equal(lse_layout(delta), deltav)


def test_varlen_sequences_are_independent():
    """Sequences of different lengths (one empty) each give exactly what the
    fixed-length oracle gives for that sequence alone.  Catches attention
    across a sequence boundary."""
    tqs = [5, 0, 13, 1, 8]
    Hq, Hkv, D = 4, 2, 6
    q, k, v, do, cu, _ = _packed(21, tqs, tqs, Hq, Hkv, D)
    for causal in (True, False):
        o, lse = oracle.attn_fwd_varlen(q, k, v, cu, cu, 0.3, causal)
        dq, dk, dv, _, _ = oracle.attn_bwd_varlen(q, k, v, do, cu, cu, 0.3, causal)
        for s, T in enumerate(tqs):
            if T == 0:
                continue
            sl = slice(cu[s], cu[s + 1])
            one = lambda x: x[sl][None]
            o1, lse1 = oracle.attn_fwd(one(q), one(k), one(v), 0.3, causal)
            dq1, dk1, dv1, _, _ = oracle.attn_bwd(one(q), one(k), one(v), one(do), 0.3, causal)
            assert np.array_equal(o[sl], o1[0]) and np.array_equal(lse[:, sl], lse1[0])
            assert np.array_equal(dq[sl], dq1[0]) and np.array_equal(dk[sl], dk1[0])
            assert np.array_equal(dv[sl], dv1[0])


def _torch_seq(q, k, v, do, scale, causal):
    """PyTorch fp64 SDPA with autograd for one sequence (q [tq, Hq, D],
    k [tk, Hkv, D]) under the bottom-right causal mask.  Rows that see no key
    are left out of the call (SDPA returns NaN for them) and returned as
    O = 0, LSE = -inf, dQ = 0: they add nothing to dK, dV."""
    tq, tk, Hq, Hkv = q.shape[0], k.shape[0], q.shape[1], k.shape[1]
    G = Hq // Hkv
    r0 = min(tq, max(0, tq - tk)) if causal else (tq if tk == 0 else 0)
    o, lse = np.zeros_like(q), np.full((Hq, tq), -np.inf)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    if r0 == tq:
        return o, lse, dq, dk, dv
    tt = lambda x: torch.tensor(x, dtype=torch.float64).permute(1, 0, 2)[None].contiguous()
    tq_, tk_, tv_ = (tt(x).requires_grad_(True) for x in (q[r0:], k, v))
    kr, vr = tk_.repeat_interleave(G, dim=1), tv_.repeat_interleave(G, dim=1)
    mask = None
    if causal:
        i = np.arange(r0, tq)[:, None]
        mask = torch.tensor(np.arange(tk)[None, :] <= i + (tk - tq))
    out = torch.nn.functional.scaled_dot_product_attention(tq_, kr, vr, attn_mask=mask,
                                                           scale=scale)
    out.backward(tt(do[r0:]))
    sc = (tq_ @ kr.transpose(-1, -2)) * scale
    if mask is not None:
        sc = sc.masked_fill(~mask, float("-inf"))
    back = lambda t: t.detach()[0].permute(1, 0, 2).numpy()
    o[r0:], dq[r0:] = back(out), back(tq_.grad)
    lse[:, r0:] = torch.logsumexp(sc, dim=-1).detach()[0].numpy()
    return o, lse, dq, back(tk_.grad), back(tv_.grad)


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_cross_attention_matches_torch(causal):
    """Tq != Tk per sequence (more queries than keys, fewer, equal, no keys,
    no queries) against PyTorch's fp64 scaled_dot_product_attention with the
    bottom-right causal mask given explicitly.  Catches a wrong mask offset,
    a wrong key offset or a wrong head mapping in the packed functions."""
    tqs, tks = [7, 3, 12, 1, 5, 0], [4, 9, 12, 6, 0, 5]
    Hq, Hkv, D = 4, 2, 8
    q, k, v, do, cu_q, cu_k = _packed(22, tqs, tks, Hq, Hkv, D)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.attn_fwd_varlen(q, k, v, cu_q, cu_k, scale, causal)
    dq, dk, dv, _, worst = oracle.attn_bwd_varlen(q, k, v, do, cu_q, cu_k, scale, causal)
    assert worst <= 1e-12
    for s in range(len(tqs)):
        sq, sk = slice(cu_q[s], cu_q[s + 1]), slice(cu_k[s], cu_k[s + 1])
        o_r, lse_r, dq_r, dk_r, dv_r = _torch_seq(q[sq], k[sk], v[sk], do[sq], scale, causal)
        if tqs[s]:
            assert _rel(o[sq], o_r, floor=1.0) <= 1e-12
            fin = np.isfinite(lse_r)
            assert np.array_equal(fin, np.isfinite(lse[:, sq]))
            if fin.any():
                assert _rel(lse[:, sq][fin], lse_r[fin], floor=1.0) <= 1e-12
            assert _rel(dq[sq], dq_r, floor=1.0) <= 1e-12
        if tks[s]:
            assert _rel(dk[sk], dk_r, floor=1.0) <= 1e-12
            assert _rel(dv[sk], dv_r, floor=1.0) <= 1e-12


def test_varlen_rows_that_see_no_key():
    """More queries than keys under the causal mask: the first tq - tk rows
    see nothing, so O = 0, LSE = -inf, dQ = 0, Delta = 0; keys that no query
    sees get dK = dV = 0."""
    tqs, tks = [6, 3], [2, 0]
    q, k, v, do, cu_q, cu_k = _packed(23, tqs, tks, 2, 1, 4)
    o, lse = oracle.attn_fwd_varlen(q, k, v, cu_q, cu_k, 0.5, True)
    dq, dk, dv, delta, _ = oracle.attn_bwd_varlen(q, k, v, do, cu_q, cu_k, 0.5, True)
    blind = list(range(0, 4)) + list(range(6, 9))  # rows 0..3 of seq 0, all of seq 1
    assert np.all(o[blind] == 0.0) and np.all(dq[blind] == 0.0) and np.all(delta[:, blind] == 0.0)
    assert np.all(np.isneginf(lse[:, blind]))
    assert np.all(np.isfinite(lse[:, 4:6])) and np.max(np.abs(o[4:6])) > 0.0
    # Row 4 sees key 0 only, row 5 both: O_4 is V_0 exactly.
    np.testing.assert_array_equal(o[4, 0], v[0, 0])
    # Non-causal: every row of seq 0 sees both keys.
    o_f, _ = oracle.attn_fwd_varlen(q, k, v, cu_q, cu_k, 0.5, False)
    assert np.all(np.abs(o_f[0:6]).sum(axis=-1) > 0.0) and np.all(o_f[6:9] == 0.0)


def test_varlen_finite_differences():
    """Central differences of L = sum(dO * O) over every entry of Q, K, V of a
    packed batch with a query row that sees no key and a key that no query
    sees match the packed backward."""
    tqs, tks = [3, 2], [2, 4]
    q, k, v, do, cu_q, cu_k = _packed(24, tqs, tks, 2, 1, 2)
    scale = 0.8
    dq, dk, dv, _, _ = oracle.attn_bwd_varlen(q, k, v, do, cu_q, cu_k, scale, True)

    def loss(args):
        o, _ = oracle.attn_fwd_varlen(args["q"], args["k"], args["v"], cu_q, cu_k, scale, True)
        return float(np.sum(do * o))

    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            base = {"q": q, "k": k, "v": v}
            fd[idx] = (loss({**base, name: xp}) - loss({**base, name: xm})) / (2 * h)
        assert np.max(np.abs(fd - grad)) <= 1e-6 * max(1.0, np.max(np.abs(grad))), name


def test_varlen_validates():
    q, k, v, _, cu_q, cu_k = _packed(25, [2, 3], [2, 3], 2, 1, 4)
    for bad_q, bad_k in (([1, 2, 5], cu_k), ([0, 3, 2, 5], [0, 2, 3, 5]), ([0, 2, 4], cu_k),
                         (cu_q, [0, 5])):
        with pytest.raises(ValueError):
            oracle.attn_fwd_varlen(q, k, v, bad_q, bad_k, 0.5, True)


# ------------------------------------------------------------ embedding-lookup gradient
def test_embed_grad_hand_case():
    """ids (2, 0, 2, 3): row 2 gets rows 0 and 2 of dY, row 0 gets row 1,
    row 3 gets row 3, row 1 nothing (exactly zero)."""
    ids = np.array([2, 0, 2, 3])
    dy = np.array([[1.0, -2.0, 0.5], [3.0, 4.0, -1.0], [5.0, 6.0, 2.0], [-7.0, 0.25, 8.0]])
    dw = oracle.embed_grad(ids, dy, 5)
    np.testing.assert_array_equal(dw, [[3.0, 4.0, -1.0], [0.0, 0.0, 0.0], [6.0, 4.0, 2.5],
                                       [-7.0, 0.25, 8.0], [0.0, 0.0, 0.0]])


def test_embed_grad_is_the_one_hot_product():
    """dW = onehot(ids)^T dY, the lookup's Jacobian transposed (a numpy fp64
    matrix product), on skewed ids with many repeats."""
    rng = np.random.default_rng(30)
    N, V, E = 700, 97, 13
    ids = np.minimum((rng.pareto(1.2, N) * 3).astype(np.int64), V - 1)
    dy = rng.standard_normal((N, E))
    onehot = np.zeros((N, V))
    onehot[np.arange(N), ids] = 1.0
    assert _rel(oracle.embed_grad(ids, dy, V), onehot.T @ dy) <= 1e-13
    # Column totals are kept, and a row no token selects is exactly zero.
    dw = oracle.embed_grad(ids, dy, V)
    assert _rel(dw.sum(axis=0), dy.sum(axis=0)) <= 1e-12
    unused = np.setdiff1d(np.arange(V), ids)
    assert unused.size > 0 and np.all(dw[unused] == 0.0)


def test_embed_grad_order_is_ascending_positions():
    """Each row is summed over its tokens in ascending position: a sum that
    rounds differently in another order shows which one was taken."""
    ids = np.array([1, 1, 1])
    dy = np.array([[1.0], [1e16], [-1e16]])
    # Ascending: (1 + 1e16) - 1e16 = 0 in fp64; descending would give 1.
    assert oracle.embed_grad(ids, dy, 2)[1, 0] == 0.0
    assert oracle.embed_grad(ids[::-1], dy[::-1], 2)[1, 0] == 1.0


def test_embed_grad_validates():
    with pytest.raises(ValueError):
        oracle.embed_grad([0, 5], np.zeros((2, 3)), 5)
    with pytest.raises(ValueError):
        oracle.embed_grad([-1, 0], np.zeros((2, 3)), 5)
    with pytest.raises(ValueError):
        oracle.embed_grad([0, 1, 2], np.zeros((2, 3)), 5)
    assert oracle.embed_grad([], np.zeros((0, 3)), 4).tolist() == [[0.0] * 3] * 4


# ------------------------------------------------------------ the pins catch planted mistakes
# Each entry plants one plausible mistake in a copy of the oracle's C source:
# (name, text in the source, its replacement, how often the text occurs).  A
# wrong sign, a dropped term or scale, a transposed operand, an off-by-one in
# the mask or a wrong head index anywhere in the forward, the backward, the
# row-sampling helpers or the standalone row dot must make at least one pin
# above fail.  The text must occur exactly as often as stated, so an edit of
# the oracle that moves a pattern fails here rather than testing nothing.
_MUTANTS = [
    ("mask_admits_next_key", "return causal ? i + 1 : T;",
     "return causal ? (i + 2 < T ? i + 2 : T) : T;", 1),
    ("causal_flag_ignored", "return causal ? i + 1 : T;", "return i + 1;", 1),
    ("score_scale_dropped", "const double s = scale * dot(qi, k + row_off(b, j, g, T, Hkv, D), D);",
     "const double s = dot(qi, k + row_off(b, j, g, T, Hkv, D), D);", 1),
    ("lse_without_row_max", "const double l = m + log(sum);", "const double l = log(sum);", 1),
    ("probs_from_max_not_lse", "p[j] = exp(p[j] - l);", "p[j] = exp(p[j] - m);", 1),
    ("scores_head_interleaved", "const int g = h / (Hq / Hkv);", "const int g = h % Hkv;", 1),
    ("fwd_values_head_interleaved", "weighted_values(p, v, b, h / G,",
     "weighted_values(p, v, b, h % Hkv,", 1),
    ("lse_in_base_2", "lse[((size_t)b * Hq + h) * T + i] = l;",
     "lse[((size_t)b * Hq + h) * T + i] = l * 1.4426950408889634;", 1),
    ("ds_sign_flipped", "const double ds = p[j] * (dp[j] - d1);",
     "const double ds = p[j] * (d1 - dp[j]);", 1),
    ("ds_delta_dropped", "const double ds = p[j] * (dp[j] - d1);", "const double ds = p[j] * dp[j];", 1),
    ("dk_from_do_not_q", "dkj[d] += ds * qi[d];", "dkj[d] += ds * doi[d];", 2),
    ("dv_weighted_by_ds", "dvj[d] += p[j] * doi[d];", "dvj[d] += ds * doi[d];", 1),
    ("dq_scale_dropped", "for (int d = 0; d < D; ++d) dqi[d] *= scale;", "", 2),
    ("dk_scale_dropped", "for (int d = 0; d < D; ++d) dkj[d] *= scale;", "", 2),
    ("dp_reads_kv_head_0", "dp[j] = dot(doi, v + row_off(b, j, g, T, Hkv, D), D);",
     "dp[j] = dot(doi, v + row_off(b, j, 0, T, Hkv, D), D);", 1),
    ("group_sum_first_head_only", "for (int h = g * G; h < (g + 1) * G; ++h)",
     "for (int h = g * G; h < g * G + 1; ++h)", 1),
    ("delta_from_do_do", "const double d1 = dot(doi, oi, D);", "const double d1 = dot(doi, doi, D);", 2),
    ("dq_weighted_by_p", "dqi[d] += ds * kj[d];", "dqi[d] += p[j] * kj[d];", 2),
    ("rowdot_do_squared",
     "dot(dout + row_off(b, i, h, T, H, D), o + row_off(b, i, h, T, H, D), D)",
     "dot(dout + row_off(b, i, h, T, H, D), dout + row_off(b, i, h, T, H, D), D)", 1),
    ("kv_rows_unscaled_score", "exp(scale * dot(qi, kj, D) - lse[(size_t)hh * T + i])",
     "exp(dot(qi, kj, D) - lse[(size_t)hh * T + i])", 1),
    ("kv_rows_range_starts_late", "for (int i = causal ? j : 0; i < T; ++i)",
     "for (int i = causal ? j + 1 : 0; i < T; ++i)", 1),
    ("rows_head_interleaved", "i = ri[s], g = h / G;", "i = ri[s], g = h % Hkv;", 1),
    ("varlen_mask_offset_flipped", "const int n = i + 1 + (tk - tq);",
     "const int n = i + 1 + (tq - tk);", 1),
    ("varlen_values_of_first_sequence",
     "seq_weighted_values(prob, v, cu_k[s], n, h / G, Hkv, D, o + packed_off(row, h, Hq, D));",
     "seq_weighted_values(prob, v, 0, n, h / G, Hkv, D, o + packed_off(row, h, Hq, D));", 1),
    ("varlen_blind_row_lse_zero", "*lse_out = -INFINITY;\n    return;", "*lse_out = 0.0;\n    return;", 1),
    ("varlen_group_interleaved", "for (int h = g * G; h < g * G + G; ++h)",
     "for (int h = g; h < Hq; h += Hkv)", 1),
    ("varlen_ds_sign_flipped", "const double dsc = prob[j] * (dprob[j] - dl);",
     "const double dsc = prob[j] * (dl - dprob[j]);", 1),
    ("varlen_dk_scale_dropped", "for (int d = 0; d < D; ++d) dkr[d] = dkr[d] * scale;", "", 1),
    ("varlen_dq_scale_dropped", "for (int d = 0; d < D; ++d) dqr[d] = dqr[d] * scale;", "", 1),
]

# Planted mistakes in embed_oracle.c (all stay in bounds).
_EMBED_MUTANTS = [
    ("embed_row_shifted", "dw[(size_t)ids[t] * E + col]", "dw[(size_t)((ids[t] + 1) % V) * E + col]", 1),
    ("embed_rows_reversed", "dy[(size_t)t * E + col]", "dy[(size_t)(N - 1 - t) * E + col]", 1),
    ("embed_columns_reversed", "dy[(size_t)t * E + col]", "dy[(size_t)t * E + (E - 1 - col)]", 1),
    ("embed_last_token_dropped", "for (int t = 0; t < N; ++t) dw", "for (int t = 0; t + 1 < N; ++t) dw", 1),
]

_SDPA_CASES = [(shape, causal) for shape in [(2, 37, 6, 2, 16), (1, 64, 4, 4, 32), (1, 1, 2, 1, 8)]
               for causal in (True, False)]
_PINS = [
    ("hand_derived", test_hand_derived_two_tokens, ()),
    ("uniform", test_uniform_attention_when_q_is_zero, ()),
    ("single_token", test_single_token, ()),
    ("constant_v", test_constant_v_rows, ()),
    ("softmax_causal", test_softmax_rows_sum_to_one_and_mask, (True,)),
    ("softmax_full", test_softmax_rows_sum_to_one_and_mask, (False,)),
    ("causality", test_causality_is_exact, ()),
    ("gqa2", test_gqa_is_repeated_kv_mha, (2,)),
    ("gqa3", test_gqa_is_repeated_kv_mha, (3,)),
    ("rowdot", test_rowdot_is_the_backward_delta, ()),
    ("delta_forms", test_delta_forms_agree, ()),
    ("fd_causal", test_finite_differences, (True,)),
    ("fd_full", test_finite_differences, (False,)),
    ("sdpa", lambda: [test_matches_torch_sdpa_fp64(s, c) for s, c in _SDPA_CASES], ()),
    ("sampled_rows", test_sampled_rows_match_full_oracle, ()),
    ("varlen_batched", test_varlen_equal_lengths_is_the_batched_oracle, ()),
    ("varlen_independent", test_varlen_sequences_are_independent, ()),
    ("varlen_torch_causal", test_varlen_cross_attention_matches_torch, (True,)),
    ("varlen_torch_full", test_varlen_cross_attention_matches_torch, (False,)),
    ("varlen_blind_rows", test_varlen_rows_that_see_no_key, ()),
    ("varlen_fd", test_varlen_finite_differences, ()),
    ("embed_hand", test_embed_grad_hand_case, ()),
    ("embed_one_hot", test_embed_grad_is_the_one_hot_product, ()),
    ("embed_order", test_embed_grad_order_is_ascending_positions, ()),
]


@pytest.mark.parametrize("source,name,old,new,count",
                         [pytest.param("attn_oracle.c", *m, id=m[0])
                          for m in [("unchanged", None, None, 0)] + _MUTANTS] +
                         [pytest.param("embed_oracle.c", *m, id=m[0]) for m in _EMBED_MUTANTS])
def test_pins_catch_planted_mistakes(source, name, old, new, count, tmp_path, monkeypatch):
    import os
    paths = []
    for src_path in oracle._SRCS:
        with open(src_path) as f:
            src = f.read()
        if os.path.basename(src_path) == source and old is not None:
            assert src.count(old) == count, name
            src = src.replace(old, new)
        paths.append(tmp_path / os.path.basename(src_path))
        paths[-1].write_text(src)
    lib = oracle._bind(ctypes.CDLL(oracle.compile_library([str(p) for p in paths],
                                                          str(tmp_path / f"{name}.so"))))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for pin, fn, args in _PINS:
        try:
            fn(*args)
        except AssertionError:
            caught.append(pin)
    if old is None:
        assert caught == [], f"the unchanged source, rebuilt, fails {caught}"
    else:
        assert caught, f"no pin catches the planted mistake {name}"
