"""Parity of the CUDA path (through the C-ABI) with the fp64 oracle.

Small and medium shapes are compared element by element against the full
oracle: several tiles per head, ragged tails (T not a multiple of 64 or 128),
T = 1 and 2, GQA group sizes 1..8, D = 64 and 128, causal and full attention.
The two largest workloads are run in the exact launch configuration the
benchmark times and compared on sampled rows the oracle computes one by one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from deterministic_attention_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import (assert_bwd_close, assert_fwd_close, rel_l2, run_gpu, to_np, widen,
                     TOL_FWD_REL)

pytestmark = pytest.mark.gpu


def _full_check(q, k, v, do, scale, causal, what):
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, scale, causal)
    qf, kf, vf, dof = (widen(t) for t in (q, k, v, do))
    o_r, lse_r = oracle.attn_fwd(qf, kf, vf, scale, causal)
    dq_r, dk_r, dv_r, _, _ = oracle.attn_bwd(qf, kf, vf, dof, scale, causal)
    assert_fwd_close(to_np(o), to_np(lse), o_r, lse_r, what)
    assert_bwd_close([("dQ", to_np(dq), dq_r), ("dK", to_np(dk), dk_r), ("dV", to_np(dv), dv_r)],
                     what)


@pytest.mark.parametrize("name", ["tiny", "small", "page3"])
def test_workload_full_oracle(name):
    w = WORKLOADS[name]
    q, k, v, do = workload_inputs(w)
    _full_check(q, k, v, do, w.softmax_scale, True, name)


RAGGED = [
    # B, T, Hq, Hkv, D, causal
    (1, 1, 2, 1, 64, True),
    (1, 2, 2, 2, 64, True),
    (1, 65, 4, 4, 64, True),
    (2, 127, 3, 1, 64, True),
    (1, 129, 8, 2, 64, True),
    (2, 200, 6, 2, 64, True),
    (1, 300, 8, 1, 64, True),
    (1, 385, 2, 1, 64, True),
    (1, 200, 4, 2, 64, False),
    (2, 129, 2, 1, 64, False),
    (1, 256, 4, 2, 128, True),
    (2, 200, 4, 1, 128, True),
    (1, 129, 2, 2, 128, True),
    (1, 1, 2, 1, 128, True),
    (1, 256, 2, 1, 128, False),
    (1, 190, 4, 4, 128, False),
]


@pytest.mark.parametrize("B,T,Hq,Hkv,D,causal", RAGGED)
def test_ragged_shapes(B, T, Hq, Hkv, D, causal):
    q, k, v, do = make_inputs(B, T, Hq, Hkv, D, seed=1000 + T + D + Hq, dout_std=0.5)
    _full_check(q, k, v, do, 1.0 / math.sqrt(D), causal, f"{(B, T, Hq, Hkv, D, causal)}")


def test_peaked_rows_small():
    """Rows with a few doubled keys (peaked softmax), D = 128, as in the
    long-context workload but short enough for the full oracle."""
    q, k, v, do = make_inputs(1, 640, 4, 1, 128, seed=44, dout_std=0.1, k_peak_frac=0.01)
    _full_check(q, k, v, do, 1.0 / math.sqrt(128), True, "peaked")


def test_large_scores_rescale_path():
    """Large scores (q scaled by 8) move the running maximum by more than the
    lazy-rescale threshold, exercising the O rescale in TMEM."""
    q, k, v, do = make_inputs(1, 512, 2, 1, 64, seed=45, dout_std=0.3, q_std=8.0)
    _full_check(q, k, v, do, 1.0 / 8.0, True, "large scores")


def _sampled_check(name, n_rows=96, n_groups=2, n_keys=12):
    w = WORKLOADS[name]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, w.softmax_scale, True)
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    qf, kf, vf, dof = (widen(t) for t in (q, k, v, do))
    rng = np.random.default_rng(7)
    B, T, Hq, Hkv, D = w.shape
    rows = [(0, 0, 0), (B - 1, Hq - 1, T - 1), (0, Hq - 1, 127), (B - 1, 0, 128)]
    rows += [(int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(T)))
             for _ in range(n_rows - len(rows))]
    o_r, lse_r, dq_r = oracle.attn_rows(qf, kf, vf, dof, rows, w.softmax_scale, True)
    o_g = np.stack([to_np(o[b, i, h]) for b, h, i in rows])
    lse_g = np.array([float(lse[b, h, i]) for b, h, i in rows])
    dq_g = np.stack([to_np(dq[b, i, h]) for b, h, i in rows])
    assert_fwd_close(o_g, lse_g, o_r, lse_r, f"{name} sampled rows")
    assert_bwd_close([("dQ", dq_g, dq_r)], f"{name} sampled rows")
    for gi in range(n_groups):
        b, g = (0, 0) if gi == 0 else (B - 1, Hkv - 1)
        js = sorted({0, T - 1, 128, 129} | {int(x) for x in rng.integers(T, size=n_keys - 4)})
        dk_r, dv_r = oracle.kv_rows(qf, kf, vf, dof, b, g, js, w.softmax_scale, True)
        dk_g = np.stack([to_np(dk[b, j, g]) for j in js])
        dv_g = np.stack([to_np(dv[b, j, g]) for j in js])
        assert_bwd_close([("dK", dk_g, dk_r), ("dV", dv_g, dv_r)], f"{name} kv group {b},{g}")


def test_wide_mha_sampled():
    _sampled_check("wide")


def test_long_context_sampled():
    _sampled_check("long", n_rows=64, n_groups=1, n_keys=10)


def test_delta_step_alone():
    """The backward's first step on seeded (O, dO, LSE): -Delta as fp32 sums
    against the fp64 rowsum, -LSE*log2(e) copied exactly, padding (-inf, -0)."""
    import deterministic_attention_gb300 as da
    for (B, T, H, D) in [(2, 333, 5, 64), (1, 129, 3, 128), (1, 1, 2, 64)]:
        o, _, _, do = make_inputs(B, T, H, H, D, seed=T)  # o: seeded bf16 standing in for O
        lse = torch.randn((B, H, T), generator=torch.Generator().manual_seed(T)) * 3 + 5
        ws = da.new_workspace(B, T, H, H, D)
        da.attn_bwd_delta(o.cuda(), do.cuda(), lse.cuda(), ws)
        torch.cuda.synchronize()
        rs = da.rowstats_view(ws, B, T, H).cpu()
        ref = oracle.rowdot(widen(o), widen(do))
        assert rel_l2(-to_np(rs[:, :, :T, 1]), ref) <= 1e-5
        assert torch.equal(rs[:, :, :T, 0], -(lse * 1.4426950408889634).to(torch.float32)) or \
            float((rs[:, :, :T, 0] + lse * 1.4426950408889634).abs().max()) <= 1e-5
        if rs.shape[2] > T:
            assert bool(torch.isneginf(rs[:, :, T:, 0]).all())
            assert bool((rs[:, :, T:, 1] == 0).all())


def test_causality_exact_on_gpu():
    """Perturbing keys/values after position i0 leaves O and LSE of rows <= i0
    bit-identical (masked keys contribute exactly nothing)."""
    q, k, v, do = make_inputs(1, 384, 4, 2, 64, seed=77)
    o1, lse1, *_ = run_gpu(q, k, v, do, 0.125, True)
    for i0 in (0, 100, 255):
        k2, v2 = k.clone(), v.clone()
        k2[:, i0 + 1:] = (k2[:, i0 + 1:].float() * -1.5 + 0.25).to(torch.bfloat16)
        v2[:, i0 + 1:] = (v2[:, i0 + 1:].float() * 2.0 - 1.0).to(torch.bfloat16)
        o2, lse2, *_ = run_gpu(q, k2, v2, do, 0.125, True)
        assert torch.equal(o1[:, : i0 + 1], o2[:, : i0 + 1])
        assert torch.equal(lse1[:, :, : i0 + 1], lse2[:, :, : i0 + 1])


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("B,T,Hq,Hkv,D,causal", [(2, 520, 6, 2, 64, True), (1, 300, 4, 1, 128, True),
                                                 (1, 256, 4, 4, 64, False)])
def test_dkdv_split_sizes(split, B, T, Hq, Hkv, D, causal):
    """Every dK/dV split (blocks per key tile, partial sums added in rank
    order through distributed shared memory) matches the oracle and repeats
    bit for bit."""
    import deterministic_attention_gb300 as da
    q, k, v, do = make_inputs(B, T, Hq, Hkv, D, seed=split * 100 + T, dout_std=0.2)
    da.set_dkdv_split(split)
    try:
        o, lse, dq, dk, dv = run_gpu(q, k, v, do, 1.0 / math.sqrt(D), causal)
        _, _, _, dk2, dv2 = run_gpu(q, k, v, do, 1.0 / math.sqrt(D), causal)
    finally:
        da.set_dkdv_split(0)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    qf, kf, vf, dof = (widen(t) for t in (q, k, v, do))
    _, dk_r, dv_r, _, _ = oracle.attn_bwd(qf, kf, vf, dof, 1.0 / math.sqrt(D), causal)
    assert_bwd_close([("dK", to_np(dk), dk_r), ("dV", to_np(dv), dv_r)], f"split {split}")


@pytest.mark.parametrize("split,D", [(1, 64), (2, 64), (4, 64), (8, 64), (1, 128), (2, 128)])
def test_dkdv_clusters_walk_several_tiles(split, D):
    """The persistent dK/dV launch with more key tiles than resident clusters:
    every cluster walks several tiles (the plain walk: every tile shared by
    its cluster), the last ones small enough that some blocks of a cluster
    get no items of them.  Sampled key rows of early and late tiles match the
    oracle, and the whole result repeats bit for bit."""
    import deterministic_attention_gb300 as da
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T, Hq, Hkv = 1024, 3, 1
    B = max(2, -(-5 * sms // (2 * split * (T // 128))))  # about 2.5 tiles per cluster
    q, k, v, do = make_inputs(B, T, Hq, Hkv, D, seed=77 + split + D, dout_std=0.2)
    scale = 1.0 / math.sqrt(D)
    da.set_dkdv_split(split)
    da.set_dkdv_deal(1)
    try:
        _, _, _, dk, dv = run_gpu(q, k, v, do, scale, True)
        _, _, _, dk2, dv2 = run_gpu(q, k, v, do, scale, True)
    finally:
        da.set_dkdv_split(0)
        da.set_dkdv_deal(0)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    js = [0, 131, 640, 897, 1023]
    for b in (0, B - 1):
        qf, kf, vf, dof = (widen(t[b:b + 1]) for t in (q, k, v, do))
        dk_r, dv_r = oracle.kv_rows(qf, kf, vf, dof, 0, 0, js, scale, True)
        got_k = to_np(dk[b:b + 1, js, 0])[0]
        got_v = to_np(dv[b:b + 1, js, 0])[0]
        assert_bwd_close([("dK", got_k, dk_r), ("dV", got_v, dv_r)], f"split {split} D {D} b {b}")


@pytest.mark.parametrize("split", [2, 4, 8])
def test_dkdv_listed_deal(split):
    """The listed dK/dV deal (D = 64): the heaviest key tiles shared by a
    cluster, lighter ones taken whole by single blocks that store all their
    rows.  Sampled key rows of shared and whole tiles match the oracle, the
    result repeats bit for bit, and the plain walk of the same tiles agrees
    within the same tolerance."""
    import deterministic_attention_gb300 as da
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T, Hq, Hkv, D = 1024, 3, 1, 64
    B = max(2, -(-5 * sms // (2 * split * (T // 128))))
    q, k, v, do = make_inputs(B, T, Hq, Hkv, D, seed=91 + split, dout_std=0.2)
    scale = 1.0 / math.sqrt(D)
    ng = min(B * Hkv * (T // 128), sms // split)
    lists = da.diag_dkdv_list(B, T, Hq, Hkv, True, split, ng, force=True)
    assert lists is not None
    kinds = {sh for lst in lists for _, sh in lst}
    assert kinds == {True, False}, kinds
    da.set_dkdv_split(split)
    try:
        da.set_dkdv_deal(2)
        _, _, _, dk, dv = run_gpu(q, k, v, do, scale, True)
        _, _, _, dk2, dv2 = run_gpu(q, k, v, do, scale, True)
        da.set_dkdv_deal(1)
        _, _, _, dk3, dv3 = run_gpu(q, k, v, do, scale, True)
    finally:
        da.set_dkdv_split(0)
        da.set_dkdv_deal(0)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert_bwd_close([("dK", to_np(dk), to_np(dk3)), ("dV", to_np(dv), to_np(dv3))],
                     f"listed vs plain, split {split}")
    js = [0, 131, 640, 897, 1023]
    for b in (0, B - 1):
        qf, kf, vf, dof = (widen(t[b:b + 1]) for t in (q, k, v, do))
        dk_r, dv_r = oracle.kv_rows(qf, kf, vf, dof, 0, 0, js, scale, True)
        got_k = to_np(dk[b:b + 1, js, 0])[0]
        got_v = to_np(dv[b:b + 1, js, 0])[0]
        assert_bwd_close([("dK", got_k, dk_r), ("dV", got_v, dv_r)], f"listed, split {split} b {b}")


def test_fma_pipe_exp2_error_bound():
    """The polynomial 2^x used for part of the exponentials: relative error
    <= 1e-4 against exact 2^x over the range the kernels feed it, the pair
    form bit-identical to the scalar form, and agreement with the
    special-function unit's ex2.approx to the same bound."""
    import numpy as np
    import deterministic_attention_gb300 as da
    xs = np.concatenate([np.linspace(-126.0, 8.0, 200001), np.array([-300.0, -126.5, -0.5, 0.5])])
    x = torch.tensor(xs, dtype=torch.float32, device="cuda")
    yp, y2, ys = (t.cpu().double().numpy() for t in da.diag_exp2(x))
    xf = x.cpu().double().numpy()
    assert np.array_equal(yp, y2)
    assert np.all(yp > 0)
    normal = xf >= -125.0  # below, the clamp at -126 leaves values under 2^-124
    assert np.max(np.abs(yp[normal] / np.exp2(xf[normal]) - 1.0)) <= 1e-4
    assert np.all(yp[~normal] <= 2.0 ** -124)
    live = xf > -120.0
    assert np.max(np.abs(yp[live] / ys[live] - 1.0)) <= 1e-4


@pytest.mark.parametrize("name", ["small", "page3", "1152-units"])
def test_dq_dynamic_and_static_deal_agree_bitwise(name):
    """With the full workspace the dQ step takes its query tiles from a counter
    (whichever block is ready first); with a workspace that holds only the row
    statistics it follows the static deal (a host list up to 1,024 tiles, past
    that rounds dealt forward and backward in turn: the 1152-unit case).  A
    tile's arithmetic does not depend on the block that computes it, so dq is
    bit-identical either way, and it matches the oracle."""
    import deterministic_attention_gb300 as da
    from helpers import sha256
    if name == "1152-units":
        B, T, Hq, Hkv, D = 12, 1024, 12, 4, 64
        q, k, v, do = make_inputs(B, T, Hq, Hkv, D, seed=13, dout_std=0.1)
        scale = 1.0 / math.sqrt(D)
    else:
        w = WORKLOADS[name]
        q, k, v, do = workload_inputs(w)
        B, T, Hq, Hkv, D = w.shape
        scale = w.softmax_scale
    tp = -(-T // 128) * 128
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = da.attn_fwd(qc, kc, vc, scale=scale)
    out = {}
    for label, nbytes in (("dynamic", da.workspace_bytes(B, T, Hq, Hkv, D)), ("static", B * Hq * tp * 8)):
        ws = torch.empty((nbytes,), dtype=torch.uint8, device="cuda")
        res = [da.attn_bwd(qc, kc, vc, o, lse, doc, scale=scale, workspace=ws) for _ in range(2)]
        torch.cuda.synchronize()
        assert [sha256(t) for t in res[0]] == [sha256(t) for t in res[1]], label
        out[label] = res[0]
    # The steps one by one: one Delta, then the dQ step twice on the same
    # workspace (each dQ call leaves the tile counter as it found it).
    ws = da.new_workspace(B, T, Hq, Hkv, D)
    da.attn_bwd_delta(o, doc, lse, ws)
    dq_a = da.attn_bwd_dq(qc, kc, vc, doc, ws, scale=scale)
    dq_b = da.attn_bwd_dq(qc, kc, vc, doc, ws, scale=scale)
    torch.cuda.synchronize()
    da.check_status()
    assert sha256(dq_a) == sha256(dq_b) == sha256(out["dynamic"][0])
    assert [sha256(t) for t in out["dynamic"]] == [sha256(t) for t in out["static"]]
    dq = out["dynamic"][0]
    rows = [(0, 0, T - 1), (B - 1, Hq - 1, T // 2), (0, Hq // 2, 0), (B - 1, 1, 129)]
    _, _, dq_r = oracle.attn_rows(widen(q), widen(k), widen(v), widen(do), rows, scale, True)
    dq_g = np.stack([to_np(dq[b, i, h]) for b, h, i in rows])
    assert_bwd_close([("dQ", dq_g, dq_r)], f"{name} sampled rows")


def test_dq_reports_a_counter_not_cleared():
    """attn_bwd_dq on a workspace that attn_bwd_delta never touched (its tile
    counter holds garbage) is reported through the status check; after
    attn_bwd_delta the same workspace works."""
    import deterministic_attention_gb300 as da
    B, T, Hq, Hkv, D = 1, 384, 4, 2, 64
    q, k, v, do = (t.cuda() for t in make_inputs(B, T, Hq, Hkv, D, seed=11))
    o, lse = da.attn_fwd(q, k, v)
    ws = torch.full((da.workspace_bytes(B, T, Hq, Hkv, D),), 0xFF, dtype=torch.uint8, device="cuda")
    da.attn_bwd_dq(q, k, v, do, ws)
    with pytest.raises(da.DetAttnError) as err:
        da.check_status()
    assert err.value.code == -9 and "not cleared" in str(err.value)
    da.attn_bwd_delta(o, do, lse, ws)
    dq = da.attn_bwd_dq(q, k, v, do, ws)
    da.check_status()
    dq_ref, _, _ = da.attn_bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq_ref)
