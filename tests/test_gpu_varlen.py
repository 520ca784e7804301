"""GPU parity of the packed variable-length calls (attn_fwd_varlen,
attn_bwd_varlen) against the fp64 oracle's varlen functions, with the
tolerances of the fixed-length tests (O, LSE rel-L2 <= 5e-3 and max-abs <=
2e-2; dQ, dK, dV rel-L2 <= 1e-2), exact values where the reading fixes them
(rows that see no key: O = 0, LSE = -inf, dQ = 0; keys no query sees: dK =
dV = 0), identity with the fixed-length kernels at equal lengths, and 20-run
SHA-256 identity."""
import math

import numpy as np
import pytest
import torch

import deterministic_attention_gb300 as da
import oracle
from deterministic_attention_gb300.inputs import (VARLEN_PAGE3, make_inputs, make_varlen_inputs,
                                                  varlen_page3_inputs)
from helpers import assert_bwd_close, assert_fwd_close, sha256, to_np, widen


def _run(q, k, v, do, cu_q, cu_k, scale, causal):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = da.attn_fwd_varlen(qd, kd, vd, cu_q, cu_k, scale=scale, causal=causal)
    dq, dk, dv = da.attn_bwd_varlen(qd, kd, vd, o, lse, dod, cu_q, cu_k, scale=scale,
                                    causal=causal)
    torch.cuda.synchronize()
    da.check_status()
    return tuple(t.cpu() for t in (o, lse, dq, dk, dv))


def _check(tqs, tks, Hq, Hkv, D, causal, seed=11, dout_std=0.3):
    q, k, v, do, cu_q, cu_k = make_varlen_inputs(tqs, tks, Hq, Hkv, D, seed, dout_std)
    scale = 1.0 / math.sqrt(D)
    o, lse, dq, dk, dv = _run(q, k, v, do, cu_q, cu_k, scale, causal)
    qf, kf, vf, dof = (widen(t) for t in (q, k, v, do))
    o_r, lse_r = oracle.attn_fwd_varlen(qf, kf, vf, cu_q, cu_k, scale, causal)
    dq_r, dk_r, dv_r, _, _ = oracle.attn_bwd_varlen(qf, kf, vf, dof, cu_q, cu_k, scale, causal)
    lse_np, lse_rn = to_np(lse), np.asarray(lse_r)
    blind = ~np.isfinite(lse_rn)
    # Rows that see no key: exact values.
    assert np.all(lse_np[blind] == -np.inf), "a row that sees no key must get LSE = -inf"
    assert np.array_equal(np.isfinite(lse_np), ~blind)
    bl_rows = blind.T  # [total_q, Hq]
    assert np.all(to_np(o)[bl_rows] == 0.0) and np.all(to_np(dq)[bl_rows] == 0.0)
    if (~blind).any():
        assert_fwd_close(to_np(o), lse_np[~blind], o_r, lse_rn[~blind], f"varlen {tqs}/{tks}")
    # Keys no query sees: exactly zero gradients.
    seen_none = np.all(np.asarray(dk_r) == 0.0, axis=-1) & np.all(np.asarray(dv_r) == 0.0, axis=-1)
    assert np.all(to_np(dk)[seen_none] == 0.0) and np.all(to_np(dv)[seen_none] == 0.0)
    pairs = [(n, to_np(x), r) for n, x, r in (("dQ", dq, dq_r), ("dK", dk, dk_r), ("dV", dv, dv_r))
             if np.linalg.norm(r) > 0]
    assert_bwd_close(pairs, f"varlen {tqs}/{tks}")
    return o, lse, dq, dk, dv


@pytest.mark.gpu
def test_varlen_page3_workload_matches_oracle():
    """4,096 tokens cut into sequences of 64..1,024 (seed 5), page-3 heads."""
    w = VARLEN_PAGE3
    q, k, v, do, cu_q, cu_k = varlen_page3_inputs()
    scale = 1.0 / math.sqrt(w["D"])
    o, lse, dq, dk, dv = _run(q, k, v, do, cu_q, cu_k, scale, True)
    qf, kf, vf, dof = (widen(t) for t in (q, k, v, do))
    o_r, lse_r = oracle.attn_fwd_varlen(qf, kf, vf, cu_q, cu_k, scale, True)
    dq_r, dk_r, dv_r, _, _ = oracle.attn_bwd_varlen(qf, kf, vf, dof, cu_q, cu_k, scale, True)
    assert_fwd_close(to_np(o), to_np(lse), o_r, lse_r, "varlen page3")
    assert_bwd_close([("dQ", to_np(dq), dq_r), ("dK", to_np(dk), dk_r), ("dV", to_np(dv), dv_r)],
                     "varlen page3")


@pytest.mark.gpu
@pytest.mark.parametrize("tqs,tks,Hq,Hkv,D,causal", [
    ([300], [100], 4, 2, 64, True),               # tq > tk: rows that see no key
    ([100], [300], 4, 2, 64, True),               # tq < tk
    ([0, 129, 0, 1, 77], [0, 129, 5, 1, 200], 6, 2, 64, True),   # empty, one-token, keys-only
    ([1, 2, 3], [1, 2, 3], 2, 1, 64, True),       # tiny sequences
    ([257, 64, 383], [90, 500, 383], 3, 1, 64, False),           # cross-attention, no mask
    ([200, 31], [50, 260], 8, 8, 64, True),       # MHA, mixed directions
    ([130, 260], [300, 10], 4, 2, 128, True),     # D = 128, rows without keys
    ([500], [0], 2, 1, 64, True),                 # no keys at all
])
def test_varlen_edge_cases(tqs, tks, Hq, Hkv, D, causal):
    _check(tqs, tks, Hq, Hkv, D, causal)


@pytest.mark.gpu
@pytest.mark.parametrize("split", [1, 2])
def test_varlen_d128_both_dkdv_kernels(split):
    """D = 128 packed batches through both dK/dV kernels: one block per key
    tile (128-query items, P^T and dS^T over the score columns) and a key tile
    split over two blocks (64-query items, partial sums exchanged)."""
    da.set_dkdv_split(split)
    try:
        _check([130, 260, 77, 0], [300, 10, 200, 64], 4, 2, 128, True)
        _check([257, 64], [90, 500], 2, 2, 128, False)
    finally:
        da.set_dkdv_split(0)


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
def test_varlen_equal_lengths_match_fixed_length_kernels(D):
    """B sequences of length T packed: O, LSE and dQ are the fixed-length
    call's bits (a query tile's arithmetic does not depend on its schedule);
    dK, dV agree within tolerance (their cluster split may differ)."""
    B, T, Hq, Hkv = 3, 333, 4, 2
    q, k, v, do = make_inputs(B, T, Hq, Hkv, D, seed=21, dout_std=0.3)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = da.attn_fwd(qd, kd, vd, scale=scale)
    dq, dk, dv = da.attn_bwd(qd, kd, vd, o, lse, dod, scale=scale)
    cu = [T * i for i in range(B + 1)]
    flat = lambda t: t.reshape(B * T, t.shape[2], D)
    o2, lse2, dq2, dk2, dv2 = _run(flat(q), flat(k), flat(v), flat(do), cu, cu, scale, True)
    assert torch.equal(o2, flat(o).cpu())
    assert torch.equal(lse2, lse.permute(1, 0, 2).reshape(Hq, B * T).cpu())
    assert torch.equal(dq2, flat(dq).cpu())
    assert_bwd_close([("dK", to_np(dk2), to_np(flat(dk).cpu())),
                      ("dV", to_np(dv2), to_np(flat(dv).cpu()))], "packed vs fixed")


@pytest.mark.gpu
def test_varlen_twenty_runs_bit_identical():
    q, k, v, do, cu_q, cu_k = varlen_page3_inputs()
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    digests = set()
    for r in range(20):
        for t in (o, dq, dk, dv):
            t.view(torch.int16).fill_(0x7FC0 + r)
        lse.fill_(float(r) - 7.5)
        da.attn_fwd_varlen(qd, kd, vd, cu_q, cu_k, out=o, lse=lse)
        da.attn_bwd_varlen(qd, kd, vd, o, lse, dod, cu_q, cu_k, dq=dq, dk=dk, dv=dv)
        torch.cuda.synchronize()
        digests.add(tuple(sha256(t) for t in (o, lse, dq, dk, dv)))
    da.check_status()
    assert len(digests) == 1
