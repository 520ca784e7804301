"""The stored-dS backward (the dK/dV step stores dS, the dQ step is one
tensor-core product per tile): full-oracle parity at the tolerances of the
other parity tests, dK and dV bit-identical to the recompute form (the dK/dV
arithmetic is the same), ragged and full-attention shapes, D = 128, and
20-run SHA-256 identity at the page-3 shape."""
import math

import pytest
import torch

import deterministic_attention_gb300 as da
import oracle
from deterministic_attention_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import assert_bwd_close, sha256, to_np, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def stored_mode():
    da.set_bwd_dq_mode(1)
    yield
    da.set_bwd_dq_mode(0)


def _both(q, k, v, do, scale, causal):
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = da.attn_fwd(qd, kd, vd, scale=scale, causal=causal)
    ws_ds = da.new_workspace(B, T, Hq, Hkv, D, stored_ds=True, causal=causal)
    assert ws_ds.numel() == da.ds_workspace_bytes(B, T, Hq, Hkv, D, causal)
    stored = da.attn_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal, workspace=ws_ds)
    da.set_bwd_dq_mode(0)
    plain = da.attn_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal, workspace=ws_ds)
    da.set_bwd_dq_mode(1)
    torch.cuda.synchronize()
    da.check_status()
    return [t.cpu() for t in stored], [t.cpu() for t in plain]


def _check(q, k, v, do, scale, causal, what):
    (dq, dk, dv), (_, dk0, dv0) = _both(q, k, v, do, scale, causal)
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0), f"{what}: dK/dV differ between forms"
    qf, kf, vf, dof = (widen(t) for t in (q, k, v, do))
    dq_r, dk_r, dv_r, _, _ = oracle.attn_bwd(qf, kf, vf, dof, scale, causal)
    assert_bwd_close([("dQ", to_np(dq), dq_r), ("dK", to_np(dk), dk_r), ("dV", to_np(dv), dv_r)],
                     what)


@pytest.mark.parametrize("name", ["tiny", "small", "page3"])
def test_stored_ds_workloads_full_oracle(name):
    w = WORKLOADS[name]
    q, k, v, do = workload_inputs(w)
    _check(q, k, v, do, w.softmax_scale, True, name)


@pytest.mark.parametrize("B,T,Hq,Hkv,D,causal", [
    (1, 1, 2, 1, 64, True),
    (1, 65, 4, 4, 64, True),
    (2, 200, 6, 2, 64, True),
    (1, 385, 2, 1, 64, True),
    (2, 129, 2, 1, 64, False),
    (1, 256, 4, 2, 128, True),
    (1, 190, 4, 4, 128, False),
])
def test_stored_ds_ragged(B, T, Hq, Hkv, D, causal):
    q, k, v, do = make_inputs(B, T, Hq, Hkv, D, seed=2000 + T + D, dout_std=0.5)
    _check(q, k, v, do, 1.0 / math.sqrt(D), causal, f"{(B, T, Hq, Hkv, D, causal)}")


def test_stored_ds_twenty_runs_bit_identical():
    w = WORKLOADS["page3"]
    q, k, v, do = (t.cuda() for t in workload_inputs(w))
    B, T, Hq, Hkv, D = w.shape
    o, lse = da.attn_fwd(q, k, v, scale=w.softmax_scale)
    ws = da.new_workspace(B, T, Hq, Hkv, D, stored_ds=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    digests = set()
    for r in range(20):
        for t in (dq, dk, dv):
            t.view(torch.int16).fill_(0x7FC0 + r)
        ws.fill_((29 * r + 3) % 256)
        da.attn_bwd(q, k, v, o, lse, do, scale=w.softmax_scale, dq=dq, dk=dk, dv=dv, workspace=ws)
        torch.cuda.synchronize()
        digests.add((sha256(dq), sha256(dk), sha256(dv)))
    da.check_status()
    assert len(digests) == 1
