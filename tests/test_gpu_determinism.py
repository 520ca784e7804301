"""Bitwise run-to-run reproducibility and memory hygiene of the CUDA path.

Reproducibility (oxide-train README, "The trainer is not bit-identical to
itself after step 1": atomic accumulation makes two runs of the same program
disagree): 20 forward+backward calls on the same device buffers, with every
output refilled by a different garbage pattern before each call, must give the
same SHA-256 of O, LSE, dQ, dK and dV.  A second process must reproduce the
digests.  Guard regions around every output must stay untouched.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

import deterministic_attention_gb300 as da
from deterministic_attention_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from helpers import sha256

pytestmark = pytest.mark.gpu

_GARBAGE = [0xFF, 0x00, 0x7F, 0xAA, 0x55, 0xC3]


def _fill_garbage(ts, run):
    for n, t in enumerate(ts):
        pat = _GARBAGE[(run + n) % len(_GARBAGE)]
        t.view(torch.uint8).fill_(pat)
        if run % 3 == 2:  # NaN bit patterns
            if t.dtype == torch.float32:
                t.fill_(float("nan"))
            else:
                t.view(torch.int16).fill_(0x7FC1)


def _digests(name, runs):
    w = WORKLOADS[name]
    q, k, v, do = (t.cuda() for t in workload_inputs(w))
    B, T, Hq, Hkv, D = w.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((da.workspace_bytes(*w.shape),), dtype=torch.uint8, device="cuda")
    out = []
    for r in range(runs):
        _fill_garbage([o, lse, dq, dk, dv, ws], r)
        da.attn_fwd(q, k, v, scale=w.softmax_scale, out=o, lse=lse)
        da.attn_bwd(q, k, v, o, lse, do, scale=w.softmax_scale, dq=dq, dk=dk, dv=dv, workspace=ws)
        torch.cuda.synchronize()
        out.append({n: sha256(t) for n, t in (("O", o), ("LSE", lse), ("dQ", dq), ("dK", dk),
                                               ("dV", dv))})
    da.check_status()
    return out


@pytest.mark.parametrize("name,runs", [("page3", 20), ("small", 20), ("long", 20)])
def test_twenty_runs_bit_identical(name, runs):
    d = _digests(name, runs)
    for r in range(1, runs):
        assert d[r] == d[0], f"run {r} differs: {d[r]} vs {d[0]}"


def test_second_process_reproduces_digests():
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import sys, json; sys.path.insert(0, %r); sys.path.insert(0, %r);"
            "import test_gpu_determinism as t; print(json.dumps(t._digests('page3', 1)[0]))"
            % (here, os.path.dirname(here)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    other = json.loads(r.stdout.strip().splitlines()[-1])
    assert other == _digests("page3", 1)[0]


def _guarded(shape, dtype, guard=4096):
    n = 1
    for s in shape:
        n *= s
    buf = torch.empty((n + 2 * guard,), dtype=dtype, device="cuda")
    buf.view(torch.uint8).fill_(0xA5)
    return buf, buf[guard:guard + n].view(shape), guard


@pytest.mark.parametrize("B,T,Hq,Hkv,D", [(2, 200, 6, 2, 64), (1, 129, 4, 1, 128),
                                          (1, 1, 2, 1, 64), (3, 65, 2, 2, 64)])
def test_outputs_stay_in_bounds(B, T, Hq, Hkv, D):
    q, k, v, do = (t.cuda() for t in make_inputs(B, T, Hq, Hkv, D, seed=5))
    bufs = {}
    for name, shape, dt in (("o", (B, T, Hq, D), torch.bfloat16), ("lse", (B, Hq, T), torch.float32),
                            ("dq", (B, T, Hq, D), torch.bfloat16), ("dk", (B, T, Hkv, D), torch.bfloat16),
                            ("dv", (B, T, Hkv, D), torch.bfloat16)):
        bufs[name] = _guarded(shape, dt)
    nws = da.workspace_bytes(B, T, Hq, Hkv, D)
    wsb = torch.empty((nws + 2 * 4096,), dtype=torch.uint8, device="cuda").fill_(0xA5)
    ws = wsb[4096:4096 + nws]
    da.attn_fwd(q, k, v, out=bufs["o"][1], lse=bufs["lse"][1])
    da.attn_bwd(q, k, v, bufs["o"][1], bufs["lse"][1], do, dq=bufs["dq"][1], dk=bufs["dk"][1],
                dv=bufs["dv"][1], workspace=ws)
    torch.cuda.synchronize()
    for name, (buf, view, guard) in bufs.items():
        raw = buf.view(torch.uint8)
        esz = buf.element_size()
        head = raw[: guard * esz]
        tail = raw[raw.numel() - guard * esz:]
        assert bool((head == 0xA5).all()) and bool((tail == 0xA5).all()), f"{name} guard overwritten"
    assert bool((wsb[:4096] == 0xA5).all()) and bool((wsb[4096 + nws:] == 0xA5).all())


def test_empty_problem_launches_nothing():
    q = torch.empty((0, 128, 2, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((0, 128, 1, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = da.attn_fwd(q, k, k)
    assert o.shape == q.shape and lse.shape == (0, 2, 128)
    q = torch.empty((2, 0, 2, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((2, 0, 1, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = da.attn_fwd(q, k, k)
    dq, dk, dv = da.attn_bwd(q, k, k, o, lse, q)
    assert dq.shape == q.shape
    da.check_status()


def test_device_wait_timeout_is_reported_and_context_survives():
    """A bounded device wait that can never complete gives up, the host reads
    DETATTN_ERR_DEVICE_TIMEOUT, and the next attention call still works."""
    da.check_status()  # clean slate
    da.selftest_wait_timeout(50_000_000)  # 50 ms
    with pytest.raises(da.DetAttnError) as e:
        da.check_status()
    assert e.value.code == -7
    da.check_status()  # the word was cleared
    q, k, v, do = (t.cuda() for t in make_inputs(1, 256, 2, 1, 64, seed=3))
    o, lse = da.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    da.check_status()
    assert torch.isfinite(o.float()).all()
