"""GPU parity and run-to-run identity of the deterministic embedding-lookup
gradient (embed_grad) against the fp64 oracle (oracle.embed_grad).

Tolerance, derived from the arithmetic: every dy value is a bf16 number, exact
in fp32, and the kernel adds the L tokens of an id in some fixed order in
fp32.  Each of the L - 1 additions rounds with relative error at most
u = 2^-24, so |gpu - exact| <= (L - 1) u sum_t |dy[t, c]| to first order; the
test allows L u sum |dy| (which also covers the second-order term).  An id
with one token is exact, and a row no token selects is exactly zero.
"""
import hashlib

import numpy as np
import pytest
import torch

import deterministic_attention_gb300 as da
import oracle
from deterministic_attention_gb300.inputs import EMBED_GRAD, make_embed_grad_inputs
from helpers import widen

U = 2.0 ** -24


def _check_against_oracle(ids, dy, V, dw):
    """Element-wise bound above; ids, dy on the CPU, dw the GPU result."""
    ids_np = ids.numpy().astype(np.int32)
    dyf = widen(dy)
    ref = oracle.embed_grad(ids_np, dyf, V)
    mag = oracle.embed_grad(ids_np, np.abs(dyf), V)
    counts = np.bincount(ids_np[(ids_np >= 0) & (ids_np < V)], minlength=V).astype(np.float64)
    got = dw.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    bound = counts[:, None] * U * mag
    bad = err > bound
    assert not bad.any(), (f"{int(bad.sum())} elements past the bound; worst excess "
                           f"{float((err - bound).max()):.3g}")
    assert np.all(got[counts == 0] == 0.0), "a row no token selects is not zero"
    single = counts == 1
    assert np.array_equal(got[single], ref[single]), "one-token rows must be exact"
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else 0.0


def _digest(t):
    return hashlib.sha256(t.contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()


@pytest.mark.gpu
@pytest.mark.parametrize("dist", ["uniform", "zipf"])
def test_embed_grad_full_size_matches_oracle(dist):
    """The trainer's shape: 32 x 1024 tokens, 50,432 rows (50,257 used), 1536 wide."""
    w = EMBED_GRAD
    ids, dy = make_embed_grad_inputs(w["N"], w["V_used"], w["E"], w["seed"], dist)
    dw = torch.full((w["V"], w["E"]), float("nan"), device="cuda")
    da.embed_grad(ids.cuda(), dy.cuda(), w["V"], dw=dw)
    torch.cuda.synchronize()
    da.check_status()
    rel = _check_against_oracle(ids, dy, w["V"], dw)
    assert rel < 1e-6, rel


@pytest.mark.gpu
@pytest.mark.parametrize("dist", ["uniform", "zipf"])
def test_embed_grad_twenty_runs_bit_identical(dist):
    """20 calls on the same inputs, dw and workspace refilled with a different
    garbage pattern before each: identical SHA-256 every time."""
    w = EMBED_GRAD
    ids, dy = make_embed_grad_inputs(w["N"], w["V_used"], w["E"], w["seed"] + 1, dist)
    ids, dy = ids.cuda(), dy.cuda()
    dw = torch.empty((w["V"], w["E"]), dtype=torch.float32, device="cuda")
    ws = torch.empty(da.embed_grad_workspace_bytes(w["N"], w["V"], w["E"]), dtype=torch.uint8,
                     device="cuda")
    digests = set()
    for r in range(20):
        dw.view(torch.int32).fill_(0x7FC00000 + r)
        ws.fill_((37 * r + 11) % 256)
        da.embed_grad(ids, dy, w["V"], dw=dw, workspace=ws)
        torch.cuda.synchronize()
        digests.add(_digest(dw))
    da.check_status()
    assert len(digests) == 1


@pytest.mark.gpu
@pytest.mark.parametrize("N,V,E,kind", [
    (0, 7, 128, "uniform"),         # no tokens: dw is all zeros
    (1, 1, 4, "uniform"),           # one token, one row, one column group
    (5000, 3, 520, "one_id"),       # one id takes every token: 157 runs; partial slab (130 groups)
    (777, 50, 1032, "uniform"),     # ragged run count, second slab partial
    (4096, 64, 256, "sorted"),      # ids already sorted: segments end exactly on run edges
    (3000, 4000, 128, "zipf"),
])
def test_embed_grad_edge_cases(N, V, E, kind):
    g = torch.Generator().manual_seed(N + V + E)
    if kind == "one_id":
        ids = torch.full((N,), 1, dtype=torch.int32)
    elif kind == "sorted":
        ids = (torch.arange(N, dtype=torch.int32) // 64) % V
    elif kind == "zipf":
        ids, _ = make_embed_grad_inputs(N, V, 4, seed=5, dist="zipf")
    else:
        ids = torch.randint(0, V, (N,), generator=g, dtype=torch.int32)
    dy = torch.randn((N, E), generator=g).to(torch.bfloat16)
    dw = torch.full((V, E), float("nan"), device="cuda")
    da.embed_grad(ids.cuda(), dy.cuda(), V, dw=dw)
    torch.cuda.synchronize()
    da.check_status()
    _check_against_oracle(ids, dy, V, dw)


@pytest.mark.gpu
def test_embed_grad_reports_ids_out_of_range():
    """Ids outside [0, V) are left out (never used as an index) and reported
    by detattn_check_status; the other tokens' gradient is unchanged."""
    N, V, E = 300, 20, 64
    g = torch.Generator().manual_seed(3)
    ids = torch.randint(0, V, (N,), generator=g, dtype=torch.int32)
    ids[7], ids[100], ids[299] = -1, V, 1 << 30
    dy = torch.randn((N, E), generator=g).to(torch.bfloat16)
    dw = da.embed_grad(ids.cuda(), dy.cuda(), V)
    torch.cuda.synchronize()
    with pytest.raises(da.DetAttnError) as ei:
        da.check_status()
    assert ei.value.code == -10
    keep = (ids >= 0) & (ids < V)
    _check_against_oracle(ids[keep], dy[keep], V, dw)
    da.check_status()  # the word was cleared
