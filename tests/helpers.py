"""Shared helpers of the GPU tests: tolerances, error metrics, running the CUDA
path on seeded inputs and widening those inputs for the oracle."""
from __future__ import annotations

import hashlib

import numpy as np
import torch

import oracle
from deterministic_attention_gb300.inputs import bf16_bits

# Tolerances (bf16 inputs, fp32 accumulation): O and LSE rel-L2 <= 5e-3 and
# max-abs <= 2e-2; dQ, dK, dV rel-L2 <= 1e-2.
TOL_FWD_REL = 5e-3
TOL_FWD_ABS = 2e-2
TOL_BWD_REL = 1e-2


def widen(t: torch.Tensor) -> np.ndarray:
    """bf16 CPU tensor -> exact fp64 numpy array (for the oracle)."""
    return oracle.bf16_bits_to_f64(bf16_bits(t)).reshape(tuple(t.shape))


def rel_l2(x: np.ndarray, ref: np.ndarray) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((x - ref).ravel()) / (den if den > 0 else 1.0))


def max_abs(x, ref) -> float:
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64))))


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def sha256(t: torch.Tensor) -> str:
    return hashlib.sha256(t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes()).hexdigest()


def run_gpu(q, k, v, do, scale, causal=True, device="cuda"):
    """Forward + backward through the library; returns CPU tensors."""
    import deterministic_attention_gb300 as da
    qd, kd, vd, dod = (t.to(device) for t in (q, k, v, do))
    o, lse = da.attn_fwd(qd, kd, vd, scale=scale, causal=causal)
    dq, dk, dv = da.attn_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal)
    torch.cuda.synchronize()
    da.check_status()
    return tuple(t.cpu() for t in (o, lse, dq, dk, dv))


def assert_fwd_close(o, lse, o_ref, lse_ref, what=""):
    e = (rel_l2(o, o_ref), max_abs(o, o_ref), rel_l2(lse, lse_ref), max_abs(lse, lse_ref))
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite forward"
    assert e[0] <= TOL_FWD_REL and e[1] <= TOL_FWD_ABS, f"{what}: O rel-L2 {e[0]:.3g} max-abs {e[1]:.3g}"
    assert e[2] <= TOL_FWD_REL and e[3] <= TOL_FWD_ABS, f"{what}: LSE rel-L2 {e[2]:.3g} max-abs {e[3]:.3g}"
    return e


def assert_bwd_close(pairs, what=""):
    out = {}
    for name, x, ref in pairs:
        assert np.all(np.isfinite(x)), f"{what}: non-finite {name}"
        r = rel_l2(x, ref)
        out[name] = r
        assert r <= TOL_BWD_REL, f"{what}: {name} rel-L2 {r:.3g} (max-abs {max_abs(x, ref):.3g})"
    return out
