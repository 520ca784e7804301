"""fp64 CPU oracle for causal grouped-query attention (forward + closed-form backward).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The attention
library never imports, links or runs it, and the two share no code.

Besides fixed-length batches [B, T, H, D] it covers packed variable-length
batches with Tq != Tk (``attn_fwd_varlen``, ``attn_bwd_varlen``), which no page
describes; the readings (bottom-right causal alignment, rows that see no key)
are stated in ``attn_oracle.h``.  ``embed_grad`` (``embed_oracle.c``) is the
gradient of an embedding lookup summed in ascending token order (oxide-train
README, "The trainer is not bit-identical to itself after step 1").
``oracle.layer`` (numpy around the attention functions here) is one attention
layer of a training step: QKV projection, rotary positions, attention, output
projection, and its closed-form backward.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over
independent heads); this module compiles it with gcc, loads it with ctypes and
marshals numpy arrays.  The only thing done here besides marshalling is the
exact widening of bf16 bit patterns to fp64.

Source of the method: RustingBrain vs PyTorch/TensorFlow page, "Step 1: measure
before changing anything" (causal softmax with a per-row logsumexp, probabilities
recomputed from it), "Step 2: fused flash attention" (forward and backward),
"The setup" (12 query heads over 4 KV heads, head_dim 64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "embed_oracle.c")]
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def compile_library(srcs, out: str) -> str:
    """Compile the oracle's C sources (the files in ``oracle/`` or copies of
    them) into the shared library ``out`` with the flags the oracle is built
    with."""
    srcs = [srcs] if isinstance(srcs, str) else list(srcs)
    # -O2 without -ffast-math: the compiler keeps every sum in source order.
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-I", _HERE, *srcs, "-o", out,
           "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle's C sources into ``_build/liboracle.so`` (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and all(
        os.path.getmtime(_LIB_PATH) >= os.path.getmtime(os.path.join(_HERE, f))
        for f in ("attn_oracle.c", "attn_oracle.h", "embed_oracle.c", "embed_oracle.h"))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    compile_library(_SRCS, tmp)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    """Declare the C signatures on a loaded oracle library and return it.  The
    tests bind copies built with planted mistakes this way, to show that the
    pins catch them."""
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int)
    i, d = ctypes.c_int, ctypes.c_double
    lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, d, i]
    lib.oracle_attn_fwd.restype = None
    lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, d, i]
    lib.oracle_attn_bwd.restype = d
    lib.oracle_attn_probs.argtypes = [dp, dp, dp, i, i, i, i, i, i, i, d, i]
    lib.oracle_attn_probs.restype = None
    lib.oracle_attn_rows.argtypes = [dp, dp, dp, dp, i, ip, ip, ip, dp, dp, dp,
                                     i, i, i, i, i, d, i]
    lib.oracle_attn_rows.restype = None
    lib.oracle_kv_rows.argtypes = [dp, dp, dp, dp, i, i, i, ip, dp, dp, i, i, i, i, i, d, i]
    lib.oracle_kv_rows.restype = None
    lib.oracle_rowdot.argtypes = [dp, dp, dp, i, i, i, i]
    lib.oracle_rowdot.restype = None
    lib.oracle_attn_fwd_varlen.argtypes = [dp, dp, dp, dp, dp, i, ip, ip, i, i, i, d, i]
    lib.oracle_attn_fwd_varlen.restype = None
    lib.oracle_attn_bwd_varlen.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i, ip, ip, i, i, i, d, i]
    lib.oracle_attn_bwd_varlen.restype = d
    lib.oracle_embed_grad.argtypes = [ip, dp, dp, i, i, i]
    lib.oracle_embed_grad.restype = i
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    return lib


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 values given as their uint16 bit patterns."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def _shape(q, k):
    B, T, Hq, D = q.shape
    Bk, Tk, Hkv, Dk = k.shape
    if (B, T, D) != (Bk, Tk, Dk) or Hkv < 1 or Hq % Hkv:
        raise ValueError(f"incompatible q {q.shape} / k {k.shape}")
    return B, T, Hq, Hkv, D


def num_threads() -> int:
    return _load().oracle_num_threads()


def attn_fwd(q, k, v, scale: float, causal: bool = True):
    """O [B,T,Hq,D] and LSE [B,Hq,T] (natural log) in fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, Hq, Hkv, D = _shape(q, k)
    o = np.empty_like(q)
    lse = np.empty((B, Hq, T), dtype=np.float64)
    _load().oracle_attn_fwd(_dp(q), _dp(k), _dp(v), _dp(o), _dp(lse),
                            B, T, Hq, Hkv, D, float(scale), int(bool(causal)))
    return o, lse


def attn_bwd(q, k, v, dout, scale: float, causal: bool = True):
    """dQ, dK, dV, Delta and the worst disagreement between the two forms of Delta."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, T, Hq, Hkv, D = _shape(q, k)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    delta = np.empty((B, Hq, T), dtype=np.float64)
    worst = _load().oracle_attn_bwd(_dp(q), _dp(k), _dp(v), _dp(dout), _dp(dq), _dp(dk), _dp(dv),
                                    _dp(delta), B, T, Hq, Hkv, D, float(scale), int(bool(causal)))
    return dq, dk, dv, delta, worst


def rowdot(o, dout):
    """Delta [B,H,T] = sum_d dout * o for given o, dout [B,T,H,D]."""
    o, dout = _f64(o), _f64(dout)
    B, T, H, D = o.shape
    delta = np.empty((B, H, T), dtype=np.float64)
    _load().oracle_rowdot(_dp(o), _dp(dout), _dp(delta), B, T, H, D)
    return delta


def attn_probs(q, k, b: int, h: int, scale: float, causal: bool = True):
    """Explicit P [T,T] of one (batch, query head)."""
    q, k = _f64(q), _f64(k)
    B, T, Hq, Hkv, D = _shape(q, k)
    p = np.empty((T, T), dtype=np.float64)
    _load().oracle_attn_probs(_dp(q), _dp(k), _dp(p), int(b), int(h), B, T, Hq, Hkv, D,
                              float(scale), int(bool(causal)))
    return p


def attn_rows(q, k, v, dout, rows, scale: float, causal: bool = True, with_dq: bool = True):
    """O, LSE (and dQ) of sampled query rows ``rows`` = [(b, h, i), ...]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    dout = _f64(dout) if dout is not None else np.zeros((1,), dtype=np.float64)
    B, T, Hq, Hkv, D = _shape(q, k)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = r.shape[0]
    rb, rh, ri = (np.ascontiguousarray(r[:, c]) for c in range(3))
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    dq = np.empty((n, D), dtype=np.float64) if with_dq else None
    _load().oracle_attn_rows(_dp(q), _dp(k), _dp(v), _dp(dout), n, _ip(rb), _ip(rh), _ip(ri),
                             _dp(o), _dp(lse), _dp(dq) if with_dq else None,
                             B, T, Hq, Hkv, D, float(scale), int(bool(causal)))
    return (o, lse, dq) if with_dq else (o, lse)


def kv_rows(q, k, v, dout, b: int, g: int, js, scale: float, causal: bool = True):
    """dK, dV of key positions ``js`` of (batch b, KV head g)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, T, Hq, Hkv, D = _shape(q, k)
    j = np.ascontiguousarray(np.asarray(js, dtype=np.int32).reshape(-1))
    dk = np.empty((j.size, D), dtype=np.float64)
    dv = np.empty((j.size, D), dtype=np.float64)
    _load().oracle_kv_rows(_dp(q), _dp(k), _dp(v), _dp(dout), int(b), int(g), j.size, _ip(j),
                           _dp(dk), _dp(dv), B, T, Hq, Hkv, D, float(scale), int(bool(causal)))
    return dk, dv


def _cu(cu, total, what):
    c = np.ascontiguousarray(np.asarray(cu, dtype=np.int64).reshape(-1))
    if c.size < 1 or c[0] != 0 or np.any(np.diff(c) < 0) or c[-1] != total:
        raise ValueError(f"{what} must start at 0, not decrease and end at {total}: {c.tolist()}")
    return np.ascontiguousarray(c.astype(np.int32))


def _varlen_shape(q, k, cu_q, cu_k):
    Nq, Hq, D = q.shape
    Nk, Hkv, Dk = k.shape
    if D != Dk or Hkv < 1 or Hq % Hkv:
        raise ValueError(f"incompatible q {q.shape} / k {k.shape}")
    cq, ck = _cu(cu_q, Nq, "cu_q"), _cu(cu_k, Nk, "cu_k")
    if cq.size != ck.size:
        raise ValueError("cu_q and cu_k must describe the same number of sequences")
    return cq, ck, cq.size - 1, Hq, Hkv, D


def attn_fwd_varlen(q, k, v, cu_q, cu_k, scale: float, causal: bool = True):
    """Packed variable-length forward: q [total_q, Hq, D], k, v [total_k, Hkv,
    D], sequence s in rows cu_q[s]..cu_q[s+1]-1 and cu_k[s]..cu_k[s+1]-1.
    Returns O [total_q, Hq, D] and LSE [Hq, total_q]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cq, ck, n_seq, Hq, Hkv, D = _varlen_shape(q, k, cu_q, cu_k)
    o = np.empty_like(q)
    lse = np.empty((Hq, q.shape[0]), dtype=np.float64)
    _load().oracle_attn_fwd_varlen(_dp(q), _dp(k), _dp(v), _dp(o), _dp(lse), n_seq, _ip(cq),
                                   _ip(ck), Hq, Hkv, D, float(scale), int(bool(causal)))
    return o, lse


def attn_bwd_varlen(q, k, v, dout, cu_q, cu_k, scale: float, causal: bool = True):
    """dQ, dK, dV, Delta [Hq, total_q] and the worst disagreement between the
    two forms of Delta, for a packed variable-length batch."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    cq, ck, n_seq, Hq, Hkv, D = _varlen_shape(q, k, cu_q, cu_k)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    delta = np.empty((Hq, q.shape[0]), dtype=np.float64)
    worst = _load().oracle_attn_bwd_varlen(_dp(q), _dp(k), _dp(v), _dp(dout), _dp(dq), _dp(dk),
                                           _dp(dv), _dp(delta), n_seq, _ip(cq), _ip(ck), Hq, Hkv,
                                           D, float(scale), int(bool(causal)))
    return dq, dk, dv, delta, worst


def embed_grad(ids, dy, V: int):
    """dW [V, E] = sum over t with ids[t] == v of dy[t, :] (ascending t, fp64)
    for ids [N] and dy [N, E]."""
    ids = np.ascontiguousarray(np.asarray(ids).reshape(-1), dtype=np.int32)
    dy = _f64(dy)
    N, E = dy.shape
    if ids.size != N:
        raise ValueError(f"{ids.size} ids for {N} gradient rows")
    dw = np.empty((V, E), dtype=np.float64)
    if _load().oracle_embed_grad(_ip(ids), _dp(dy), _dp(dw), N, int(V), E) != 0:
        raise ValueError(f"ids must lie in [0, {V})")
    return dw
