"""Seeded synthetic attention inputs and the named workloads.

This module holds no attention arithmetic.  It only draws random tensors, so
the CUDA path and the fp64 oracle can be fed the very same bf16 values.

Recipe (the pages measure on synthetic data only: RustingBrain page, "The
setup", trains on synthetic token IDs):
  * ``torch.Generator('cpu').manual_seed(seed)``;
  * draw Q, K, V, dO in that order with ``torch.randn(shape, float32)``;
  * multiply dO by its standard deviation, then round every tensor to bf16
    (round to nearest even);
  * for a peaked workload, draw ``ceil(frac*T)`` positions with
    ``torch.randperm(T)`` after dO and multiply K by 2 there (exact in bf16),
    for every batch and KV head.

"N(0, 1e-2)" in the workload descriptions is read as variance 1e-2, i.e. a
standard deviation of 0.1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    seed: int
    dout_std: float = 1.0
    k_peak_frac: float = 0.0
    scale: float | None = None  # None: 1/sqrt(D)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def shape(self):
        return (self.B, self.T, self.Hq, self.Hkv, self.D)

    def fwd_flops(self) -> float:
        """Algorithmic causal forward FLOPs: 2 matmuls over half the score matrix."""
        return 2.0 * self.B * self.Hq * self.T * self.T * self.D

    def fwd_bwd_flops(self) -> float:
        """Forward plus a 5-matmul backward: 3.5x the forward."""
        return 3.5 * self.fwd_flops()


# The five workloads of the attention hot path.  "page3" is one attention
# layer of the 16-layer d_model 768 GQA model at batch 4 x 1024 tokens
# (RustingBrain page, "The setup" and the 4 x 1024 measurements).
WORKLOADS = {
    "tiny": Workload("tiny_b1_t128_hq2_hkv1_d64", 1, 128, 2, 1, 64, seed=0, scale=0.125),
    "small": Workload("small_b1_t512_hq12_hkv4_d64", 1, 512, 12, 4, 64, seed=1),
    "page3": Workload("page3_b4_t1024_hq12_hkv4_d64", 4, 1024, 12, 4, 64, seed=2, dout_std=0.1),
    "wide": Workload("wide_mha_b32_t1024_h24_d64", 32, 1024, 24, 24, 64, seed=3, dout_std=0.1),
    "long": Workload("long_b1_t8192_hq32_hkv8_d128", 1, 8192, 32, 8, 128, seed=4, dout_std=0.1,
                     k_peak_frac=0.01),
}


def make_inputs(B: int, T: int, Hq: int, Hkv: int, D: int, seed: int, dout_std: float = 1.0,
                k_peak_frac: float = 0.0, q_std: float = 1.0):
    """bf16 CPU tensors q, k, v, dout in the [B, T, H, D] layout."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn((B, T, Hq, D), dtype=torch.float32, generator=g)
    k = torch.randn((B, T, Hkv, D), dtype=torch.float32, generator=g)
    v = torch.randn((B, T, Hkv, D), dtype=torch.float32, generator=g)
    dout = torch.randn((B, T, Hq, D), dtype=torch.float32, generator=g)
    if q_std != 1.0:
        q = q * q_std
    if dout_std != 1.0:
        dout = dout * dout_std
    q, k, v, dout = (t.to(torch.bfloat16) for t in (q, k, v, dout))
    if k_peak_frac > 0.0 and T > 0:
        pos = torch.randperm(T, generator=g)[: math.ceil(k_peak_frac * T)]
        k[:, pos] = k[:, pos] * 2
    return q, k, v, dout


def varlen_lengths(total: int, lo: int, hi: int, seed: int) -> list[int]:
    """Sequence lengths that sum to `total`: each drawn uniformly from
    [lo, hi] with ``torch.randint`` on a generator seeded with `seed`, the
    last one cut to what is left (so it may be shorter than lo)."""
    if not (0 < lo <= hi) or total < 0:
        raise ValueError(f"need 0 < lo <= hi and total >= 0 (lo={lo}, hi={hi}, total={total})")
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    out, left = [], total
    while left > 0:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g))
        out.append(min(n, left))
        left -= out[-1]
    return out


def make_varlen_inputs(tqs, tks, Hq: int, Hkv: int, D: int, seed: int, dout_std: float = 1.0):
    """Packed bf16 CPU tensors q, dout [sum(tqs), Hq, D] and k, v [sum(tks), Hkv, D],
    and the int32 offsets cu_q, cu_k (sequence s: rows cu[s] .. cu[s+1]-1).
    Same draw order as make_inputs, so B sequences of length T give exactly
    make_inputs' values in the packed layout."""
    if len(tqs) != len(tks) or min(list(tqs) + list(tks) + [0]) < 0:
        raise ValueError("tqs and tks must be equally long lists of lengths >= 0")
    cu_q = torch.tensor([0] + list(tqs), dtype=torch.int64).cumsum(0).to(torch.int32)
    cu_k = torch.tensor([0] + list(tks), dtype=torch.int64).cumsum(0).to(torch.int32)
    nq, nk = int(cu_q[-1]), int(cu_k[-1])
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn((nq, Hq, D), dtype=torch.float32, generator=g)
    k = torch.randn((nk, Hkv, D), dtype=torch.float32, generator=g)
    v = torch.randn((nk, Hkv, D), dtype=torch.float32, generator=g)
    dout = torch.randn((nq, Hq, D), dtype=torch.float32, generator=g)
    if dout_std != 1.0:
        dout = dout * dout_std
    q, k, v, dout = (t.to(torch.bfloat16) for t in (q, k, v, dout))
    return q, k, v, dout, cu_q, cu_k


def visible_pairs(tq: int, tk: int, causal: bool) -> int:
    """(query, key) pairs a sequence attends over: every pair, or under the
    bottom-right causal mask (query i sees key j iff j <= i + tk - tq) the sum
    over rows of clamp(i + 1 + tk - tq, 0, tk)."""
    if not causal:
        return tq * tk
    off = tk - tq
    # Rows with i + 1 + off <= 0 see nothing; rows with i + 1 + off >= tk see all.
    lo = max(0, -off)                      # first row that sees a key
    hi = min(tq, max(lo, tk - off - 1))    # first row that sees every key
    partial = sum(range(lo + 1 + off, hi + 1 + off)) if hi > lo else 0
    return partial + (tq - hi) * tk


def varlen_fwd_flops(tqs, tks, Hq: int, D: int, causal: bool) -> float:
    """Algorithmic forward FLOPs of a packed batch: 4 * Hq * D per visible
    pair (Q K^T and P V).  With tq = tk = T causal this is the fixed-length
    2 * Hq * T^2 * D plus its diagonal term 2 * Hq * T * D."""
    return 4.0 * Hq * D * sum(visible_pairs(a, b, causal) for a, b in zip(tqs, tks))


# Packed variable-length workload next to page3 (no page describes one): the
# same 4 x 1024 = 4,096 tokens per step and heads, cut into sequences of
# 64..1,024 tokens (self-attention, Tq = Tk), seed 5, dO sigma 0.1.
VARLEN_PAGE3 = dict(total=4096, lo=64, hi=1024, Hq=12, Hkv=4, D=64, seed=5, dout_std=0.1)


def varlen_page3_inputs():
    w = VARLEN_PAGE3
    tqs = varlen_lengths(w["total"], w["lo"], w["hi"], w["seed"])
    return make_varlen_inputs(tqs, tqs, w["Hq"], w["Hkv"], w["D"], w["seed"], w["dout_std"])


# Embedding-lookup gradient of the trainer the oxide-train README profiles
# ("Full-step profiling": B = 32, T = 1024, a vocabulary of 50,257 padded to
# 50,432, width 1536): N = 32,768 token ids and their gradient rows.
EMBED_GRAD = dict(N=32 * 1024, V=50432, V_used=50257, E=1536, seed=6)


def make_embed_grad_inputs(N: int, V_used: int, E: int, seed: int, dist: str = "uniform",
                           zipf_s: float = 1.1):
    """int32 token ids [N] in [0, V_used) and a bf16 gradient dY [N, E] ~ N(0, 1).

    dist "uniform": ids from ``torch.randint`` (synthetic token IDs, as the
    throughput runs use); "zipf": id r drawn with weight 1 / (r + 1)^zipf_s by
    ``torch.multinomial`` (a natural-text stand-in, where a few ids take most
    tokens and collide often).  Ids are drawn first, then dY."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    if dist == "uniform":
        ids = torch.randint(0, V_used, (N,), generator=g, dtype=torch.int64)
    elif dist == "zipf":
        w = torch.arange(1, V_used + 1, dtype=torch.float64).pow(-zipf_s)
        ids = torch.multinomial(w, N, replacement=True, generator=g)
    else:
        raise ValueError(f"dist must be 'uniform' or 'zipf', not {dist!r}")
    dy = torch.randn((N, E), dtype=torch.float32, generator=g).to(torch.bfloat16)
    return ids.to(torch.int32), dy


# One attention layer of the page-3 model for the training micro-loop
# (RustingBrain page, "The setup": d_model 768, 12 query heads over 4 KV
# heads of head_dim 64, batch 4 x 1024 tokens).
LAYER_PAGE3 = dict(B=4, T=1024, d=768, Hq=12, Hkv=4, D=64, seed=7, w_std=0.02, dy_std=0.1)


def make_layer_inputs(B: int, T: int, d: int, Hq: int, Hkv: int, D: int, seed: int,
                      w_std: float = 0.02, dy_std: float = 0.1):
    """bf16 CPU tensors X [B, T, d], Wq [d, Hq*D], Wk, Wv [d, Hkv*D],
    Wo [Hq*D, d] and dY [B, T, d], drawn in that order with ``torch.randn``:
    X ~ N(0, 1), weights ~ N(0, w_std^2), dY ~ N(0, dy_std^2)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    shapes = [((B, T, d), 1.0), ((d, Hq * D), w_std), ((d, Hkv * D), w_std),
              ((d, Hkv * D), w_std), ((Hq * D, d), w_std), ((B, T, d), dy_std)]
    return tuple((torch.randn(shp, dtype=torch.float32, generator=g) * sd).to(torch.bfloat16)
                 for shp, sd in shapes)


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.T, w.Hq, w.Hkv, w.D, w.seed, w.dout_std, w.k_peak_frac)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 CPU tensor's bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
