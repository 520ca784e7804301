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


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.T, w.Hq, w.Hkv, w.D, w.seed, w.dout_std, w.k_peak_frac)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 CPU tensor's bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
