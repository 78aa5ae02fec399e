"""Seeded synthetic inputs for the MoE layer.

This module only draws inputs; it holds none of the layer's arithmetic. The
GPU path and the CPU oracle both consume exactly these host arrays.

Recipe (one CPU ``torch.Generator`` seeded with ``seed``; draws in this
order):
  W_r [H, E] fp32 ~ N(0, 0.02)
  W_gate [E, H, I], W_up [E, H, I], W_down [E, I, H] ~ N(0, 0.02), drawn in
      fp32 expert by expert and rounded to BF16 (round to nearest even)
  shared expert (optional) W_sg [H, Is], W_su [H, Is], W_sd [Is, H] likewise
  x [T, H] ~ N(0, 1) rounded to BF16, from a generator seeded
      ``seed + batch + SHARD_STRIDE * shard``
  dY [T, H] ~ N(0, 1) rounded to BF16, from a generator seeded
      ``seed + 1000 + SHARD_STRIDE * shard``
Data-parallel shards (one per rank) share every weight and draw their own
tokens; shard 0 is the single-GPU input.
Skewed routing uses a per-expert logit bias b_e = ln(p_e) with p a Zipf law
of exponent s over the E experts: p_e = (e+1)^-s / sum_n n^-s.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """Shape and input recipe of one layer invocation."""
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    dtype: str = "bf16"          # routed-expert operand type: "bf16" or "mxfp8"
    zipf_s: float = 0.0          # 0 = no bias (uniform routing)
    shared_I: int = 0            # 0 = no shared expert
    batches: int = 1             # macro-batches (independent x per batch)
    ring_rows: int = 0           # 0 = ring holds every routed row of a batch
    backward: bool = False

    @property
    def R(self) -> int:
        return self.T * self.k

    def fwd_flops(self) -> float:
        f = 6.0 * self.H * self.I * self.T * self.k
        if self.shared_I:
            f += 6.0 * self.H * self.shared_I * self.T
        return f * self.batches

    def bwd_flops(self) -> float:
        return 12.0 * self.H * self.I * self.T * self.k


# Named workloads: the layer shapes the pages discuss (H=7168, I=2048, as in
# the Kimi-2.5-shaped experts of the KuCoin article, section 02) plus a tiny
# case the oracle finishes in seconds.
WORKLOADS = {
    "tiny_bf16": Workload("tiny_bf16", T=64, H=128, I=64, E=8, k=2),
    "bf16_fwd_T2560": Workload("bf16_fwd_T2560", T=2560, H=7168, I=2048, E=32, k=8),
    **{f"mxfp8_zipf_T{T}": Workload(f"mxfp8_zipf_T{T}", T=T, H=7168, I=2048, E=32, k=8,
                                    dtype="mxfp8", zipf_s=1.2)
       for T in (512, 1024, 2560, 4096, 8192)},
    "ring_stream_16x4096": Workload("ring_stream_16x4096", T=4096, H=7168, I=2048, E=32, k=8,
                                    dtype="mxfp8", zipf_s=1.2, shared_I=2048, batches=16,
                                    ring_rows=16384),
    "bf16_bwd_T4096": Workload("bf16_bwd_T4096", T=4096, H=7168, I=2048, E=32, k=8,
                               backward=True),
    # the same training step with MXFP8 routed experts (forward and backward)
    "mxfp8_bwd_T4096": Workload("mxfp8_bwd_T4096", T=4096, H=7168, I=2048, E=32, k=8, dtype="mxfp8",
                                backward=True),
    # profiling case: the same expert shape with 8 experts (about 1 GB of
    # weights, still well above the 129 MB L2) for counter captures
    "bf16_fwd_E8_T2560": Workload("bf16_fwd_E8_T2560", T=2560, H=7168, I=2048, E=8, k=2),
    # 1024 rows per expert as at T=4096 with 32 experts
    "bf16_fwd_E8_T4096": Workload("bf16_fwd_E8_T4096", T=4096, H=7168, I=2048, E=8, k=2),
    "mxfp8_fwd_E8_T2560": Workload("mxfp8_fwd_E8_T2560", T=2560, H=7168, I=2048, E=8, k=2, dtype="mxfp8"),
    # backward profiling case: 1024 rows per expert, as in the 32-expert T=4096 backward
    "bf16_bwd_E8_T4096": Workload("bf16_bwd_E8_T4096", T=4096, H=7168, I=2048, E=8, k=2, backward=True),
    "mxfp8_bwd_E8_T4096": Workload("mxfp8_bwd_E8_T4096", T=4096, H=7168, I=2048, E=8, k=2, dtype="mxfp8",
                                   backward=True),
}


def zipf_bias(E: int, s: float) -> np.ndarray:
    """ln of a Zipf(s) distribution over E experts, computed in fp64, as fp32."""
    z = np.array([(n + 1) ** (-s) for n in range(E)], dtype=np.float64)
    return np.log(z / z.sum()).astype(np.float32)


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _normal_bf16(g: torch.Generator, shape, std: float) -> np.ndarray:
    return _bf16_bits(torch.randn(shape, generator=g, dtype=torch.float32) * std)


@dataclass
class LayerInputs:
    """Host arrays of one workload. BF16 tensors are uint16 bit patterns."""
    wl: Workload
    W_r: np.ndarray
    bias: np.ndarray | None
    Wg: np.ndarray
    Wu: np.ndarray
    Wd: np.ndarray
    shared: tuple | None
    xs: list = field(default_factory=list)
    dY: np.ndarray | None = None

    @property
    def x(self) -> np.ndarray:
        return self.xs[0]


SHARD_STRIDE = 100_003


def make_x(wl: Workload, batch: int = 0, seed: int = 0, shard: int = 0) -> np.ndarray:
    g = torch.Generator().manual_seed(seed + batch + SHARD_STRIDE * shard)
    return _normal_bf16(g, (wl.T, wl.H), 1.0)


def make_inputs(wl: Workload, seed: int = 0, with_x: bool = True, shard: int = 0) -> LayerInputs:
    g = torch.Generator().manual_seed(seed)
    W_r = (torch.randn((wl.H, wl.E), generator=g, dtype=torch.float32) * 0.02).numpy()
    Wg = np.empty((wl.E, wl.H, wl.I), np.uint16)
    Wu = np.empty((wl.E, wl.H, wl.I), np.uint16)
    Wd = np.empty((wl.E, wl.I, wl.H), np.uint16)
    for dst in (Wg, Wu, Wd):
        for e in range(wl.E):
            dst[e] = _normal_bf16(g, dst.shape[1:], 0.02)
    shared = None
    if wl.shared_I:
        shared = (_normal_bf16(g, (wl.H, wl.shared_I), 0.02),
                  _normal_bf16(g, (wl.H, wl.shared_I), 0.02),
                  _normal_bf16(g, (wl.shared_I, wl.H), 0.02))
    bias = zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None
    inp = LayerInputs(wl, W_r, bias, Wg, Wu, Wd, shared)
    if with_x:
        inp.xs = [make_x(wl, b, seed, shard) for b in range(wl.batches)]
    if wl.backward:
        inp.dY = make_dY(wl, seed, shard)
    return inp


def make_dY(wl: Workload, seed: int = 0, shard: int = 0) -> np.ndarray:
    """Upstream gradient dY [T, H] ~ N(0, 1) rounded to BF16."""
    gd = torch.Generator().manual_seed(seed + 1000 + SHARD_STRIDE * shard)
    return _normal_bf16(gd, (wl.T, wl.H), 1.0)


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to fp32 values (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def small(name: str, **kw) -> Workload:
    """A custom workload (used by tests for shapes between the named ones)."""
    return Workload(name=name, **kw)
