"""Seeded synthetic inputs for the MoE layer forward.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It draws random numbers and rounds them to the storage dtype; it holds none of
the layer's arithmetic (no routing, no scoring, no expert math).

Workload shapes
---------------
The five named workloads follow the sizes that the pages use as sizing
context (a Mixtral-shaped 8-expert top-2 layer, a fine-grained 256-expert top-8
layer with one shared expert, a Switch-style top-1 layer) plus one tiny fp32
case:

=====================  =====  ====  ===  =====  ==  =====  ========  ========
name                   T      d     N    F      k   F_sh   score     norm
=====================  =====  ====  ===  =====  ==  =====  ========  ========
tiny_fp32              64     128   4    256    2   0      softmax   selected
mixtral_prefill        4096   4096  8    14336  2   0      softmax   selected
mixtral_decode         16     4096  8    14336  2   0      softmax   selected
fine_grained_shared    8192   7168  256  2048   8   2048   sigmoid   selected
switch_top1            65536  2048  128  768    1   0      softmax   none
=====================  =====  ====  ===  =====  ==  =====  ========  ========

Distributions: h ~ N(0, 1); W_r ~ N(0, wr_std); expert weights
~ N(0, 1/sqrt(fan_in)) with fan_in = d for W_gate / W_up and F for W_down
(the second parameter is the standard deviation; ``wd_scale``, 1.0 for the
named workloads, multiplies W_down's). fine_grained_shared adds a
per-expert selection bias with a Zipf(s = 1.1) profile:
bias_i = beta * r_i ** -1.1 with r a seeded random permutation of 1..N and
beta = 4.0, which leaves several experts with no tokens.

Values are drawn in fp32 from one ``torch.Generator`` in the fixed order
h, W_r, W_gate, W_up, W_down, shared W_gate, shared W_up, shared W_down, bias
ranks, then rounded to the workload's dtype. The CPU oracle reads the rounded
values, so both sides see identical inputs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    N: int
    F: int
    k: int
    F_sh: int = 0
    score: str = "softmax"      # "softmax" | "sigmoid"
    norm: str = "selected"      # "selected" | "none"
    dtype: str = "bf16"         # "bf16" | "f32"
    wr_std: float = 0.02
    bias_zipf_s: Optional[float] = None
    bias_beta: float = 4.0
    # multiplier on the standard deviation of W_down (and the shared W_down);
    # the named workloads keep 1.0, small test cases may draw smaller
    # down-projection weights so that their outputs stay of order one
    wd_scale: float = 1.0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", T=64, d=128, N=4, F=256, k=2,
                          dtype="f32", wr_std=0.1),
    "mixtral_prefill": Workload("mixtral_prefill", T=4096, d=4096, N=8,
                                F=14336, k=2),
    "mixtral_decode": Workload("mixtral_decode", T=16, d=4096, N=8,
                               F=14336, k=2),
    "fine_grained_shared": Workload("fine_grained_shared", T=8192, d=7168,
                                    N=256, F=2048, k=8, F_sh=2048,
                                    score="sigmoid", bias_zipf_s=1.1),
    "switch_top1": Workload("switch_top1", T=65536, d=2048, N=128, F=768,
                            k=1, norm="none"),
}


# Reduced cases of the same kernels for profiler captures: weights still
# larger than L2, a few hundred MB of activations. prof_prefill holds 2 of the
# Mixtral-shaped prefill's 8 experts with the same ~1024 rows each, so its
# grouped-GEMM traffic is a quarter of the full batch's.
PROFILE_WORKLOADS = {
    "prof_prefill": Workload("prof_prefill", T=1024, d=4096, N=2, F=14336, k=2),
    "prof_fine_grained": Workload("prof_fine_grained", T=2048, d=7168, N=64, F=2048, k=8,
                                  F_sh=2048, score="sigmoid", bias_zipf_s=1.1),
    "prof_switch": Workload("prof_switch", T=16384, d=2048, N=32, F=768, k=1, norm="none"),
    # the named batches' T, d, N, k, scoring and bias with narrow experts:
    # h and W_r are drawn first, so the routing, dispatch and combine see the
    # same data as the full workloads while the device holds a few hundred MB
    "io_prefill": Workload("io_prefill", T=4096, d=4096, N=8, F=128, k=2),
    "io_fine_grained": Workload("io_fine_grained", T=8192, d=7168, N=256, F=64, k=8, F_sh=64,
                                score="sigmoid", bias_zipf_s=1.1),
    "io_switch": Workload("io_switch", T=65536, d=2048, N=128, F=64, k=1, norm="none"),
}


def _randn(gen: torch.Generator, shape, std: float, dtype: torch.dtype,
           device) -> torch.Tensor:
    """N(0, std) drawn in fp32 on ``device`` then rounded to ``dtype``.

    Large tensors are drawn slab by slab along dim 0 so that the fp32
    temporary stays small.
    """
    out = torch.empty(shape, dtype=dtype, device=device)
    if len(shape) == 0 or shape[0] == 0:
        return out
    per_row = max(1, math.prod(shape[1:]))
    rows = max(1, (1 << 26) // per_row)
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        t = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=gen,
                        dtype=torch.float32, device=device)
        if std != 1.0:
            t.mul_(std)
        out[r0:r1].copy_(t)
    return out


def zipf_bias(gen: torch.Generator, N: int, s: float, beta: float,
              device) -> torch.Tensor:
    """Per-expert selection bias beta * r**-s, r a seeded permutation of 1..N."""
    ranks = torch.randperm(N, generator=gen, device=device).to(torch.float64) + 1.0
    return (beta * ranks.pow(-s)).to(torch.float32)


def make_inputs(w: Workload, seed: int = 0, device="cpu", shared: bool = True):
    """All inputs of one workload, drawn from one seeded generator.

    Returns a dict of tensors on ``device``: h [T,d], W_r [N,d],
    W_gate [N,F,d], W_up [N,F,d], W_down [N,d,F], and when F_sh > 0 and
    ``shared``: Ws_gate [F_sh,d], Ws_up [F_sh,d], Ws_down [d,F_sh]; plus
    sel_bias [N] fp32 when the workload has a bias profile (else None).
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    dt = w.torch_dtype
    out = {}
    out["h"] = _randn(gen, (w.T, w.d), 1.0, dt, dev)
    out["W_r"] = _randn(gen, (w.N, w.d), w.wr_std, dt, dev)
    out["W_gate"] = _randn(gen, (w.N, w.F, w.d), 1.0 / math.sqrt(w.d), dt, dev)
    out["W_up"] = _randn(gen, (w.N, w.F, w.d), 1.0 / math.sqrt(w.d), dt, dev)
    out["W_down"] = _randn(gen, (w.N, w.d, w.F), w.wd_scale / math.sqrt(w.F), dt, dev)
    if w.F_sh > 0 and shared:
        out["Ws_gate"] = _randn(gen, (w.F_sh, w.d), 1.0 / math.sqrt(w.d), dt, dev)
        out["Ws_up"] = _randn(gen, (w.F_sh, w.d), 1.0 / math.sqrt(w.d), dt, dev)
        out["Ws_down"] = _randn(gen, (w.d, w.F_sh), w.wd_scale / math.sqrt(w.F_sh), dt, dev)
    else:
        out["Ws_gate"] = out["Ws_up"] = out["Ws_down"] = None
    if w.bias_zipf_s is not None:
        out["sel_bias"] = zipf_bias(gen, w.N, w.bias_zipf_s, w.bias_beta, dev)
    else:
        out["sel_bias"] = None
    return out


def random_logits(T: int, N: int, seed: int = 0, std: float = 1.0,
                  ties: bool = False) -> torch.Tensor:
    """fp32 logits [T,N] for route-from-logits cases.

    With ``ties`` the values are drawn from a coarse grid so that many rows
    hold exact ties, which exercises the lowest-index tie-break.
    """
    gen = torch.Generator().manual_seed(seed)
    z = torch.randn((T, N), generator=gen, dtype=torch.float32) * std
    if ties:
        z = torch.round(z * 2.0) / 2.0
    return z


def to_f64(t: Optional[torch.Tensor]):
    """The exact values of a (possibly bf16) tensor as a float64 numpy array."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()
