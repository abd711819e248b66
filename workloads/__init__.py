"""Synthetic MoE-layer workloads: the layer shapes and their seeded inputs.

This module holds no MoE arithmetic. It defines the five layer shapes that the
library is measured and checked on, plus the recipe that draws their inputs
from a seeded ``torch.Generator``. Both the CPU oracle tests and the CUDA path
take their inputs from here, so they see the same tensors.

Shapes (all bf16 activations/weights, fp32 router):

  tiny     T=256   H=128  E=8        k=2 F=256   softmax top-2, renormalised
  mixtral  T=4096  H=4096 E=8        k=2 F=14336 softmax top-2
  dsv3     T=8192  H=7168 E=256(+1)  k=8 F=2048  sigmoid + bias, 8 groups keep 4
  qwen3    T=16384 H=4096 E=128      k=8 F=1536  softmax + Zipf(1.2) logit bias
  dsv3_fp8 T=16384 H=7168 E=256      k=8 F=2048  as dsv3, FP8 E4M3 blocks,
                                                 capacity factor 1.25

Input recipe (per shape): x ~ N(0,1) rounded to bf16; router weight W_r ~
N(0, router_std^2) in fp32; expert weights W13 [E+S, 2F, H] (gate rows then up
rows) and W2 [E+S, H, F] ~ N(0, 0.02^2) rounded to bf16; upstream gradient dY
~ N(0,1) rounded to bf16. Router bias: none (tiny, mixtral); 0.05*N(0,1) per
expert (dsv3, dsv3_fp8); for qwen3 a Zipf(s=1.2) logit bias
b_e = alpha * (-1.2 * ln r_e), r_e a seeded permutation of the ranks 1..E, with
alpha fixed so that the hottest expert receives about ten times the mean load
(``ZIPF_ALPHA``, written by ``workloads/calibrate_zipf.py``).
"""
from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass, replace

import torch

SOFTMAX = 0
SIGMOID = 1
GROUP_TOP2_SUM = 0
GROUP_MAX = 1
DT_BF16 = 0
DT_FP8 = 1
DT_MXFP8 = 2
FP8_DTYPES = (DT_FP8, DT_MXFP8)

_HERE = os.path.dirname(os.path.abspath(__file__))


def _load_zipf_alpha() -> float:
    path = os.path.join(_HERE, "zipf_alpha.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["alpha"])
    return 1.0


ZIPF_ALPHA = _load_zipf_alpha()


@dataclass(frozen=True)
class MoEShape:
    """One MoE layer configuration plus its input recipe."""
    name: str
    T: int
    H: int
    E: int
    k: int
    F: int
    n_shared: int = 0
    score_fn: int = SOFTMAX
    n_groups: int = 1
    topk_groups: int = 1
    group_score: int = GROUP_TOP2_SUM
    route_scale: float = 1.0
    dtype: int = DT_BF16
    capacity_factor: float = 0.0     # 0 = dropless
    row_align: int = 128             # per-expert segment alignment in rows
    weights_in_expert: int = 0       # 1: routing weight applied inside the expert (bf16)
    recompute_h: int = 0             # 1: the backward rewrites h from GU
    # input recipe
    router_std: float = 0.0          # 0 -> 1/sqrt(H)
    weight_std: float = 0.02
    bias_kind: str = "none"          # none | normal | zipf
    bias_scale: float = 0.05

    @property
    def A(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "MoEShape":
        return replace(self, **kw)


TINY = MoEShape("tiny", T=256, H=128, E=8, k=2, F=256)
MIXTRAL = MoEShape("mixtral", T=4096, H=4096, E=8, k=2, F=14336, router_std=0.02)
DSV3 = MoEShape("dsv3", T=8192, H=7168, E=256, k=8, F=2048, n_shared=1,
                score_fn=SIGMOID, n_groups=8, topk_groups=4, bias_kind="normal")
QWEN3 = MoEShape("qwen3", T=16384, H=4096, E=128, k=8, F=1536, bias_kind="zipf")
DSV3_FP8 = MoEShape("dsv3_fp8", T=16384, H=7168, E=256, k=8, F=2048,
                    score_fn=SIGMOID, n_groups=8, topk_groups=4, bias_kind="normal",
                    dtype=DT_FP8, capacity_factor=1.25)

SHAPES = {s.name: s for s in (TINY, MIXTRAL, DSV3, QWEN3, DSV3_FP8)}

# Small cases of the same kernels for detailed profiles (a few GB on the device,
# operands still larger than L2): Mixtral-sized experts, 2 of them with 2048
# rows each (CTA-pair GEMM tiles, K = 4096); DeepSeek-V3-sized experts, 16 of
# them with about 256 rows each (single-CTA tiles, short weight-gradient K);
# the FP8 layer's experts, 16 of them (the FP8 GEMMs at a few GB).
PROFILE_SHAPES = {
    "mixtral_2experts": MIXTRAL.with_(name="mixtral_2experts", T=2048, E=2),
    "dsv3_16experts": DSV3.with_(name="dsv3_16experts", T=512, E=16),
    # the FP8 layer's experts (capacity 640 rows, about 380 kept on average), 16 of them
    "dsv3_fp8_16experts": DSV3_FP8.with_(name="dsv3_fp8_16experts", T=1024, E=16),
    # Mixtral-shaped experts (1024 rows each, F = 14336) in the FP8 block recipe
    "mixtral_fp8": MIXTRAL.with_(name="mixtral_fp8", dtype=DT_FP8),
    # the same layer in the MXFP8 recipe (32-element blocks), full size and 16 experts
    "dsv3_mxfp8": DSV3_FP8.with_(name="dsv3_mxfp8", dtype=DT_MXFP8),
    "dsv3_mxfp8_16experts": DSV3_FP8.with_(name="dsv3_mxfp8_16experts", T=1024, E=16,
                                           dtype=DT_MXFP8),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, std, g, device, chunk_dim0: bool = False) -> torch.Tensor:
    """N(0, std^2) rounded to bf16; drawn slab by slab along dim 0 when asked."""
    if not chunk_dim0:
        return (torch.randn(*shape, generator=g, device=device) * std).to(torch.bfloat16)
    out = torch.empty(*shape, dtype=torch.bfloat16, device=device)
    for i in range(shape[0]):
        out[i] = (torch.randn(*shape[1:], generator=g, device=device) * std).to(torch.bfloat16)
    return out


def router_bias(shape: MoEShape, seed: int) -> torch.Tensor | None:
    """Per-expert router bias [E] fp32 on the CPU (None when the shape has none)."""
    g = _gen("cpu", seed + 7919)
    if shape.bias_kind == "none":
        return None
    if shape.bias_kind == "normal":
        return torch.randn(shape.E, generator=g) * shape.bias_scale
    if shape.bias_kind == "zipf":
        ranks = torch.randperm(shape.E, generator=g).to(torch.float64) + 1.0
        return (ZIPF_ALPHA * (-1.2) * torch.log(ranks)).to(torch.float32)
    raise ValueError(shape.bias_kind)


def make_inputs(shape: MoEShape, seed: int = 0, device: str = "cpu",
                weights: bool = True, grad: bool = True) -> dict:
    """Draw every input of one layer step from a seeded generator on ``device``.

    Returns a dict with x [T,H] bf16, W_r [E,H] f32, bias [E] f32 or None,
    W13 [E+S,2F,H] bf16, W2 [E+S,H,F] bf16 and dY [T,H] bf16.
    """
    g = _gen(device, seed)
    T, H, E, F, S = shape.T, shape.H, shape.E, shape.F, shape.n_shared
    rstd = shape.router_std if shape.router_std > 0 else 1.0 / math.sqrt(H)
    out = {}
    out["x"] = torch.randn(T, H, generator=g, device=device).to(torch.bfloat16)
    out["W_r"] = (torch.randn(E, H, generator=g, device=device) * rstd).contiguous()
    b = router_bias(shape, seed)
    out["bias"] = None if b is None else b.to(device)
    if weights:
        big = (E + S) * 2 * F * H > (1 << 26)
        out["W13"] = _randn_bf16((E + S, 2 * F, H), shape.weight_std, g, device, big)
        out["W2"] = _randn_bf16((E + S, H, F), shape.weight_std, g, device, big)
    if grad:
        out["dY"] = torch.randn(T, H, generator=g, device=device).to(torch.bfloat16)
    return out
