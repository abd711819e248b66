"""Routing selection on crafted logits: exact ties and keys one fp32 ulp apart.

Token t is the one-hot row e_t, so its router logits are exactly column t of
W_r (every other product is zero), and the test chooses every logit. The
sigmoid router's selection keys are fp64 (sigmoid(l) + b); logits one fp32 ulp
apart give fp64 keys about 1e-8 apart, which fp32 arithmetic cannot order, so
these rows check that the kernel's fp64 decisions match the oracle's exactly.
Exact ties must go to the lower expert index (and to the lower group).
"""
import numpy as np
import pytest
import torch

import routing_dispatch_expert_router_gb300.binding as B
from oracle import moe_oracle as O
from workloads import GROUP_MAX, SIGMOID, MoEShape

import harness as H_

pytestmark = pytest.mark.gpu


def crafted_logits(T, E, rng, per_group=None):
    """[T, E] fp32 logits full of near-ties and exact ties."""
    L = np.empty((T, E), np.float32)
    for t in range(T):
        base = rng.standard_normal(E).astype(np.float32)
        mode = t % 4
        if mode == 0:          # runs of neighbours one ulp apart
            v = np.float32(rng.standard_normal())
            for e in rng.permutation(E)[: E // 2]:
                base[e] = v
                v = np.nextafter(v, np.float32(np.inf))
        elif mode == 1:        # many exact ties
            base[rng.permutation(E)[: E // 2]] = np.float32(0.75)
        elif mode == 2 and per_group:
            # every group's two best logits are the same two values: all group
            # scores tie (without bias) and the lower groups must win
            base = np.minimum(base, np.float32(1.9))
            hi, lo = np.float32(2.0), np.nextafter(np.float32(2.0), np.float32(0))
            for g in range(E // per_group):
                e1, e2 = rng.choice(per_group, size=2, replace=False) + g * per_group
                base[e1], base[e2] = hi, lo
        L[t] = base
    return L


def route_on(shape, logits, bias):
    """Runs moe_route on one-hot tokens whose logits are `logits` exactly."""
    T, E = logits.shape
    H = shape.H
    assert T <= H
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    x[torch.arange(T), torch.arange(T)] = 1.0
    W_r = torch.zeros(E, H, dtype=torch.float32)
    W_r[:, :T] = torch.from_numpy(logits.T.copy())
    cfg = B.config(shape)
    sz = B.moe_query_sizes(cfg)
    dev = "cuda"
    sc = torch.zeros(sz.scratch_bytes, dtype=torch.uint8, device=dev)
    lg = torch.empty(T, E, dtype=torch.float32, device=dev)
    idx = torch.empty(T, shape.k, dtype=torch.int32, device=dev)
    w = torch.empty(T, shape.k, dtype=torch.float32, device=dev)
    b = None if bias is None else torch.from_numpy(bias).to(dev)
    B.moe_route(cfg, x.to(dev), W_r.to(dev), b, lg, idx, w, sc)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(sc) == 0
    return H_.f64(lg), H_.i64(idx), H_.f64(w)


CASES = [
    # (name, shape, bias kind)
    ("sigmoid_groups_e256", MoEShape("t", T=128, H=128, E=256, k=8, F=128, score_fn=SIGMOID,
                                     n_groups=8, topk_groups=4), "normal"),
    ("sigmoid_groups_e256_nobias", MoEShape("t", T=128, H=128, E=256, k=8, F=128,
                                            score_fn=SIGMOID, n_groups=8, topk_groups=4), None),
    ("sigmoid_groupmax_e64", MoEShape("t", T=128, H=128, E=64, k=6, F=128, score_fn=SIGMOID,
                                      n_groups=8, topk_groups=3, group_score=GROUP_MAX),
     "normal"),
    ("sigmoid_flat_e16", MoEShape("t", T=128, H=128, E=16, k=4, F=128, score_fn=SIGMOID), None),
    ("softmax_e128", MoEShape("t", T=128, H=128, E=128, k=8, F=128), None),
    ("softmax_groups_e32", MoEShape("t", T=128, H=128, E=32, k=4, F=128, n_groups=4,
                                    topk_groups=2), "normal"),
    ("softmax_e8", MoEShape("t", T=128, H=128, E=8, k=2, F=128), None),
]


@pytest.mark.parametrize("name,shape,bias_kind", CASES, ids=[c[0] for c in CASES])
def test_selection_on_ties_matches_oracle(name, shape, bias_kind):
    rng = np.random.default_rng(7)
    per = shape.E // shape.n_groups if shape.n_groups > 1 else None
    L = crafted_logits(shape.T, shape.E, rng, per)
    bias = None
    if bias_kind == "normal":
        bias = (0.05 * rng.standard_normal(shape.E)).astype(np.float32)
        # a few exact bias ties too
        bias[: shape.E // 4] = bias[0]
    lg, idx, w = route_on(shape, L, bias)
    H_.assert_equal("logits", lg, L.astype(np.float64))
    idx_ref, w_ref = O.route(lg, shape, bias)
    H_.assert_equal("idx", idx, idx_ref)
    H_.assert_close("w", w, w_ref, atol=1e-6, rtol=1e-5)
