"""Fine-grained recompute of the activation function (recompute_h).

"Scalable Training of Mixture-of-Experts Models with Megatron Core" (es
summary, Resumen técnico §2.3.A) lists recomputing activation functions among
the memory optimisations. With recompute_h = 1 the backward rewrites the SwiGLU
output h from the stored G and U in the FC2 data-gradient epilogue, so the h the
forward wrote need not survive until the backward. These tests run the forward,
overwrite h with 0xFF bytes, run the backward with recompute_h = 1, and check
that h comes back bit for bit as the forward wrote it and that every gradient
equals, bit for bit, the run that keeps h (the same kernels in the same order;
the recompute uses the forward epilogue's arithmetic on the stored bf16 G, U).
Paths: bf16 single-CTA tiles, bf16 CTA pairs (the SwiGLU-backward ring), the
routing weight inside the expert (h_s = w silu(G) U), FP8 block and MXFP8.
"""
import numpy as np
import pytest
import torch

import routing_dispatch_expert_router_gb300.binding as B
from oracle import moe_oracle as O
from workloads import DT_FP8, DT_MXFP8, SIGMOID, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

H_ = pytest.importorskip("harness")

SHAPES = [
    MoEShape("rc_single", T=256, H=128, E=8, k=2, F=256),
    # 512 rows per expert, F a multiple of 256: CTA-pair tiles with the GU ring
    MoEShape("rc_pairs", T=1024, H=256, E=2, k=1, F=512),
    MoEShape("rc_inside", T=256, H=128, E=8, k=2, F=256, weights_in_expert=1),
    MoEShape("rc_inside_pairs", T=1024, H=256, E=2, k=1, F=512, weights_in_expert=1),
    MoEShape("rc_fp8", T=512, H=256, E=16, k=4, F=256, score_fn=SIGMOID, n_groups=4,
             topk_groups=2, bias_kind="normal", dtype=DT_FP8),
    MoEShape("rc_mxfp8", T=512, H=256, E=16, k=4, F=256, score_fn=SIGMOID, n_groups=4,
             topk_groups=2, bias_kind="normal", dtype=DT_MXFP8),
]


def _run(shape, inp, poison_h: bool):
    dev = "cuda"
    cfg = B.config(shape)
    bufs = B.alloc_buffers(cfg, dev)
    for t in list(bufs.fwd.values()) + list(bufs.bwd.values()):
        t.view(torch.uint8).fill_(0xFF)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    T, H, E, F = shape.T, shape.H, shape.E, shape.F
    G = E + shape.n_shared
    P = B.params(d["W_r"], d["bias"], d["W13"], d["W2"])
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    B.moe_layer_fwd(cfg, P, d["x"], out, bufs.fwd_struct, bufs.scratch)
    h_fwd = bufs.fwd["h"].clone()
    if poison_h:
        bufs.fwd["h"].view(torch.uint8).fill_(0xFF)
    dx = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    dW_r = torch.empty(E, H, dtype=torch.float32, device=dev)
    dW13 = torch.empty(G, 2 * F, H, dtype=torch.bfloat16, device=dev)
    dW2 = torch.empty(G, H, F, dtype=torch.bfloat16, device=dev)
    B.moe_layer_bwd(cfg, P, d["x"], d["dY"], bufs.fwd_struct, bufs.bwd_struct, dx, dW_r, dW13,
                    dW2, bufs.scratch)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(bufs.scratch) == 0
    return {"out": out, "h_fwd": h_fwd, "h_bwd": bufs.fwd["h"].clone(), "dx": dx, "dW_r": dW_r,
            "dW13": dW13, "dW2": dW2, "idx": bufs.fwd["idx"].clone(),
            "counts": bufs.fwd["counts"].clone(), "offsets": bufs.fwd["offsets"].clone()}


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_recompute_h_is_bit_identical(shape):
    inp = make_inputs(shape, seed=3)
    keep = _run(shape, inp, poison_h=False)
    rec = _run(shape.with_(recompute_h=1), inp, poison_h=True)
    m = O.permutation_maps(keep["idx"].cpu().numpy().astype(np.int64), shape)
    live = torch.as_tensor(H_.read_rows(m), device="cuda")
    R = int(m["R"])
    # h rewritten on every row a GEMM reads, equal to the forward's
    assert torch.equal(rec["h_bwd"][:R][live].view(torch.int16),
                       keep["h_fwd"][:R][live].view(torch.int16))
    for n in ("out", "dx", "dW_r", "dW13", "dW2"):
        a, b = keep[n], rec[n]
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), n
