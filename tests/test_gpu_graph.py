"""The layer step captured in a CUDA graph and replayed.

moe_layer_fwd and moe_layer_bwd never synchronise with the host (token counts
stay on the device), so one forward + backward can be recorded into a CUDA
graph once and replayed; the replay must give the same bits as the eager
calls (the kernels are deterministic). Two shapes: single-CTA GEMM tiles
(few rows per expert) and CTA-pair tiles (>= 512 rows per expert).
"""
import pytest
import torch

import routing_dispatch_expert_router_gb300.binding as B
from workloads import TINY, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

SHAPES = [TINY, MoEShape("pairs", T=2100, H=512, E=4, k=2, F=512, n_shared=1)]


def _step(cfg, P, d, bufs, outs, stream):
    B.moe_layer_fwd(cfg, P, d["x"], outs["out"], bufs.fwd_struct, bufs.scratch, stream=stream)
    B.moe_layer_bwd(cfg, P, d["x"], d["dY"], bufs.fwd_struct, bufs.bwd_struct, outs["dx"],
                    outs["dW_r"], outs["dW13"], outs["dW2"], bufs.scratch, stream=stream)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_layer_step_replays_from_a_cuda_graph(shape):
    d = make_inputs(shape, seed=5, device="cuda")
    cfg = B.config(shape)
    bufs = B.alloc_buffers(cfg, "cuda")
    T, H, E, F, G = shape.T, shape.H, shape.E, shape.F, shape.E + shape.n_shared
    P = B.params(d["W_r"], d["bias"], d["W13"], d["W2"])
    outs = {"out": torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
            "dx": torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
            "dW_r": torch.empty(E, H, dtype=torch.float32, device="cuda"),
            "dW13": torch.empty(G, 2 * F, H, dtype=torch.bfloat16, device="cuda"),
            "dW2": torch.empty(G, H, F, dtype=torch.bfloat16, device="cuda")}
    # eager reference (also the first call of every kernel: attributes set here)
    _step(cfg, P, d, bufs, outs, None)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(bufs.scratch) == 0
    ref = {k: v.clone() for k, v in outs.items()}
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _step(cfg, P, d, bufs, outs, s)           # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        _step(cfg, P, d, bufs, outs, s)
    for _ in range(2):
        for v in outs.values():
            v.view(torch.uint8).fill_(0xFF)
        g.replay()
        torch.cuda.synchronize()
        assert B.moe_last_device_status(bufs.scratch) == 0
        for k in outs:
            assert torch.equal(outs[k], ref[k]), k


def test_layer_step_with_the_balance_loss_replays_from_a_cuda_graph():
    """Forward + load-balancing loss (with the bias update) + backward + the
    loss's backward, recorded once and replayed: the same bits as eager (the
    aux kernels keep their arrival counter at zero between launches)."""
    shape = MoEShape("aux_e128", T=700, H=256, E=128, k=4, F=128, bias_kind="zipf")
    d = make_inputs(shape, seed=9, device="cuda")
    cfg = B.config(shape)
    bufs = B.alloc_buffers(cfg, "cuda")
    T, H, E, F = shape.T, shape.H, shape.E, shape.F
    P = B.params(d["W_r"], d["bias"], d["W13"], d["W2"])
    lg, idx = bufs.fwd["logits"], bufs.fwd["idx"]
    outs = {"out": torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
            "dx": torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
            "dW_r": torch.empty(E, H, dtype=torch.float32, device="cuda"),
            "dW13": torch.empty(E, 2 * F, H, dtype=torch.bfloat16, device="cuda"),
            "dW2": torch.empty(E, H, F, dtype=torch.bfloat16, device="cuda"),
            "cnt": torch.empty(E, dtype=torch.int32, device="cuda"),
            "P": torch.empty(E, dtype=torch.float32, device="cuda"),
            "loss": torch.empty(1, dtype=torch.float32, device="cuda"),
            "bias_out": torch.empty(E, dtype=torch.float32, device="cuda"),
            "dl_aux": torch.empty(T, E, dtype=torch.float32, device="cuda")}

    def step(stream):
        _step(cfg, P, d, bufs, outs, stream)
        B.moe_route_aux(cfg, lg, d["bias"], idx, 0.01, 1e-3, outs["cnt"], outs["P"],
                        outs["loss"], outs["bias_out"], bufs.scratch, stream=stream)
        B.moe_route_aux_bwd(cfg, d["x"], lg, d["bias"], d["W_r"], outs["cnt"], 0.01, 1.0,
                            outs["dl_aux"], outs["dx"], outs["dW_r"], bufs.scratch, stream=stream)

    step(None)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(bufs.scratch) == 0
    ref = {k: v.clone() for k, v in outs.items()}
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for _ in range(2):
        for v in outs.values():
            v.view(torch.uint8).fill_(0xFF)
        g.replay()
        torch.cuda.synchronize()
        assert B.moe_last_device_status(bufs.scratch) == 0
        for k in outs:
            assert torch.equal(outs[k], ref[k]), k
