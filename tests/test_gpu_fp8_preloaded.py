"""E4M3 expert weights quantised by the caller (moe_load_fp8_weights).

A caller that keeps its expert weights in E4M3 with one UE8M0 scale per 128x128
tile hands them to the library instead of the bf16 weights; the layer then
runs with params.W13 = params.W2 = NULL. The codes and scales here are the
oracle's tile quantisation of the bf16 weights (oracle.e4m3_scale,
oracle.round_e4m3), so the layer must give the same bits as the layer that
quantises the same bf16 weights itself (moe_quantize_weights inside
moe_layer_fwd), whose results the FP8 parity tests check against the oracle.
"""
import numpy as np
import pytest
import torch

import routing_dispatch_expert_router_gb300.binding as B
from oracle import moe_oracle as O
from workloads import DT_FP8, SIGMOID, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

SHAPES = [
    MoEShape("pre_fp8", T=1024, H=768, E=8, k=2, F=256, score_fn=SIGMOID, capacity_factor=0.5,
             bias_kind="normal", dtype=DT_FP8),
    MoEShape("pre_fp8_groups", T=512, H=256, E=16, k=4, F=256, score_fn=SIGMOID, n_groups=4,
             topk_groups=2, bias_kind="normal", dtype=DT_FP8),
]

OUTS = ("out", "dx", "dW_r", "dW13", "dW2")


def tile_e4m3(W: torch.Tensor):
    """E4M3 codes [G, rows, cols] (uint8) and UE8M0 tile codes [G, rows/128, cols/128]."""
    Wn = W.to(torch.float64).cpu().numpy()
    G, r, c = Wn.shape
    Wb = Wn.reshape(G, r // 128, 128, c // 128, 128)
    s = O.e4m3_scale(np.abs(Wb).max(axis=(2, 4), keepdims=True))
    vals = O.round_e4m3(Wb / s).reshape(G, r, c)
    codes = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8)
    exps = np.log2(s.reshape(G, r // 128, c // 128)).astype(np.int64) + 127
    assert (exps >= 0).all() and (exps <= 254).all()
    return codes.contiguous().cuda(), torch.from_numpy(exps.astype(np.uint8)).contiguous().cuda()


def run(shape, d, cfg, bufs, W13, W2):
    T, H, E, F = shape.T, shape.H, shape.E, shape.F
    e = lambda *s, dt=torch.bfloat16: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    o = {"out": e(T, H), "dx": e(T, H), "dW_r": e(E, H, dt=torch.float32),
         "dW13": e(E, 2 * F, H), "dW2": e(E, H, F)}
    P = B.params(d["W_r"], d["bias"], W13, W2)
    B.moe_layer_fwd(cfg, P, d["x"], o["out"], bufs.fwd_struct, bufs.scratch)
    B.moe_layer_bwd(cfg, P, d["x"], d["dY"], bufs.fwd_struct, bufs.bwd_struct, o["dx"],
                    o["dW_r"], o["dW13"], o["dW2"], bufs.scratch)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(bufs.scratch) == 0
    return o


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_caller_quantised_weights_give_the_same_layer(shape):
    d = make_inputs(shape, seed=0, device="cuda")
    cfg = B.config(shape)
    ref = run(shape, d, cfg, B.alloc_buffers(cfg, "cuda"), d["W13"], d["W2"])
    c13, s13 = tile_e4m3(d["W13"])
    c2, s2 = tile_e4m3(d["W2"])
    bufs = B.alloc_buffers(cfg, "cuda")
    B.moe_load_fp8_weights(cfg, c13, s13, c2, s2, bufs.scratch)
    got = run(shape, d, cfg, bufs, None, None)
    for name in OUTS:
        assert torch.equal(got[name], ref[name]), name
    # a second step reuses the loaded weights (nothing is quantised again)
    again = run(shape, d, cfg, bufs, None, None)
    for name in OUTS:
        assert torch.equal(again[name], ref[name]), name


def test_load_refuses_the_mx_recipe_and_bf16():
    from workloads import DT_MXFP8
    for dt in (DT_MXFP8, 0):
        cfg = B.config(SHAPES[0].with_(dtype=dt))
        with pytest.raises(B.MoEError) as e:
            B.moe_load_fp8_weights(cfg, 4096, 4096, 4096, 4096, 4096)
        assert e.value.code == 2
