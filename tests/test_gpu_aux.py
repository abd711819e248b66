"""Load-balancing loss on the GPU (moe_route_aux, moe_route_aux_bwd) against the oracle.

Forward: the selection counts are compared bit for bit, the mean
probabilities and the loss within fp32 summation error, the bias update bit
for bit; a second call gives the same bits (fixed summation order, the
arrival counter left at zero). Backward: dlogits of the loss, dx (bf16, one
rounding of dx + dl W_r) and dW_r (fp32, dW_r + dl^T x) with dloss scaled so
that the loss's share of dx is of order one. Shapes cover one to eight
experts per lane, ragged token blocks, the CUDA-core and the tensor-core
router weight gradient, both score functions, and a Qwen3-sized batch
(T=16384, H=4096, E=128, k=8); plus the empty batch and an out-of-range index.
"""
import numpy as np
import pytest
import torch

import routing_dispatch_expert_router_gb300.binding as B
from oracle import moe_oracle as O
from workloads import SIGMOID, TINY, MoEShape, make_inputs

import harness as H_

pytestmark = pytest.mark.gpu

SHAPES = [
    TINY,
    MoEShape("sigmoid_groups_e64", T=700, H=256, E=64, k=6, F=128, score_fn=SIGMOID, n_groups=8,
             topk_groups=4, bias_kind="normal"),
    MoEShape("softmax_zipf_e128_tc", T=1100, H=384, E=128, k=8, F=128, bias_kind="zipf"),
    MoEShape("sigmoid_e256_tc", T=300, H=256, E=256, k=8, F=128, score_fn=SIGMOID, n_groups=8,
             topk_groups=4, bias_kind="normal"),
]
COEFF, RATE = 0.01, 1e-3


def _bufs(shape, dev="cuda"):
    cfg = B.config(shape)
    sc = torch.zeros(B.moe_query_sizes(cfg).scratch_bytes, dtype=torch.uint8, device=dev)
    E = shape.E
    return cfg, sc, {"counts": torch.empty(E, dtype=torch.int32, device=dev),
                     "P": torch.empty(E, dtype=torch.float32, device=dev),
                     "loss": torch.empty(1, dtype=torch.float32, device=dev),
                     "bias_out": torch.empty(E, dtype=torch.float32, device=dev)}


def _route(shape, d, cfg, sc):
    T, E, k = shape.T, shape.E, shape.k
    lg = torch.empty(T, E, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    b = None if d["bias"] is None else d["bias"].cuda()
    B.moe_route(cfg, d["x"].cuda(), d["W_r"].cuda(), b, lg, idx, w, sc)
    return lg, idx, b


def _aux(cfg, sc, lg, b, idx, o, bias_out="separate"):
    bo = o["bias_out"] if bias_out == "separate" else bias_out
    B.moe_route_aux(cfg, lg, b, idx, COEFF, RATE, o["counts"], o["P"], o["loss"], bo, sc)
    torch.cuda.synchronize()
    return B.moe_last_device_status(sc)


def _check_fwd(shape, lg, b, idx, o):
    l64, i64 = H_.f64(lg), H_.i64(idx)
    bnp = None if b is None else b.cpu().numpy()
    loss, counts, P = O.aux_loss(l64, shape, bnp, i64, COEFF)
    H_.assert_equal("sel_counts", H_.i64(o["counts"]), counts)
    H_.assert_close("p_mean", H_.f64(o["P"]), P, atol=1e-7, rtol=2e-5)
    H_.assert_close("loss", H_.f64(o["loss"]), np.array([loss]), atol=0, rtol=2e-5)
    H_.assert_equal("bias_out", o["bias_out"].cpu().numpy(), O.bias_update(bnp, counts, shape, RATE))
    return counts


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_aux_loss_forward_matches_oracle(shape):
    d = make_inputs(shape, seed=21)
    cfg, sc, o = _bufs(shape)
    lg, idx, b = _route(shape, d, cfg, sc)
    assert _aux(cfg, sc, lg, b, idx, o) == 0
    _check_fwd(shape, lg, b, idx, o)
    first = {n: v.clone() for n, v in o.items()}
    # again: the same bits (fixed order; the arrival counter was reset)
    for v in o.values():
        v.view(torch.uint8).fill_(0xFF)
    assert _aux(cfg, sc, lg, b, idx, o) == 0
    for n in o:
        assert torch.equal(o[n], first[n]), n
    # the bias updated in place equals the separate output
    if b is not None:
        b2 = b.clone()
        assert _aux(cfg, sc, lg, b2, idx, o, bias_out=b2) == 0
        assert torch.equal(b2, first["bias_out"])


def _check_bwd(shape, x, W_r, lg, b, counts, cfg, sc, seed):
    T, H, E = shape.T, shape.H, shape.E
    l64 = H_.f64(lg)
    bnp = None if b is None else b.cpu().numpy()
    x64, W64 = H_.f64(x), H_.f64(W_r)
    # dloss that gives the loss's dx term a largest entry of about 1
    dl1 = O.aux_loss_dlogits(l64, shape, bnp, counts, COEFF, 1.0)
    dloss = float(1.0 / max(np.abs(dl1 @ W64).max(), 1e-30))
    g = torch.Generator().manual_seed(seed)
    dx0 = (0.1 * torch.randn(T, H, generator=g)).to(torch.bfloat16)
    dW0 = 0.1 * torch.randn(E, H, generator=g)
    dx, dW = dx0.cuda(), dW0.cuda()
    dl = torch.full((T, E), float("nan"), device="cuda")
    cnt = torch.as_tensor(counts, dtype=torch.int32).cuda()
    B.moe_route_aux_bwd(cfg, x, lg, b, W_r, cnt, COEFF, dloss, dl, dx, dW, sc)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(sc) == 0
    ref_dl, ref_dx, ref_dW = O.aux_loss_backward(shape, x64, W64, l64, bnp, counts, COEFF, dloss,
                                                 H_.f64(dx0), H_.f64(dW0))
    H_.assert_close("dlogits_aux", H_.f64(dl), ref_dl, atol=1e-6 * np.abs(ref_dl).max(),
                    rtol=1e-4)
    assert np.abs(ref_dx - H_.f64(dx0)).max() > 0.5          # the loss's term is not lost in dx
    H_.assert_close("dx", H_.f64(dx), ref_dx)
    scale = np.abs(H_.f64(dW0)) + np.abs(ref_dl).T @ np.abs(x64)
    H_.assert_close("dW_r", H_.f64(dW), ref_dW, atol=1e-6 * scale.max(), rtol=1e-5, scale=scale)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_aux_loss_backward_matches_oracle(shape):
    d = make_inputs(shape, seed=22)
    cfg, sc, o = _bufs(shape)
    lg, idx, b = _route(shape, d, cfg, sc)
    assert _aux(cfg, sc, lg, b, idx, o) == 0
    counts = _check_fwd(shape, lg, b, idx, o)
    _check_bwd(shape, d["x"].cuda(), d["W_r"].cuda(), lg, b, counts, cfg, sc, seed=5)


def test_aux_loss_qwen3_sized_batch():
    """T=16384, H=4096, E=128, k=8, softmax with a Zipf logit bias: 128 token
    blocks, the tensor-core dW_r path, every element compared."""
    shape = MoEShape("qwen3_sized", T=16384, H=4096, E=128, k=8, F=1536, bias_kind="zipf")
    g = torch.Generator().manual_seed(3)
    x = torch.randn(shape.T, shape.H, generator=g).to(torch.bfloat16).cuda()
    W_r = (torch.randn(shape.E, shape.H, generator=g) / 64).cuda()
    b = (0.5 * torch.log1p(torch.arange(shape.E, dtype=torch.float32))).flip(0).cuda()
    d = {"x": x, "W_r": W_r, "bias": b}
    cfg, sc, o = _bufs(shape)
    lg, idx, b = _route(shape, d, cfg, sc)
    assert _aux(cfg, sc, lg, b, idx, o) == 0
    counts = _check_fwd(shape, lg, b, idx, o)
    _check_bwd(shape, x, W_r, lg, b, counts, cfg, sc, seed=6)


def test_aux_loss_empty_batch():
    shape = MoEShape("empty", T=0, H=128, E=16, k=2, F=128)
    cfg, sc, o = _bufs(shape)
    b = torch.linspace(-1, 1, 16, device="cuda")
    assert _aux(cfg, sc, None, b, None, o) == 0
    assert torch.equal(o["counts"].cpu(), torch.zeros(16, dtype=torch.int32))
    assert torch.equal(o["P"].cpu(), torch.zeros(16))
    assert o["loss"].item() == 0.0
    assert torch.equal(o["bias_out"], b)
    dW = torch.ones(16, 128, device="cuda")
    B.moe_route_aux_bwd(cfg, None, None, b, torch.zeros(16, 128, device="cuda"), o["counts"],
                        COEFF, 1.0, None, None, dW, sc)
    torch.cuda.synchronize()
    assert torch.equal(dW, torch.ones_like(dW))


def test_aux_loss_out_of_range_index_is_reported_and_not_counted():
    shape = MoEShape("bad_idx", T=64, H=128, E=8, k=2, F=128)
    cfg, sc, o = _bufs(shape)
    lg = torch.zeros(64, 8, device="cuda")
    idx = torch.zeros(64, 2, dtype=torch.int32)
    idx[:, 1] = 1
    idx[7, 1] = 8                                   # outside [0, E)
    assert _aux(cfg, sc, lg, None, idx.cuda(), o) == 6
    assert o["counts"].cpu().tolist() == [64, 63, 0, 0, 0, 0, 0, 0]
    B.moe_clear_device_status(sc)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(sc) == 0
