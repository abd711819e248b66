"""Paged stashing: the rows layers keep for their backward in one shared pool.

Reading of "Scalable Training of Mixture-of-Experts Models with Megatron Core"
(es summary, Resumen técnico §2.3.C, paged stashing: the dynamic buffers are
managed inside the CUDA graph instead of being reserved for the worst case).
With cfg.stash_pool_pages = P, x_perm, GU, h and y_perm are the tensors of a
pool of P pages of 128 rows shared by the layers of a step; each forward takes
the pages its kept rows need on the device, each backward gives them back.

Two layers share a pool sized to exactly what they need: forward A, forward B,
backward B, backward A. Every output must be bit-identical to the same layer run
on its own worst-case buffers (the kernels are deterministic, and that path is
checked against the oracle elsewhere), and every page table must equal the
oracle's (oracle.stash_page_table) for the counts and offsets the GPU produced.
"""
import numpy as np
import pytest
import torch

import routing_dispatch_expert_router_gb300.binding as B
from oracle import moe_oracle as O
from workloads import DT_FP8, DT_MXFP8, SIGMOID, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

SHAPES = [
    # dropless, one shared expert, group-limited sigmoid routing (single-CTA tiles)
    MoEShape("paged_shared", T=512, H=256, E=16, k=4, F=256, n_shared=1, score_fn=SIGMOID,
             n_groups=4, topk_groups=2, bias_kind="normal"),
    # capacity mode: segments of C rows, only their first ceil(kept/128) blocks paged
    MoEShape("paged_capacity", T=1024, H=256, E=8, k=2, F=256, capacity_factor=0.5),
    # >= 512 rows per expert: CTA-pair tiles and the pair kernel's GU ring
    MoEShape("paged_pairs", T=2100, H=512, E=4, k=2, F=512, n_shared=1),
    # the routing weight inside the expert and the recompute of h
    MoEShape("paged_reordered", T=600, H=256, E=8, k=2, F=256, weights_in_expert=1,
             recompute_h=1),
    MoEShape("paged_fp8", T=1024, H=768, E=8, k=2, F=256, score_fn=SIGMOID,
             capacity_factor=0.5, bias_kind="normal", dtype=DT_FP8),
    MoEShape("paged_fp8_recompute", T=700, H=256, E=8, k=2, F=256, dtype=DT_FP8,
             recompute_h=1),
    MoEShape("paged_mxfp8", T=1024, H=512, E=8, k=2, F=256, score_fn=SIGMOID,
             capacity_factor=0.75, bias_kind="normal", dtype=DT_MXFP8),
]

OUTS = ("out", "dx", "dW_r", "dW13", "dW2")


def _outs(shape):
    T, H, E, F, G = shape.T, shape.H, shape.E, shape.F, shape.E + shape.n_shared
    e = lambda *s, dt=torch.bfloat16: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    o = {"out": e(T, H), "dx": e(T, H), "dW_r": e(E, H, dt=torch.float32),
         "dW13": e(G, 2 * F, H), "dW2": e(G, H, F)}
    for t in o.values():
        t.view(torch.uint8).fill_(0xFF)
    return o


def _fwd(cfg, d, bufs, o, stream=None):
    P = B.params(d["W_r"], d["bias"], d["W13"], d["W2"])
    B.moe_layer_fwd(cfg, P, d["x"], o["out"], bufs.fwd_struct, bufs.scratch, stream=stream)


def _bwd(cfg, d, bufs, o, stream=None):
    P = B.params(d["W_r"], d["bias"], d["W13"], d["W2"])
    B.moe_layer_bwd(cfg, P, d["x"], d["dY"], bufs.fwd_struct, bufs.bwd_struct, o["dx"],
                    o["dW_r"], o["dW13"], o["dW2"], bufs.scratch, stream=stream)


def _own_buffers(shape, d):
    """The layer on its own worst-case buffers: outputs, counts, offsets."""
    cfg = B.config(shape)
    bufs = B.alloc_buffers(cfg, "cuda")
    o = _outs(shape)
    _fwd(cfg, d, bufs, o)
    _bwd(cfg, d, bufs, o)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(bufs.scratch) == 0
    return o, bufs.fwd["counts"].cpu().numpy(), bufs.fwd["offsets"].cpu().numpy()


def _pages(counts) -> int:
    return int(sum(-(-int(c) // 128) for c in counts))


def _paged_cfg(shape, pages):
    cfg = B.config(shape)
    cfg.stash_pool_pages = pages
    return cfg


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_two_layers_share_a_pool_bit_identical(shape):
    dA = make_inputs(shape, seed=0, device="cuda")
    dB = make_inputs(shape, seed=1, device="cuda")
    refA, cA, oA = _own_buffers(shape, dA)
    refB, cB, oB = _own_buffers(shape, dB)
    nA, nB = _pages(cA), _pages(cB)
    P = nA + nB                                       # exactly what the two layers need
    cfg = _paged_cfg(shape, P)
    pool = B.alloc_stash_pool(cfg, P)
    for t in pool.tensors.values():
        t.view(torch.uint8).fill_(0xFF)               # NaN: a row read before it is written shows
    bA = B.alloc_buffers(cfg, "cuda", pool=pool)
    bB = B.alloc_buffers(cfg, "cuda", pool=pool)
    R = int(bA.sizes.rows_max)
    assert int(bA.sizes.stash_table_len) == R // 128 + 2
    assert P * 128 <= 2 * R                           # the pool is never more than worst case
    oA_, oB_ = _outs(shape), _outs(shape)
    _fwd(cfg, dA, bA, oA_)
    _fwd(cfg, dB, bB, oB_)
    torch.cuda.synchronize()
    assert int(pool.top.item()) == P
    for bufs, counts, offsets, top in ((bA, cA, oA, 0), (bB, cB, oB, nA)):
        table, _, full = O.stash_page_table(counts, offsets, R, P, top)
        assert not full
        np.testing.assert_array_equal(bufs.fwd["stash_table"].cpu().numpy(), table)
    _bwd(cfg, dB, bB, oB_)
    torch.cuda.synchronize()
    assert int(pool.top.item()) == nA                 # B's pages are back
    _bwd(cfg, dA, bA, oA_)
    torch.cuda.synchronize()
    assert int(pool.top.item()) == 0
    for bufs in (bA, bB):
        assert B.moe_last_device_status(bufs.scratch) == 0
    for name in OUTS:
        assert torch.equal(oA_[name], refA[name]), f"layer A {name}"
        assert torch.equal(oB_[name], refB[name]), f"layer B {name}"


@pytest.mark.parametrize("shape", [SHAPES[1], SHAPES[4]], ids=lambda s: s.name)
def test_a_layer_that_does_not_fit_reports_and_takes_nothing(shape):
    """One page short: the layer takes no page, maps every block to the spill
    page, records MOE_ERR_STASH_FULL, and the step runs to its end inside the
    pool; the counter is unchanged."""
    d = make_inputs(shape, seed=0, device="cuda")
    _, counts, _ = _own_buffers(shape, d)
    P = _pages(counts) - 1
    cfg = _paged_cfg(shape, P)
    pool = B.alloc_stash_pool(cfg, P)
    bufs = B.alloc_buffers(cfg, "cuda", pool=pool)
    o = _outs(shape)
    _fwd(cfg, d, bufs, o)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(bufs.scratch) == 7          # MOE_ERR_STASH_FULL
    assert int(pool.top.item()) == 0
    table = bufs.fwd["stash_table"].cpu().numpy()
    assert (table[:-1] == P).all() and table[-1] == 0
    _bwd(cfg, d, bufs, o)
    torch.cuda.synchronize()
    assert int(pool.top.item()) == 0
    # the library stays usable: the next step with a pool that fits is exact
    ref, counts, _ = _own_buffers(shape, d)
    cfg2 = _paged_cfg(shape, _pages(counts))
    pool2 = B.alloc_stash_pool(cfg2, _pages(counts))
    b2 = B.alloc_buffers(cfg2, "cuda", pool=pool2)
    o2 = _outs(shape)
    _fwd(cfg2, d, b2, o2)
    _bwd(cfg2, d, b2, o2)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(b2.scratch) == 0
    for name in OUTS:
        assert torch.equal(o2[name], ref[name]), name


@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[4]], ids=lambda s: s.name)
def test_two_layer_step_with_a_pool_replays_from_a_cuda_graph(shape):
    """The page allocation and release happen on the device, so the two-layer
    step (forward A, forward B, backward B, backward A) is captured once and
    replayed with the same bits."""
    dA = make_inputs(shape, seed=2, device="cuda")
    dB = make_inputs(shape, seed=3, device="cuda")
    _, cA, _ = _own_buffers(shape, dA)
    _, cB, _ = _own_buffers(shape, dB)
    P = _pages(cA) + _pages(cB) + 3
    cfg = _paged_cfg(shape, P)
    pool = B.alloc_stash_pool(cfg, P)
    bA = B.alloc_buffers(cfg, "cuda", pool=pool)
    bB = B.alloc_buffers(cfg, "cuda", pool=pool)
    oA, oB = _outs(shape), _outs(shape)

    def step(s):
        _fwd(cfg, dA, bA, oA, s)
        _fwd(cfg, dB, bB, oB, s)
        _bwd(cfg, dB, bB, oB, s)
        _bwd(cfg, dA, bA, oA, s)

    step(None)
    torch.cuda.synchronize()
    ref = {("A", k): v.clone() for k, v in oA.items()}
    ref.update({("B", k): v.clone() for k, v in oB.items()})
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
        for t in list(oA.values()) + list(oB.values()):
            t.view(torch.uint8).fill_(0xFF)
        g.replay()
        torch.cuda.synchronize()
        assert int(pool.top.item()) == 0
        for bufs in (bA, bB):
            assert B.moe_last_device_status(bufs.scratch) == 0
        for (who, k), v in ref.items():
            got = (oA if who == "A" else oB)[k]
            assert torch.equal(got, v), (who, k)


@pytest.mark.slow
def test_paged_stash_at_full_size_is_bit_identical():
    """The FP8 DeepSeek-V3-shaped layer (T=16384, H=7168, E=256, top-8, capacity 1.25),
    the benched workload, on a pool of exactly its live pages -- fewer rows than its
    worst-case buffers -- against the same layer on its own buffers: every output the
    same bits."""
    from workloads import DSV3_FP8
    shape = DSV3_FP8
    torch.cuda.empty_cache()
    d = make_inputs(shape, seed=0, device="cuda")
    ref, counts, _ = _own_buffers(shape, d)
    torch.cuda.empty_cache()
    P = _pages(counts)
    cfg = _paged_cfg(shape, P)
    pool = B.alloc_stash_pool(cfg, P)
    bufs = B.alloc_buffers(cfg, "cuda", pool=pool)
    assert (P + 1) * 128 < int(bufs.sizes.rows_max)      # capacity mode: the pool is smaller
    o = _outs(shape)
    _fwd(cfg, d, bufs, o)
    torch.cuda.synchronize()
    assert int(pool.top.item()) == P
    _bwd(cfg, d, bufs, o)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(bufs.scratch) == 0
    assert int(pool.top.item()) == 0
    for name in OUTS:
        assert torch.equal(o[name], ref[name]), name
