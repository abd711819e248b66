"""moe_permute_noalloc: dispatch for callers that cannot provide scratch memory.

Some callers cannot allocate device memory for this library -- code inside a
framework that owns every byte of device memory (a caching allocator, a plugin
host without a workspace API), or a path where cudaMalloc must not be called.
moe_permute_noalloc serves them with a fixed scratch array inside the library.
These tests call it through the C-ABI and check that its results equal
moe_permute's (maps bit-exact, dispatched rows exact) on two calls in a row,
the second with a smaller problem that runs on whatever the first call left in
the shared array; that a problem too large for the array is refused before
anything is launched; and that an index problem found on the device is read
back through moe_permute_noalloc_status.
"""
import pytest
import torch

import routing_dispatch_expert_router_gb300.binding as B
from workloads import SIGMOID, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

MAPS = ("counts", "offsets", "row_of", "token_of", "sel_offsets", "sel_tokens", "x_perm")

SHAPES = [
    MoEShape("first", T=1500, H=256, E=64, k=8, F=128, n_shared=1, score_fn=SIGMOID, n_groups=8,
             topk_groups=4, bias_kind="normal"),
    MoEShape("second", T=1000, H=128, E=16, k=4, F=128, score_fn=SIGMOID, capacity_factor=0.5,
             bias_kind="normal"),
]


def _routed(shape, dev):
    inp = make_inputs(shape, seed=5, weights=False, grad=False)
    cfg = B.config(shape)
    bufs = B.alloc_buffers(cfg, dev, backward=False)
    x = inp["x"].to(dev)
    bias = None if inp["bias"] is None else inp["bias"].to(dev)
    f = bufs.fwd
    B.moe_route(cfg, x, inp["W_r"].to(dev), bias, f["logits"], f["idx"], f["w"], bufs.scratch)
    return cfg, bufs, x


def _permute(fn, cfg, bufs, x, *extra):
    f = bufs.fwd
    fn(cfg, x, f["idx"], f["counts"], f["offsets"], f["row_of"], f["token_of"], f["sel_offsets"],
       f["sel_tokens"], f["x_perm"], *extra)


def test_noalloc_matches_permute_on_two_calls_in_a_row():
    dev = torch.device("cuda")
    for shape in SHAPES:
        cfg, bufs, x = _routed(shape, dev)
        _permute(B.moe_permute, cfg, bufs, x, bufs.scratch)
        ref = {n: bufs.fwd[n].clone() for n in MAPS}
        for n in MAPS:
            bufs.fwd[n].view(torch.uint8).fill_(0xFF)
        _permute(B.moe_permute_noalloc, cfg, bufs, x)
        torch.cuda.synchronize()
        R = int(ref["offsets"][-1])
        A = shape.T * shape.k
        # the rows the grouped GEMMs read: each segment's last 128-row block ends
        # them (rows past it, in capacity mode, are not written by either call)
        off = ref["offsets"].cpu().numpy()
        cnt = ref["counts"].cpu().numpy()
        live = torch.zeros(R, dtype=torch.bool)
        for gi in range(len(cnt)):
            live[off[gi]: min(off[gi + 1], off[gi] + -(-int(cnt[gi]) // 128) * 128)] = True
        live = live.to(dev)
        for n in ("counts", "offsets", "row_of", "sel_offsets"):
            assert torch.equal(bufs.fwd[n], ref[n]), (shape.name, n)
        assert torch.equal(bufs.fwd["token_of"][:R], ref["token_of"][:R]), shape.name
        assert torch.equal(bufs.fwd["sel_tokens"][:A], ref["sel_tokens"][:A]), shape.name
        assert torch.equal(bufs.fwd["x_perm"][:R][live].view(torch.uint8),
                           ref["x_perm"][:R][live].view(torch.uint8)), shape.name
        if shape.capacity_factor > 0:
            assert (bufs.fwd["row_of"] < 0).any(), "capacity case should drop assignments"


def test_noalloc_refuses_problems_larger_than_its_array():
    dev = torch.device("cuda")
    big = MoEShape("big", T=1 << 20, H=128, E=256, k=1, F=128)    # needs ~1 MiB of scratch
    cfg = B.config(big)
    t = lambda n, dt=torch.int32: torch.zeros(n, dtype=dt, device=dev)  # noqa: E731
    with pytest.raises(B.MoEError) as e:
        B.moe_permute_noalloc(cfg, t(64, torch.bfloat16), t(64), t(300), t(300), t(64), t(64),
                              t(300), t(64), t(64, torch.bfloat16))
    assert e.value.code == 3     # MOE_ERR_WORKSPACE, nothing launched


def test_noalloc_status_reports_index_problems():
    """An expert index past the last expert, and one repeated within a token,
    are recorded in the array's status word (MOE_ERR_DEVICE_CHECK) and dropped
    (row_of = -1); the next clean call starts from a cleared word."""
    dev = torch.device("cuda")
    shape = SHAPES[1]
    cfg, bufs, x = _routed(shape, dev)
    f = bufs.fwd
    idx = f["idx"].clone()
    _permute(B.moe_permute_noalloc, cfg, bufs, x)
    assert B.moe_permute_noalloc_status() == 0
    bad = idx.clone()
    bad[3, 0] = shape.E                 # out of range
    bad[7, 1] = bad[7, 0]               # the same expert twice
    f["idx"].copy_(bad)
    _permute(B.moe_permute_noalloc, cfg, bufs, x)
    assert B.moe_permute_noalloc_status() == 6
    assert int(f["row_of"][3, 0]) == -1 and int(f["row_of"][7, 1]) == -1
    f["idx"].copy_(idx)
    _permute(B.moe_permute_noalloc, cfg, bufs, x)
    assert B.moe_permute_noalloc_status() == 0
