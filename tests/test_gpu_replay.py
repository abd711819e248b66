"""Router Replay on the GPU (moe_route_replay) against the oracle.

The experts of every token are given (recorded decisions) instead of taken
from the router's top-k; the weights are the router's for them. Checked:
replaying the router's own choice reproduces its weights (bit for bit for the
softmax router, whose replay runs the selection kernel's arithmetic); a replay
of other experts (seeded random, distinct per token, in random order) matches
the oracle step by step through the whole layer, forward and backward; an
expert index outside [0, E) is reported by the device status word.
"""
import numpy as np
import pytest
import torch

import routing_dispatch_expert_router_gb300.binding as B
from oracle import moe_oracle as O
from workloads import GROUP_MAX, SIGMOID, TINY, MoEShape, make_inputs

import harness as H_

pytestmark = pytest.mark.gpu

SHAPES = [
    TINY,
    MoEShape("sigmoid_groups_shared", T=512, H=256, E=64, k=8, F=128, n_shared=1,
             score_fn=SIGMOID, n_groups=8, topk_groups=4, bias_kind="normal"),
    MoEShape("e128_tensor_core_router", T=700, H=256, E=128, k=4, F=128, bias_kind="zipf"),
]


def _route(shape, d, replay=None):
    cfg = B.config(shape)
    sz = B.moe_query_sizes(cfg)
    dev = "cuda"
    sc = torch.zeros(sz.scratch_bytes, dtype=torch.uint8, device=dev)
    T, E, k = shape.T, shape.E, shape.k
    lg = torch.empty(T, E, dtype=torch.float32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    x, Wr = d["x"].to(dev), d["W_r"].to(dev)
    b = None if d["bias"] is None else d["bias"].to(dev)
    if replay is None:
        idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        B.moe_route(cfg, x, Wr, b, lg, idx, w, sc)
    else:
        idx = torch.as_tensor(replay, dtype=torch.int32).to(dev)
        B.moe_route_replay(cfg, x, Wr, b, idx, lg, w, sc)
    torch.cuda.synchronize()
    return lg, idx, w, B.moe_last_device_status(sc)


def _other_experts(shape, seed):
    """k distinct experts per token in random order (not the router's top-k)."""
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(shape.E)[: shape.k] for _ in range(shape.T)]).astype(np.int32)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_replaying_the_routers_choice_reproduces_its_weights(shape):
    d = make_inputs(shape, seed=11)
    lg, idx, w, st = _route(shape, d)
    assert st == 0
    lg2, idx2, w2, st2 = _route(shape, d, replay=idx.cpu().numpy())
    assert st2 == 0
    assert torch.equal(lg, lg2)
    assert torch.equal(idx, idx2)
    if shape.score_fn == SIGMOID:
        # tokens whose selection took fp64 keys weight with fp64 sigmoids there
        H_.assert_close("w", H_.f64(w2), H_.f64(w), atol=1e-6, rtol=1e-5)
    else:
        assert torch.equal(w.view(torch.int32), w2.view(torch.int32))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_replayed_layer_steps_match_oracle(shape):
    inp = make_inputs(shape, seed=12)
    idx = _other_experts(shape, seed=13)
    g = H_.run_layer(shape, inp, replay_idx=idx)
    H_.check_steps(shape, inp, g, replay_idx=idx)


def test_replayed_index_out_of_range_is_reported():
    shape = TINY
    d = make_inputs(shape, seed=14)
    idx = _other_experts(shape, seed=15)
    idx[5, 1] = shape.E            # one index past the last expert
    _, _, w, st = _route(shape, d, replay=idx)
    assert st == 6                 # MOE_ERR_DEVICE_CHECK
    assert float(w[5, 1]) == 0.0


def test_replayed_repeated_expert_is_reported_and_dropped():
    """A recorded idx row that names one expert twice: the second copy is
    reported (MOE_ERR_DEVICE_CHECK), weighted 0 by the replay and dropped by
    the dispatch (row_of = -1, not counted), so every counted row of an expert
    segment is written once. The expected maps are the stable counting sort of
    the remaining assignments, written out here."""
    shape = TINY
    d = make_inputs(shape, seed=16)
    idx = _other_experts(shape, seed=17)
    idx[9, 1] = idx[9, 0]          # token 9 names its first expert twice
    _, idx_d, w, st = _route(shape, d, replay=idx)
    assert st == 6
    assert float(w[9, 1]) == 0.0 and float(w[9, 0]) > 0.0
    cfg = B.config(shape)
    bufs = B.alloc_buffers(cfg, "cuda", backward=False)
    f = bufs.fwd
    x = d["x"].to("cuda")
    B.moe_permute(cfg, x, idx_d, f["counts"], f["offsets"], f["row_of"], f["token_of"],
                  f["sel_offsets"], f["sel_tokens"], f["x_perm"], bufs.scratch)
    torch.cuda.synchronize()
    assert B.moe_last_device_status(bufs.scratch) == 6
    T, E, k, a = shape.T, shape.E, shape.k, shape.row_align
    keep = np.ones((T, k), dtype=bool)
    keep[9, 1] = False
    toks = [[t for t in range(T) for j in range(k) if keep[t, j] and idx[t, j] == e]
            for e in range(E)]
    counts = np.array([len(v) for v in toks])
    offsets = np.concatenate([[0], np.cumsum((counts + a - 1) // a * a)])
    row_of = np.full((T, k), -1)
    for e in range(E):
        for r, t in enumerate(toks[e]):
            row_of[t, int(np.nonzero((idx[t] == e) & keep[t])[0][0])] = offsets[e] + r
    H_.assert_equal("counts", H_.i64(f["counts"]), counts)
    H_.assert_equal("offsets", H_.i64(f["offsets"]), offsets)
    H_.assert_equal("row_of", H_.i64(f["row_of"]), row_of)
    token_of = np.full(int(offsets[-1]), -1)
    token_of[row_of[keep]] = np.nonzero(keep)[0]
    H_.assert_equal("token_of", H_.i64(f["token_of"])[:offsets[-1]], token_of)
