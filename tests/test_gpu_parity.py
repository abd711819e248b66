"""Parity of the CUDA path (through the C-ABI) with the CPU oracle.

Small shapes that the oracle finishes in seconds but that still span several
GEMM tiles and ragged tails, plus edge cases: one expert, empty experts, every
token on one expert, capacity drops, shared experts, group-limited sigmoid
routing, 256 experts, and an empty batch.
"""
import numpy as np
import pytest
import torch

from workloads import SIGMOID, TINY, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

H_ = pytest.importorskip("harness")

SHAPES = [
    TINY,
    MoEShape("one_expert", T=200, H=256, E=1, k=1, F=128),
    MoEShape("ragged", T=333, H=384, E=2, k=2, F=384),
    MoEShape("grouped_shared", T=512, H=256, E=64, k=8, F=128, n_shared=1, score_fn=SIGMOID,
             n_groups=8, topk_groups=4, bias_kind="normal"),
    MoEShape("e256", T=300, H=128, E=256, k=8, F=128, score_fn=SIGMOID, n_groups=8,
             topk_groups=4, bias_kind="normal"),
    MoEShape("capacity_drop", T=1024, H=128, E=16, k=4, F=128, score_fn=SIGMOID,
             capacity_factor=0.5, bias_kind="normal"),
    MoEShape("wide_tiles", T=640, H=512, E=4, k=2, F=768, n_shared=2),
    # >= 512 rows per expert: the CTA-pair GEMM tiles (256 rows), ragged counts
    MoEShape("pair_tiles", T=2100, H=512, E=4, k=2, F=512, n_shared=1),
    # tensor-core router (E % 128 == 0) with T past one 1024-token weight-gradient
    # chunk: chunks of 1024, 1024 and 452 tokens, the last ragged within a k-block
    MoEShape("e128_chunks", T=2500, H=256, E=128, k=4, F=128, bias_kind="zipf"),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_layer_steps_match_oracle(shape):
    inp = make_inputs(shape, seed=0)
    g = H_.run_layer(shape, inp)
    H_.check_steps(shape, inp, g)


@pytest.mark.parametrize("shape", SHAPES[:4] + SHAPES[-2:], ids=lambda s: s.name)
def test_layer_end_to_end_matches_oracle(shape):
    inp = make_inputs(shape, seed=1)
    g = H_.run_layer(shape, inp)
    H_.check_end_to_end(shape, inp, g)


def test_all_tokens_on_one_expert_and_empty_experts():
    shape = MoEShape("hot", T=700, H=128, E=8, k=2, F=256)
    inp = make_inputs(shape, seed=2)
    b = torch.zeros(8)
    b[3] = 100.0                       # every token picks expert 3 first
    b[5] = 50.0                        # ... and expert 5 second; 6 experts stay empty
    inp["bias"] = b
    g = H_.run_layer(shape, inp)
    cnt = g["counts"].cpu().numpy()
    assert cnt[3] == 700 and cnt[5] == 700 and cnt.sum() == 1400
    H_.check_steps(shape, inp, g)


@pytest.mark.parametrize("E", [4, 128], ids=["simt_router", "tensor_core_router"])
def test_empty_batch(E):
    shape = MoEShape("empty", T=0, H=128, E=E, k=2, F=128)
    inp = make_inputs(shape.with_(T=1), seed=3)
    inp["x"] = inp["x"][:0].contiguous()
    inp["dY"] = inp["dY"][:0].contiguous()
    g = H_.run_layer(shape, inp)
    assert (g["counts"].cpu() == 0).all()
    assert (g["dW13"].float().cpu() == 0).all() and (g["dW2"].float().cpu() == 0).all()
    assert (g["dW_r"].cpu() == 0).all()


def test_repeat_runs_are_bitwise_identical():
    shape = SHAPES[3]
    inp = make_inputs(shape, seed=4)
    a = H_.run_layer(shape, inp)
    b = H_.run_layer(shape, inp)
    for name in ("logits", "idx", "row_of", "token_of", "out", "dx", "dW_r", "dW13", "dW2"):
        assert torch.equal(a[name].view(torch.uint8), b[name].view(torch.uint8)), name
