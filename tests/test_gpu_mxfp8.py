"""The MXFP8 configuration (E4M3 with one power-of-two scale per 32 elements)
on the GPU.

Same path as the block-scaled FP8 configuration with the MX formats' 32-element
blocks: activations in 1x32 slices along each GEMM's reduced dimension,
weight-gradient operands in 32x1 slices along the tokens, and every expert
weight in two E4M3 forms (1x32 along its input dimension for the forward GEMMs,
32x1 along its output dimension for the data gradients). The block-scaled MMA
applies one scale per 32-deep K slice. Every step is checked against the oracle
fed the GPU's own inputs of that step and quantised the same way (exact on both
sides, so the bf16 per-element tolerance applies); the whole layer against the
oracle's MXFP8 layer run from the raw inputs with the 5e-2 rule.
"""
import pytest

from workloads import DT_MXFP8, SIGMOID, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

H_ = pytest.importorskip("harness")

SHAPES = [
    # one expert, k = 1: every GEMM one or two tiles
    MoEShape("mx_single_tile", T=64, H=256, E=1, k=1, F=256, score_fn=SIGMOID,
             bias_kind="normal", dtype=DT_MXFP8),
    MoEShape("mx_groups", T=512, H=256, E=16, k=4, F=256, score_fn=SIGMOID, n_groups=4,
             topk_groups=2, bias_kind="normal", dtype=DT_MXFP8),
    # H = 768: six K blocks of 128 (24 scale slices of 32) per row
    MoEShape("mx_capacity_drop", T=1024, H=768, E=8, k=2, F=256, score_fn=SIGMOID,
             capacity_factor=0.5, bias_kind="normal", dtype=DT_MXFP8),
    MoEShape("mx_dsv3_like", T=2048, H=512, E=32, k=8, F=768, score_fn=SIGMOID, n_groups=8,
             topk_groups=4, bias_kind="normal", dtype=DT_MXFP8, capacity_factor=1.25),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_mxfp8_steps_match_oracle(shape):
    inp = make_inputs(shape, seed=0)
    g = H_.run_layer(shape, inp)
    H_.check_steps(shape, inp, g)


# (the single-tile case: routing weight 1 for every token, a zero router
# gradient; its steps are checked above)
@pytest.mark.parametrize("shape", SHAPES[1:], ids=lambda s: s.name)
def test_mxfp8_layer_end_to_end(shape):
    inp = make_inputs(shape, seed=1)
    g = H_.run_layer(shape, inp)
    H_.check_end_to_end_fp8(shape, inp, g)
