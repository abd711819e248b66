"""The FP8 configuration (E4M3 with power-of-two block scales) on the GPU.

Every step is checked against the oracle fed the GPU's own inputs of that
step and quantised the same way (exact on both sides, so the bf16 per-element
tolerance applies); the whole layer is checked against the oracle's FP8 layer
run from the raw inputs with the 5e-2 rule (per element against
|ref| + rms(ref), and on the relative Frobenius error).
"""
import pytest

from workloads import DT_FP8, SIGMOID, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

H_ = pytest.importorskip("harness")

SHAPES = [
    MoEShape("fp8_groups", T=512, H=256, E=16, k=4, F=256, score_fn=SIGMOID, n_groups=4,
             topk_groups=2, bias_kind="normal", dtype=DT_FP8),
    MoEShape("fp8_capacity_drop", T=1024, H=384, E=8, k=2, F=256, score_fn=SIGMOID,
             capacity_factor=0.5, bias_kind="normal", dtype=DT_FP8),
    MoEShape("fp8_dsv3_like", T=2048, H=512, E=32, k=8, F=256, score_fn=SIGMOID, n_groups=8,
             topk_groups=4, bias_kind="normal", dtype=DT_FP8, capacity_factor=1.25),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_fp8_steps_match_oracle(shape):
    inp = make_inputs(shape, seed=0)
    g = H_.run_layer(shape, inp)
    H_.check_steps(shape, inp, g)


@pytest.mark.parametrize("shape", SHAPES[:2], ids=lambda s: s.name)
def test_fp8_layer_end_to_end(shape):
    inp = make_inputs(shape, seed=1)
    g = H_.run_layer(shape, inp)
    H_.check_end_to_end_fp8(shape, inp, g)
