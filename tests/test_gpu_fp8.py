"""The FP8 configuration (E4M3 with power-of-two block scales) on the GPU.

All six expert GEMMs run on the block-scaled FP8 tensor cores (E4M3 codes,
UE8M0 scales in tensor memory). Every step is checked against the
oracle fed the GPU's own inputs of that step and quantised the same way (exact
on both sides, so the bf16 per-element tolerance applies); the whole layer is checked against the oracle's FP8 layer
run from the raw inputs with the 5e-2 rule (per element against
|ref| + rms(ref), and on the relative Frobenius error).
"""
import pytest
import torch

from workloads import DT_FP8, DT_MXFP8, SIGMOID, MoEShape, make_inputs

pytestmark = pytest.mark.gpu

H_ = pytest.importorskip("harness")

# One expert, 64 tokens, k = 1: every FP8 GEMM is one or two 128 x 256 tiles
# (FC2: one tile over two 128-deep k-blocks). The first case to run.
SINGLE_TILE = MoEShape("fp8_single_tile", T=64, H=256, E=1, k=1, F=256, score_fn=SIGMOID,
                       bias_kind="normal", dtype=DT_FP8)

# Two experts of 512 rows each (four 128-row tiles), one 256-wide N tile of FC2
# and two of FC1, every token on both experts.
PAIR_TILES = MoEShape("fp8_two_experts", T=512, H=256, E=2, k=2, F=256, score_fn=SIGMOID,
                      bias_kind="normal", dtype=DT_FP8)

SHAPES = [
    SINGLE_TILE,
    PAIR_TILES,
    MoEShape("fp8_groups", T=512, H=256, E=16, k=4, F=256, score_fn=SIGMOID, n_groups=4,
             topk_groups=2, bias_kind="normal", dtype=DT_FP8),
    # H = 768: six 128-deep k-blocks (a partly used scale atom), three N tiles
    MoEShape("fp8_capacity_drop", T=1024, H=768, E=8, k=2, F=256, score_fn=SIGMOID,
             capacity_factor=0.5, bias_kind="normal", dtype=DT_FP8),
    # F = 768: FC1 over six tiles of 128 gate + 128 up columns, 2F = 1536 deep FC1 dgrad
    MoEShape("fp8_dsv3_like", T=2048, H=512, E=32, k=8, F=768, score_fn=SIGMOID, n_groups=8,
             topk_groups=4, bias_kind="normal", dtype=DT_FP8, capacity_factor=1.25),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_fp8_steps_match_oracle(shape):
    inp = make_inputs(shape, seed=0)
    g = H_.run_layer(shape, inp)
    H_.check_steps(shape, inp, g)


# (the single-tile case has one expert and k = 1: its routing weight is 1 for
# every token, so the router gradient is identically zero and a relative rule
# has nothing to compare; its steps are checked above)
@pytest.mark.parametrize("shape", SHAPES[1:], ids=lambda s: s.name)
def test_fp8_layer_end_to_end(shape):
    inp = make_inputs(shape, seed=1)
    g = H_.run_layer(shape, inp)
    H_.check_end_to_end_fp8(shape, inp, g)


@pytest.mark.parametrize("dtype", [DT_FP8, DT_MXFP8], ids=["block", "mx"])
def test_fp8_hot_and_empty_experts(dtype):
    """Every token on experts 3 and 5, six experts without a row: the column
    quantisers must deal only the two live segments' blocks, and the empty
    experts' weight-gradient tiles come out as zeros."""
    shape = MoEShape("fp8_hot", T=700, H=256, E=8, k=2, F=256, dtype=dtype)
    inp = make_inputs(shape, seed=2)
    b = torch.zeros(8)
    b[3] = 100.0                       # every token picks expert 3 first
    b[5] = 50.0                        # ... and expert 5 second
    inp["bias"] = b
    g = H_.run_layer(shape, inp)
    cnt = g["counts"].cpu().numpy()
    assert cnt[3] == 700 and cnt[5] == 700 and cnt.sum() == 1400
    for e in (0, 1, 2, 4, 6, 7):
        assert (g["dW13"][e].float().cpu() == 0).all() and (g["dW2"][e].float().cpu() == 0).all()
    H_.check_steps(shape, inp, g)
