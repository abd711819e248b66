"""The layer with the routing weight inside the expert (weights_in_expert = 1)
on the GPU against the oracle's reordered layer.

Per step, each fed the GPU's own inputs of that step: routing and maps
bit-exact, then per group the weighted h_s = bf16(w silu(G) U), y = bf16(h_s
W2^T), the unweighted combine, dO_perm = dY rows (exact copies), dw =
<dY W2, silu(G) U> from the FC2 data gradient, dlogits from that dw, the
weighted SwiGLU backward (dGU), dX_perm with the router term, dW2 = dO^T h_s,
dW13, dx and dW_r; end to end from the raw inputs against
layer_forward_reordered / layer_backward_reordered with the same rules as the
plain layer. One case runs CTA-pair GEMM tiles (the ring path of the FC2 data
gradient).
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from workloads import SIGMOID, TINY, MoEShape, make_inputs

import harness as H_

pytestmark = pytest.mark.gpu

SHAPES = [
    TINY.with_(name="tiny_reordered", weights_in_expert=1),
    MoEShape("groups_shared_reordered", T=512, H=256, E=64, k=8, F=128, n_shared=1,
             score_fn=SIGMOID, n_groups=8, topk_groups=4, bias_kind="normal", weights_in_expert=1),
    MoEShape("capacity_reordered", T=1024, H=384, E=8, k=2, F=384, score_fn=SIGMOID,
             capacity_factor=0.5, bias_kind="normal", weights_in_expert=1),
    # 2 experts x ~1024 rows, F % 256 == 0: CTA-pair tiles everywhere
    MoEShape("pair_tiles_reordered", T=1024, H=512, E=2, k=2, F=1024, router_std=0.02,
             weights_in_expert=1),
]


def check_steps_reordered(shape, inp, g):
    f64, i64 = H_.f64, H_.i64
    T, H, E, k, F, S = shape.T, shape.H, shape.E, shape.k, shape.F, shape.n_shared
    G = E + S
    x = f64(inp["x"])
    Wr = f64(inp["W_r"])
    bias = None if inp["bias"] is None else f64(inp["bias"])
    lg = f64(g["logits"])
    idx_ref, w_ref = O.route(lg, shape, bias)
    H_.assert_equal("idx", i64(g["idx"]), idx_ref)
    H_.assert_close("w", f64(g["w"]), w_ref, atol=1e-6, rtol=1e-5)
    m = O.permutation_maps(i64(g["idx"]), shape)
    R = m["R"]
    for n in ("counts", "offsets", "row_of"):
        H_.assert_equal(n, i64(g[n]), m[n])
    H_.assert_equal("token_of", i64(g["token_of"])[:R], m["token_of"])
    live = H_.read_rows(m)
    xp = f64(g["x_perm"])[:R]
    xp[~live] = 0.0                     # rows no GEMM reads are not written
    H_.assert_equal("x_perm", xp, O.permute(x, m))
    off, cnt, rof, tok = m["offsets"], m["counts"], m["row_of"], m["token_of"]
    wg = f64(g["w"])
    # the routing weight of every used row: w of its assignment, 1 for shared rows
    row_w = np.zeros(R)
    for j in range(k):
        ok = rof[:, j] >= 0
        row_w[rof[ok, j]] = wg[ok, j]
    row_w[off[E]:R] = np.where(tok[off[E]:R] >= 0, 1.0, 0.0)
    GU, hs, yp = f64(g["GU"]), f64(g["h"]), f64(g["y_perm"])
    for gi in range(G):
        if cnt[gi] == 0:
            continue
        rows = slice(off[gi], off[gi] + cnt[gi])
        w13, w2 = f64(inp["W13"][gi]), f64(inp["W2"][gi])
        H_.assert_close(f"GU[g={gi}]", GU[rows], O.expert_fc1(xp[rows], w13)[0])
        ref_h = O.round_bf16(row_w[rows][:, None] * O.silu(GU[rows, :F]) * GU[rows, F:])
        H_.assert_close(f"h_s[g={gi}]", hs[rows], ref_h)
        H_.assert_close(f"y[g={gi}]", yp[rows], O.expert_fc2(hs[rows], w2))
    acc = np.zeros((T, H))
    for j in range(k):
        ok = rof[:, j] >= 0
        acc[ok] += yp[rof[ok, j]]
    for s in range(S):
        acc += yp[off[E + s]: off[E + s] + T]
    H_.assert_close("out (unweighted combine)", f64(g["out"]), O.round_bf16(acc))
    dY = f64(inp["dY"])
    dO = f64(g["dO_perm"])
    for j in range(k):
        ok = rof[:, j] >= 0
        H_.assert_equal(f"dO[slot {j}]", dO[rof[ok, j]], dY[ok])
    pad = (tok < 0) & live
    H_.assert_equal("dO padding", dO[:R][pad], np.zeros((int(pad.sum()), H)))
    dGU, dX = f64(g["dGU"]), f64(g["dX_perm"])
    dw_ref = np.zeros((T, k))
    dl = f64(g["dlogits"])
    for gi in range(G):
        if cnt[gi] == 0:
            continue
        rows = slice(off[gi], off[gi] + cnt[gi])
        w13, w2 = f64(inp["W13"][gi]), f64(inp["W2"][gi])
        d_ref, dw_rows = O.expert_fc2_dgrad_swiglu_weighted(dO[rows], w2, GU[rows], row_w[rows])
        H_.assert_close(f"dGU[g={gi}]", dGU[rows], d_ref)
        if gi < E:
            r_idx = np.arange(off[gi], off[gi] + cnt[gi])
            for j in range(k):
                hit = np.isin(rof[:, j], r_idx)
                dw_ref[hit, j] = dw_rows[rof[hit, j] - off[gi]]
        ref_dx = O.expert_fc1_dgrad(dGU[rows], w13, rounding=False)
        if gi < E:
            ref_dx = ref_dx + dl[tok[rows], gi][:, None] * Wr[gi][None, :]
        H_.assert_close(f"dX[g={gi}]", dX[rows], O.round_bf16(ref_dx))
        H_.assert_close(f"dW2[g={gi}]", f64(g["dW2"][gi]), O.wgrad(dO[rows], hs[rows]))
        H_.assert_close(f"dW13[g={gi}]", f64(g["dW13"][gi]), O.wgrad(dGU[rows], xp[rows]))
    H_.assert_close("dw", f64(g["dw"]), dw_ref, atol=1e-3, rtol=1e-3)
    H_.assert_close("dlogits", dl, O.router_dlogits(shape, lg, i64(g["idx"]), wg, f64(g["dw"])),
                    atol=1e-4, rtol=1e-4)
    acc = np.zeros((T, H))
    idx_g = i64(g["idx"])
    for j in range(k):
        ok = rof[:, j] >= 0
        acc[ok] += dX[rof[ok, j]]
        drop = ~ok
        if drop.any():
            e_d = idx_g[drop, j]
            acc[drop] += dl[np.nonzero(drop)[0], e_d][:, None] * Wr[e_d]
    for s in range(S):
        acc += dX[off[E + s]: off[E + s] + T]
    H_.assert_close("dx", f64(g["dx"]), O.round_bf16(acc))
    H_.assert_close("dW_r", f64(g["dW_r"]), dl.T @ x, atol=1e-3, rtol=1e-4)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_reordered_steps_match_oracle(shape):
    inp = make_inputs(shape, seed=41)
    g = H_.run_layer(shape, inp)
    check_steps_reordered(shape, inp, g)


@pytest.mark.parametrize("shape", SHAPES[:3], ids=lambda s: s.name)
def test_reordered_layer_end_to_end(shape):
    f64 = H_.f64
    inp = make_inputs(shape, seed=42)
    g = H_.run_layer(shape, inp)
    x, Wr, W13, W2, dY = (f64(inp[n]) for n in ("x", "W_r", "W13", "W2", "dY"))
    bias = None if inp["bias"] is None else f64(inp["bias"])
    fwd = O.layer_forward_reordered(shape, x, Wr, bias, W13, W2, logits=f64(g["logits"]))
    H_.assert_equal("idx (e2e)", H_.i64(g["idx"]), fwd["idx"])
    H_.plain_rule(f"{shape.name} out", f64(g["out"]), fwd["out"])
    H_.assert_close("out (e2e)", f64(g["out"]), fwd["out"])
    bwd = O.layer_backward_reordered(shape, x, Wr, W13, W2, fwd, dY)
    # sums of independently rounded bf16 summands, as for the plain layer
    router = np.abs(np.take_along_axis(bwd["dlogits"], fwd["idx"], axis=1))[:, :, None] * \
        np.abs(Wr)[fwd["idx"]]
    mag = np.abs(bwd["dx"]) + np.abs(bwd["dX"]).sum(axis=1) + np.abs(bwd["dX_s"]).sum(axis=0) + \
        router.sum(axis=1)
    assert H_.plain_rule(f"{shape.name} dx", f64(g["dx"]), bwd["dx"]) <= H_.PLAIN_CAP
    H_.assert_close("dx (e2e)", f64(g["dx"]), bwd["dx"], scale=mag)
    # dW2 = dY^T h_s and dW13 = dGU^T x over each group's rows: the relative
    # part of the rule scales with |dW| plus the summands' magnitudes, as for
    # the plain layer's weight gradients
    idx, kept = fwd["idx"], fwd["maps"]["row_of"] >= 0
    s13, s2 = np.zeros_like(bwd["dW13"]), np.zeros_like(bwd["dW2"])
    for e in range(shape.E):
        tt, jj = np.nonzero((idx == e) & kept)
        if tt.size:
            s13[e] = np.abs(bwd["dGU"][tt, jj]).T @ np.abs(x[tt])
            s2[e] = np.abs(dY[tt]).T @ np.abs(fwd["hs"][tt, jj])
    for s_ in range(shape.n_shared):
        s13[shape.E + s_] = np.abs(bwd["dGU_s"][s_]).T @ np.abs(x)
        s2[shape.E + s_] = np.abs(dY).T @ np.abs(fwd["h_s"][s_])
    for n, summ in (("dW13", s13), ("dW2", s2)):
        assert H_.plain_rule(f"{shape.name} {n}", f64(g[n]), bwd[n]) <= H_.PLAIN_CAP
        H_.assert_close(f"{n} (e2e)", f64(g[n]), bwd[n], scale=np.abs(bwd[n]) + summ)
    H_.assert_close("dW_r (e2e)", f64(g["dW_r"]), bwd["dW_r"], atol=1e-2, rtol=1e-2)
