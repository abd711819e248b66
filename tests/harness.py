"""GPU-vs-oracle parity harness shared by the GPU tests.

Runs one layer step through the C-ABI (forward and backward), returns every
output and intermediate as host arrays, and checks each step against the CPU
oracle applied to the GPU's own inputs of that step (so a mismatch points at
one kernel), plus the whole layer against the oracle from the raw inputs.
"""
from __future__ import annotations

import numpy as np
import torch

import routing_dispatch_expert_router_gb300.binding as B
from oracle import moe_oracle as O

BF16_ATOL = 1e-2
BF16_RTOL = 1e-2


def f64(t) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def i64(t) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)


def assert_close(name, got, ref, atol=BF16_ATOL, rtol=BF16_RTOL, scale=None):
    """|got - ref| <= atol + rtol * scale, scale = |ref| unless given (NaN fails)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    err = np.abs(got - ref)
    scale = np.abs(ref) if scale is None else np.asarray(scale, np.float64)
    bad = ~(err <= atol + rtol * scale)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err, -1)), bad.shape)
        raise AssertionError(f"{name}: {int(bad.sum())}/{bad.size} elements out of tolerance; "
                             f"worst at {i}: gpu={got[i]!r} ref={ref[i]!r}")


def assert_equal(name, got, ref):
    got = np.asarray(got)
    ref = np.asarray(ref)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    bad = got != ref
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{name}: {int(bad.sum())}/{bad.size} differ; first at {tuple(i)}: "
                             f"gpu={got[tuple(i)]} ref={ref[tuple(i)]}")


# End-to-end comparisons (from the raw inputs) against the plain per-element
# rule of the bf16 outputs, 1e-2 + 1e-2 |ref|, or the FP8 configuration's
# 5e-2 relative, whatever tolerance the check itself applies: one record per
# tensor (name, elements beyond the plain rule, elements, largest ratio of
# error to the plain bound). tests/conftest.py prints them after the run.
PLAIN_RECORDS: list = []
# The bf16 end-to-end checks that need the widened bound (sums of independently
# rounded bf16 summands: dx, dW13, dW2) are also capped at this many times the
# plain bound; the largest ratio observed over the GPU suite is 1.8 (dW13 of
# the CTA-pair case; 1.7 for Mixtral-sized dx), so the cap leaves about a
# factor of two.
PLAIN_CAP = 4.0


def plain_rule(name, got, ref, fp8: bool = False) -> float:
    """Records how far `got` sits from the plain per-element rule; returns the
    largest error / bound ratio (<= 1 where the plain rule holds)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = 5e-2 * np.abs(ref) if fp8 else BF16_ATOL + BF16_RTOL * np.abs(ref)
    err = np.abs(got - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(err == 0, 0.0, err / bound)
    worst = float(ratio.max()) if ratio.size else 0.0
    PLAIN_RECORDS.append((name, int((ratio > 1).sum()), int(ratio.size), worst))
    return worst


def read_rows(m) -> np.ndarray:
    """Rows of the permuted buffers that the grouped GEMMs read (and the
    dispatch writes): each segment's kept rows plus the rest of its last
    128-row block."""
    R, off, cnt = m["R"], m["offsets"], m["counts"]
    live = np.zeros(R, dtype=bool)
    for g in range(len(cnt)):
        live[off[g]: min(off[g + 1], off[g] + -(-int(cnt[g]) // 128) * 128)] = True
    return live


def _poison(t: torch.Tensor):
    """Fill with 0xFF bytes (NaN for floats, -1 for int32): unwritten output shows."""
    t.view(torch.uint8).fill_(0xFF)


def run_layer(shape, inp: dict, backward: bool = True, device: str = "cuda",
              replay_idx=None) -> dict:
    """One forward (+backward) through moe_layer_fwd / moe_layer_bwd; with
    replay_idx [T,k], the forward runs its stages with moe_route_replay on those
    experts in place of moe_route."""
    cfg = B.config(shape)
    bufs = B.alloc_buffers(cfg, device, backward=backward)
    for t in list(bufs.fwd.values()) + list(bufs.bwd.values()):
        _poison(t)
    d = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    T, H, E, F = shape.T, shape.H, shape.E, shape.F
    G = E + shape.n_shared
    P = B.params(d["W_r"], d["bias"], d["W13"], d["W2"])
    out = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    _poison(out)
    if replay_idx is None:
        B.moe_layer_fwd(cfg, P, d["x"], out, bufs.fwd_struct, bufs.scratch)
    else:
        f = bufs.fwd
        f["idx"].copy_(torch.as_tensor(replay_idx, dtype=torch.int32).reshape(f["idx"].shape))
        B.moe_quantize_weights(cfg, d["W13"], d["W2"], bufs.scratch)
        B.moe_route_replay(cfg, d["x"], d["W_r"], d["bias"], f["idx"], f["logits"], f["w"],
                           bufs.scratch)
        B.moe_permute(cfg, d["x"], f["idx"], f["counts"], f["offsets"], f["row_of"],
                      f["token_of"], f["sel_offsets"], f["sel_tokens"], f["x_perm"], bufs.scratch)
        B.moe_grouped_ffn_fwd(cfg, f["x_perm"], f["counts"], f["offsets"], d["W13"], d["W2"],
                              f["GU"], f["h"], f["y_perm"], bufs.scratch)
        B.moe_unpermute(cfg, f["y_perm"], f["row_of"], f["w"], f["offsets"], out)
    res = {"out": out}
    if backward:
        dx = torch.empty(T, H, dtype=torch.bfloat16, device=device)
        dW_r = torch.empty(E, H, dtype=torch.float32, device=device)
        dW13 = torch.empty(G, 2 * F, H, dtype=torch.bfloat16, device=device)
        dW2 = torch.empty(G, H, F, dtype=torch.bfloat16, device=device)
        for t in (dx, dW_r, dW13, dW2):
            _poison(t)
        B.moe_layer_bwd(cfg, P, d["x"], d["dY"], bufs.fwd_struct, bufs.bwd_struct, dx, dW_r,
                        dW13, dW2, bufs.scratch)
        res.update(dx=dx, dW_r=dW_r, dW13=dW13, dW2=dW2)
    torch.cuda.synchronize()
    status = B.moe_last_device_status(bufs.scratch)
    assert status == 0, f"device status {status}"
    res.update(bufs.fwd)
    res.update(bufs.bwd)
    res["rows_max"] = int(bufs.sizes.rows_max)
    return res


def _ident(a):
    return a


def check_steps(shape, inp: dict, g: dict, backward: bool = True, replay_idx=None):
    """Every step of the GPU path against the oracle fed the GPU's step inputs.

    In the FP8 configurations the oracle quantises those inputs the way the
    layer does (block recipe: weights in 128x128 tiles, activations in 1x128
    slices along the reduction, weight-gradient operands in 128x1 slices along
    tokens; MXFP8: 32-element slices, each weight in its forward and its
    data-gradient form); quantising identical inputs is exact on both sides, so
    the same per-element tolerance applies."""
    fp8 = getattr(shape, "dtype", 0) in (1, 2)
    blk = O.fp8_block(shape) if fp8 else 128
    qr = (lambda a: O.quant_rows(a, blk)) if fp8 else _ident
    qc = (lambda a: O.quant_cols(a, blk)) if fp8 else _ident
    # the weights as the forward GEMMs and as the data gradients read them
    wf = (lambda W: O.fp8_weights(shape, W)[0]) if fp8 else _ident
    wd = (lambda W: O.fp8_weights(shape, W)[1]) if fp8 else _ident
    T, H, E, k, F, S = shape.T, shape.H, shape.E, shape.k, shape.F, shape.n_shared
    G = E + S
    x = f64(inp["x"])
    Wr = f64(inp["W_r"])
    bias = None if inp["bias"] is None else f64(inp["bias"])
    W13 = inp["W13"]
    W2 = inp["W2"]
    # a1: logits within the fp32 accumulation bound
    lg = f64(g["logits"])
    ref_l = O.router_logits(x, Wr)
    scale = np.abs(x) @ np.abs(Wr).T
    bad = np.abs(lg - ref_l) > 1e-5 * scale + 1e-30
    assert not bad.any(), f"logits: {int(bad.sum())} beyond 1e-5*sum|x w|"
    # a2: selection bit-exact on the GPU's logits (or the replayed experts),
    # weights close
    if replay_idx is None:
        idx_ref, w_ref = O.route(lg, shape, bias)
    else:
        idx_ref, w_ref = O.route_replay(lg, shape, bias, np.asarray(replay_idx).reshape(-1, shape.k))
    assert_equal("idx", i64(g["idx"]), idx_ref)
    assert_close("w", f64(g["w"]), w_ref, atol=1e-6, rtol=1e-5)
    # a3/a4: maps bit-exact, x_perm exact
    m = O.permutation_maps(i64(g["idx"]), shape)
    R = m["R"]
    assert_equal("counts", i64(g["counts"]), m["counts"])
    assert_equal("offsets", i64(g["offsets"]), m["offsets"])
    assert_equal("row_of", i64(g["row_of"]), m["row_of"])
    assert_equal("token_of", i64(g["token_of"])[:R], m["token_of"])
    assert_equal("sel_offsets", i64(g["sel_offsets"]), m["sel_offsets"])
    assert_equal("sel_tokens", i64(g["sel_tokens"])[:T * k], m["sel_tokens"])
    live = read_rows(m)
    xp = f64(g["x_perm"])[:R]
    xp[~live] = 0.0                     # rows no GEMM reads are not written
    assert_equal("x_perm", xp, O.permute(x, m))
    # a5/a6 per group on the GPU's rows
    off, cnt = m["offsets"], m["counts"]
    GU = f64(g["GU"])
    hh = f64(g["h"])
    yp = f64(g["y_perm"])
    for gi in range(G):
        if cnt[gi] == 0:
            continue
        rows = slice(off[gi], off[gi] + cnt[gi])
        w13 = wf(f64(W13[gi]))
        w2 = wf(f64(W2[gi]))
        gu_ref, h_ref = O.expert_fc1(qr(xp[rows]), w13)
        assert_close(f"GU[g={gi}]", GU[rows], gu_ref)
        assert_close(f"h[g={gi}]", hh[rows], O.round_bf16(O.silu(GU[rows, :F]) * GU[rows, F:]))
        assert_close(f"y[g={gi}]", yp[rows], O.expert_fc2(qr(hh[rows]), w2))
    # a7 combine on the GPU's y and weights
    wg = f64(g["w"])
    rof = m["row_of"]
    acc = np.zeros((T, H))
    for j in range(k):
        ok = rof[:, j] >= 0
        acc[ok] += wg[ok, j:j + 1] * yp[rof[ok, j]]
    for s in range(S):
        acc += yp[off[E + s]: off[E + s] + T]
    assert_close("out", f64(g["out"]), O.round_bf16(acc))
    if not backward:
        return
    dY = f64(inp["dY"])
    # a8 combine backward
    dO = f64(g["dO_perm"])
    dw = f64(g["dw"])
    for j in range(k):
        ok = rof[:, j] >= 0
        assert_close(f"dO[slot {j}]", dO[rof[ok, j]], O.round_bf16(wg[ok, j:j + 1] * dY[ok]))
        ref_dw = np.where(ok, np.einsum("th,th->t", dY, yp[np.maximum(rof[:, j], 0)]), 0.0)
        assert_close(f"dw[slot {j}]", dw[:, j], ref_dw, atol=1e-3, rtol=1e-3)
    for s in range(S):
        assert_equal("dO[shared]", dO[off[E + s]: off[E + s] + T], dY)
    pad = (m["token_of"] < 0) & live
    assert_equal("dO padding", dO[:R][pad], np.zeros((int(pad.sum()), H)))
    assert_equal("x_perm padding", xp[pad], np.zeros((int(pad.sum()), H)))
    # a14a: dlogits on the GPU's dw
    dl = f64(g["dlogits"])
    dl_ref = O.router_dlogits(shape, lg, i64(g["idx"]), wg, dw)
    assert_close("dlogits", dl, dl_ref, atol=1e-4, rtol=1e-4)
    # a9..a12 per group
    dGU = f64(g["dGU"])
    dX = f64(g["dX_perm"])
    dW13 = g["dW13"]
    dW2 = g["dW2"]
    for gi in range(G):
        w13 = wd(f64(W13[gi]))
        w2 = wd(f64(W2[gi]))
        if cnt[gi] == 0:
            assert_equal(f"dW2[g={gi}] empty", f64(dW2[gi]), np.zeros((H, F)))
            assert_equal(f"dW13[g={gi}] empty", f64(dW13[gi]), np.zeros((2 * F, H)))
            continue
        rows = slice(off[gi], off[gi] + cnt[gi])
        assert_close(f"dGU[g={gi}]", dGU[rows],
                     O.expert_fc2_dgrad_swiglu(qr(dO[rows]), w2, GU[rows]))
        # routed rows also carry their assignment's router-logit gradient,
        # added in fp32 before the one bf16 rounding
        ref_dx = O.expert_fc1_dgrad(qr(dGU[rows]), w13, rounding=False)
        if gi < E:
            ref_dx = ref_dx + dl[m["token_of"][rows], gi][:, None] * Wr[gi][None, :]
        assert_close(f"dX[g={gi}]", dX[rows], O.round_bf16(ref_dx))
        assert_close(f"dW2[g={gi}]", f64(dW2[gi]), O.wgrad(qc(dO[rows]), qc(hh[rows])))
        assert_close(f"dW13[g={gi}]", f64(dW13[gi]), O.wgrad(qc(dGU[rows]), qc(xp[rows])))
    # a13: the kept rows (router terms included) plus the router terms of the
    # assignments dropped by the capacity limit
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
    assert_close("dx", f64(g["dx"]), O.round_bf16(acc))
    # a14b
    assert_close("dW_r", f64(g["dW_r"]), dl.T @ x, atol=1e-3, rtol=1e-4)


def wgrad_summand_scale(shape, x, dY, fwd, bwd):
    """Sum over each group's rows of |a_r| |b_r|^T for dW13 = dGU^T x_perm and
    dW2 = dO^T h. End to end, the GPU and the oracle round every dGU, GU and h
    element to bf16 independently, so one summand can move by up to 2^-8 of
    itself; over K rows the weight gradient can then differ by up to 2^-8 of
    this sum (far more than 2^-8 of |result| when K is large and the terms
    cancel). The end-to-end weight-gradient checks scale the relative
    tolerance by |result| plus this sum; the per-step checks, which feed the
    GPU's own dGU and x_perm to the oracle, keep the plain tolerance."""
    E, S = shape.E, shape.n_shared
    idx, kept = fwd["idx"], fwd["maps"]["row_of"] >= 0
    s13 = np.zeros_like(bwd["dW13"])
    s2 = np.zeros_like(bwd["dW2"])
    for e in range(E):
        tt, jj = np.nonzero((idx == e) & kept)
        if tt.size == 0:
            continue
        s13[e] = np.abs(bwd["dGU"][tt, jj]).T @ np.abs(x[tt])
        s2[e] = np.abs(bwd["dO"][tt, jj]).T @ np.abs(fwd["h"][tt, jj])
    for s in range(S):
        s13[E + s] = np.abs(bwd["dGU_s"][s]).T @ np.abs(x)
        s2[E + s] = np.abs(O.round_bf16(dY)).T @ np.abs(fwd["h_s"][s])
    return s13, s2


def check_end_to_end(shape, inp: dict, g: dict, backward: bool = True):
    """The whole layer against the oracle run from the raw inputs."""
    x = f64(inp["x"])
    Wr = f64(inp["W_r"])
    bias = None if inp["bias"] is None else f64(inp["bias"])
    W13 = f64(inp["W13"])
    W2 = f64(inp["W2"])
    fwd = O.layer_forward(shape, x, Wr, bias, W13, W2, logits=f64(g["logits"]))
    assert_equal("idx (e2e)", i64(g["idx"]), fwd["idx"])
    plain_rule(f"{shape.name} out", f64(g["out"]), fwd["out"])
    assert_close("out (e2e)", f64(g["out"]), fwd["out"])
    if not backward:
        return
    dY = f64(inp["dY"])
    bwd = O.layer_backward(shape, x, Wr, W13, W2, fwd, dY)
    # dx is a sum of bf16 summands that the two sides round independently
    # (each expert's input gradient, which on the GPU also holds its router
    # term): tolerance relative to |dx| plus the summands' magnitudes
    router = np.abs(np.take_along_axis(bwd["dlogits"], fwd["idx"], axis=1))[:, :, None] * \
        np.abs(Wr)[fwd["idx"]]
    mag = np.abs(bwd["dx"]) + np.abs(bwd["dX"]).sum(axis=1) + np.abs(bwd["dX_s"]).sum(axis=0) + \
        router.sum(axis=1)
    assert plain_rule(f"{shape.name} dx", f64(g["dx"]), bwd["dx"]) <= PLAIN_CAP
    assert_close("dx (e2e)", f64(g["dx"]), bwd["dx"], scale=mag)
    s13, s2 = wgrad_summand_scale(shape, x, dY, fwd, bwd)
    assert plain_rule(f"{shape.name} dW13", f64(g["dW13"]), bwd["dW13"]) <= PLAIN_CAP
    assert plain_rule(f"{shape.name} dW2", f64(g["dW2"]), bwd["dW2"]) <= PLAIN_CAP
    assert_close("dW13 (e2e)", f64(g["dW13"]), bwd["dW13"], scale=np.abs(bwd["dW13"]) + s13)
    assert_close("dW2 (e2e)", f64(g["dW2"]), bwd["dW2"], scale=np.abs(bwd["dW2"]) + s2)
    plain_rule(f"{shape.name} dW_r", f64(g["dW_r"]), bwd["dW_r"])
    assert_close("dW_r (e2e)", f64(g["dW_r"]), bwd["dW_r"], atol=1e-2, rtol=1e-2)


def assert_close_fp8(name, got, ref, rel=5e-2, extra=None):
    """The FP8 rule: |gpu-ref| <= rel*(|ref| + rms(ref) + extra) per element
    (extra: an added per-element scale, 0 unless given) and a relative
    Frobenius error <= rel over the tensor."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    scale = np.abs(ref) + rms + (0.0 if extra is None else extra)
    assert_close(name, got, ref, atol=0.0, rtol=rel, scale=scale)
    den = float(np.linalg.norm(ref))
    if den > 0:
        fro = float(np.linalg.norm(got - ref)) / den
        assert fro <= rel, f"{name}: relative Frobenius error {fro:.3g} > {rel}"


def check_end_to_end_fp8(shape, inp: dict, g: dict):
    """The FP8 layer against the oracle's FP8 layer run from the raw inputs."""
    x = f64(inp["x"])
    Wr = f64(inp["W_r"])
    bias = None if inp["bias"] is None else f64(inp["bias"])
    W13 = f64(inp["W13"])
    W2 = f64(inp["W2"])
    fwd = O.layer_forward_fp8(shape, x, Wr, bias, W13, W2, logits=f64(g["logits"]))
    assert_equal("idx (fp8 e2e)", i64(g["idx"]), fwd["idx"])
    plain_rule(f"{shape.name} out", f64(g["out"]), fwd["out"], fp8=True)
    assert_close_fp8("out (fp8 e2e)", f64(g["out"]), fwd["out"])
    dY = f64(inp["dY"])
    bwd = O.layer_backward_fp8(shape, x, Wr, W13, W2, fwd, dY)
    # The weight gradients sum, over an expert's rows, products of operands
    # that each side quantises to E4M3 from its own bf16 tensors (dGU, h, dO,
    # x_perm differ by bf16 roundings between the two sides). Where such a
    # difference straddles an E4M3 rounding boundary the operand moves by one
    # E4M3 step, up to 2^-3 of itself; with hundreds of rows and cancellation
    # that exceeds 5e-2 of a small |dW| element. So, as for the bf16 layer's
    # weight gradients, the per-element part of the rule adds the summands'
    # magnitudes S = sum_r |a_r| |b_r|, here weighted by 2^-4 (half an E4M3
    # step); the relative Frobenius error stays <= 5e-2 on every tensor.
    s13, s2 = wgrad_summand_scale(shape, x, dY, fwd, bwd)
    extra = {"dW13": 2.0 ** -4 * s13, "dW2": 2.0 ** -4 * s2}
    for n in ("dx", "dW13", "dW2", "dW_r"):
        plain_rule(f"{shape.name} {n}", f64(g[n]), bwd[n], fp8=True)
        assert_close_fp8(f"{n} (fp8 e2e)", f64(g[n]), bwd[n], extra=extra.get(n))
