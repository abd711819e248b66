"""Parity at the full workload sizes, in the launch configuration bench.py times.

The whole layer (fwd + bwd) runs at the Mixtral-, DeepSeek-V3- and
Qwen3-shaped sizes with inputs drawn on the device. Against the CPU oracle:
  * routing indices, weights, counts and every permutation map over ALL tokens
    (bit-exact; selection on the GPU's fp32 logits);
  * logits of sampled tokens;
  * each later step on sampled rows of sampled groups (the hottest, the
    coldest non-empty, the shared one, random ones), fed the GPU's own inputs
    of that step; weight gradients of sampled groups on sampled output rows;
  * dlogits over all tokens, dW_r of sampled experts;
  * out[t] and dx[t] of sampled tokens end to end from the raw inputs (both
    depend only on token t). Both are sums of several bf16 tensors that the
    two sides round independently (y or dX per expert, then the sum), so a
    rounding flip in one summand moves the sum by up to 2^-8 of that summand:
    these two comparisons scale the relative tolerance by |result| plus the
    summands' magnitudes instead of |result| alone. Every per-step comparison
    above uses the plain per-element tolerance.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from workloads import DSV3, DSV3_FP8, MIXTRAL, QWEN3, make_inputs

import harness as H_

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def host(t):
    return t.detach().to(torch.float64).cpu().numpy()


def group_weights(inp, g):
    return host(inp["W13"][g]), host(inp["W2"][g])


def pick_groups(counts, E, S, rng, n_random=3):
    routed = counts[:E]
    nz = np.nonzero(routed)[0]
    gs = {int(np.argmax(routed)), int(nz[np.argmin(routed[nz])])}
    gs |= set(int(v) for v in rng.choice(nz, size=min(n_random, nz.size), replace=False))
    gs |= {E + s for s in range(S)}
    return sorted(gs)


@pytest.mark.parametrize("shape", [MIXTRAL, QWEN3, DSV3, DSV3_FP8], ids=lambda s: s.name)
def test_full_size_layer_matches_oracle_on_samples(shape):
    torch.cuda.empty_cache()
    fp8 = shape.dtype == 1
    ident = lambda a: a  # noqa: E731
    qr = O.quant_rows if fp8 else ident
    qc = O.quant_cols if fp8 else ident
    qt = O.quant_tiles if fp8 else ident
    inp = make_inputs(shape, seed=0, device="cuda")
    g = H_.run_layer(shape, inp)
    rng = np.random.default_rng(0)
    T, Hd, E, k, F, S = shape.T, shape.H, shape.E, shape.k, shape.F, shape.n_shared
    x_dev = inp["x"]
    Wr = host(inp["W_r"])
    bias = None if inp["bias"] is None else host(inp["bias"])
    # ---- routing over all tokens
    lg = host(g["logits"])
    toks = rng.choice(T, size=128, replace=False)
    xs = host(x_dev[toks])
    ref_l = O.router_logits(xs, Wr)
    bound = 1e-5 * (np.abs(xs) @ np.abs(Wr).T)
    assert (np.abs(lg[toks] - ref_l) <= bound).all(), "logits"
    idx = H_.i64(g["idx"])
    idx_ref, w_ref = O.route(lg, shape, bias)
    H_.assert_equal("idx", idx, idx_ref)
    wg = host(g["w"])
    H_.assert_close("w", wg, w_ref, atol=1e-6, rtol=1e-5)
    m = O.permutation_maps(idx, shape)
    R = m["R"]
    for name in ("counts", "offsets", "row_of", "sel_offsets"):
        H_.assert_equal(name, H_.i64(g[name]), m[name])
    H_.assert_equal("token_of", H_.i64(g["token_of"])[:R], m["token_of"])
    H_.assert_equal("sel_tokens", H_.i64(g["sel_tokens"])[:T * k], m["sel_tokens"])
    cnt, off, rof = m["counts"], m["offsets"], m["row_of"]
    if shape is QWEN3:
        assert cnt.max() >= 8 * (T * k / E), "the Zipf bias should make hot experts"
    # ---- x_perm: sampled rows and padding rows
    rows = rng.choice(np.nonzero(H_.read_rows(m))[0], size=512, replace=False)
    tok_of = m["token_of"][rows]
    xp_rows = host(g["x_perm"][torch.as_tensor(rows, device="cuda")])
    ref_rows = np.zeros_like(xp_rows)
    ok = tok_of >= 0
    ref_rows[ok] = host(x_dev[torch.as_tensor(tok_of[ok], device="cuda")])
    H_.assert_equal("x_perm rows", xp_rows, ref_rows)
    # ---- per-group steps on sampled rows
    dY_dev = inp["dY"]
    dl_all = host(g["dlogits"])
    for gi in pick_groups(cnt, E, S, rng):
        n = int(cnt[gi])
        sel = np.sort(rng.choice(n, size=min(n, 48), replace=False)) + off[gi]
        rs = torch.as_tensor(sel, device="cuda")
        w13, w2 = (qt(a) for a in group_weights(inp, gi))
        xp = host(g["x_perm"][rs])
        GU = host(g["GU"][rs])
        hh = host(g["h"][rs])
        gu_ref, _ = O.expert_fc1(qr(xp), w13)
        H_.assert_close(f"GU g={gi}", GU, gu_ref)
        H_.assert_close(f"h g={gi}", hh, O.round_bf16(O.silu(GU[:, :F]) * GU[:, F:]))
        H_.assert_close(f"y g={gi}", host(g["y_perm"][rs]), O.expert_fc2(qr(hh), w2))
        dO = host(g["dO_perm"][rs])
        dGU = host(g["dGU"][rs])
        H_.assert_close(f"dGU g={gi}", dGU, O.expert_fc2_dgrad_swiglu(qr(dO), w2, GU))
        ref_dx = O.expert_fc1_dgrad(qr(dGU), w13, rounding=False)
        if gi < E:   # the row's router-logit gradient, added before the bf16 rounding
            ref_dx = ref_dx + dl_all[m["token_of"][sel], gi][:, None] * Wr[gi][None, :]
        H_.assert_close(f"dX g={gi}", host(g["dX_perm"][rs]), O.round_bf16(ref_dx))
        # weight gradients over all the group's rows, on sampled output rows
        allr = slice(int(off[gi]), int(off[gi]) + n)
        oh = rng.choice(Hd, size=32, replace=False)
        of = rng.choice(2 * F, size=32, replace=False)
        # (128x1 quantisation is per column, so sampling columns commutes with it)
        dO_all = qc(host(g["dO_perm"][allr][:, torch.as_tensor(oh, device="cuda")]))
        h_all = qc(host(g["h"][allr]))
        H_.assert_close(f"dW2 g={gi}", host(g["dW2"][gi][torch.as_tensor(oh, device="cuda")]),
                        O.wgrad(dO_all, h_all))
        dGU_all = qc(host(g["dGU"][allr][:, torch.as_tensor(of, device="cuda")]))
        xp_all = qc(host(g["x_perm"][allr]))
        H_.assert_close(f"dW13 g={gi}", host(g["dW13"][gi][torch.as_tensor(of, device="cuda")]),
                        O.wgrad(dGU_all, xp_all))
    # ---- combine and its backward on sampled tokens (GPU step inputs)
    ts = rng.choice(T, size=64, replace=False)
    yrows = {}
    for t in ts:
        acc = np.zeros(Hd)
        for j in range(k):
            r = rof[t, j]
            if r >= 0:
                yrows[r] = host(g["y_perm"][int(r)])
                acc += wg[t, j] * yrows[r]
        for s in range(S):
            acc += host(g["y_perm"][int(off[E + s] + t)])
        H_.assert_close(f"out[{t}]", host(g["out"][int(t)]), O.round_bf16(acc))
        dy = host(dY_dev[int(t)])
        for j in range(k):
            r = rof[t, j]
            if r < 0:
                continue
            H_.assert_close(f"dO[{t},{j}]", host(g["dO_perm"][int(r)]), O.round_bf16(wg[t, j] * dy))
            H_.assert_close(f"dw[{t},{j}]", host(g["dw"][int(t), j]), float(dy @ yrows[r]),
                            atol=1e-3, rtol=1e-3)
    dl = host(g["dlogits"])
    H_.assert_close("dlogits", dl, O.router_dlogits(shape, lg, idx, wg, host(g["dw"])),
                    atol=1e-4, rtol=1e-4)
    for t in ts[:16]:
        acc = np.zeros(Hd)
        for j in range(k):
            if rof[t, j] >= 0:        # kept rows already hold their router term
                acc += host(g["dX_perm"][int(rof[t, j])])
            else:                     # dropped by the capacity limit
                acc += dl[t, idx[t, j]] * Wr[idx[t, j]]
        for s in range(S):
            acc += host(g["dX_perm"][int(off[E + s] + t)])
        H_.assert_close(f"dx[{t}]", host(g["dx"][int(t)]), O.round_bf16(acc))
    for e in rng.choice(E, size=4, replace=False):
        st = m["sel_tokens"][m["sel_offsets"][e]:m["sel_offsets"][e + 1]]
        ref = dl[st, e] @ host(x_dev[torch.as_tensor(st, device="cuda")]) if st.size else np.zeros(Hd)
        H_.assert_close(f"dW_r[{e}]", host(g["dW_r"][int(e)]), ref, atol=1e-3, rtol=1e-4)
    # ---- end to end from raw inputs for a few tokens: out[t] and dx[t]
    e2e = {"out": ([], []), "dx": ([], [])}
    for t in ts[:4]:
        xt = host(x_dev[int(t):int(t) + 1])
        lt = O.router_logits(xt, Wr)
        it, wt = O.route(lg[t:t + 1], shape, bias)
        H_.assert_equal(f"idx e2e[{t}]", it[0], idx[t])
        dy = host(dY_dev[int(t)])
        acc = np.zeros(Hd)
        mag = np.zeros(Hd)
        dw_t = np.zeros(k)
        dXs = []
        for j in range(k):
            if rof[t, j] < 0:
                continue
            w13, w2 = (qt(a) for a in group_weights(inp, int(it[0, j])))
            gu, hh = O.expert_fc1(qr(xt), w13)
            y = O.expert_fc2(qr(hh), w2)
            acc += wt[0, j] * y[0]
            mag += np.abs(wt[0, j] * y[0])
            dw_t[j] = dy @ y[0]
            dO = O.round_bf16(wt[0, j] * dy[None, :])
            dG = O.expert_fc2_dgrad_swiglu(qr(dO), w2, gu)
            dXs.append(O.expert_fc1_dgrad(qr(dG), w13)[0])
        for s in range(S):
            w13, w2 = group_weights(inp, E + s)
            gu, hh = O.expert_fc1(xt, w13)
            ys = O.expert_fc2(hh, w2)[0]
            acc += ys
            mag += np.abs(ys)
            dXs.append(O.expert_fc1_dgrad(O.expert_fc2_dgrad_swiglu(dy[None, :], w2, gu), w13)[0])
        ref = O.round_bf16(acc)
        e2e["out"][0].append(host(g["out"][int(t)]))
        e2e["out"][1].append(ref)
        if fp8:
            H_.assert_close_fp8(f"out e2e[{t}]", host(g["out"][int(t)]), ref)
        else:
            H_.assert_close(f"out e2e[{t}]", host(g["out"][int(t)]), ref, scale=np.abs(ref) + mag)
        dlt = O.router_dlogits(shape, lt, it, wt, dw_t[None, :])
        router = dlt[0] @ Wr
        ref = O.round_bf16(sum(dXs) + router)
        mag = np.abs(ref) + sum(np.abs(d) for d in dXs) + np.abs(router)
        e2e["dx"][0].append(host(g["dx"][int(t)]))
        e2e["dx"][1].append(ref)
        if fp8:
            H_.assert_close_fp8(f"dx e2e[{t}]", host(g["dx"][int(t)]), ref)
        else:
            H_.assert_close(f"dx e2e[{t}]", host(g["dx"][int(t)]), ref, scale=mag)
    for name, (got, ref) in e2e.items():
        worst = H_.plain_rule(f"{shape.name} {name} (4 tokens)", np.stack(got), np.stack(ref),
                              fp8=fp8)
        if not fp8:
            assert worst <= H_.PLAIN_CAP, (name, worst)
    del g, inp
    torch.cuda.empty_cache()
