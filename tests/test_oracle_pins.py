"""Pins of the CPU oracle against things other than itself (CPU only).

Each test checks the oracle against a brute-force restatement in plain Python,
an independent library routine (torch), a closed form, or an invariant of the
MoE layer (per-expert counts sum to T*k; permute then unpermute with identity
experts returns sum_k w_k x; top-k equals a full sort; the grouped FFN equals
per-token dense products; gradients equal autograd and finite differences).
"""
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from workloads import GROUP_MAX, GROUP_TOP2_SUM, SIGMOID, SOFTMAX, TINY, MoEShape, make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


# --------------------------------------------------------------------------- #
# bf16 rounding against torch's own conversion
# --------------------------------------------------------------------------- #
def test_round_bf16_matches_torch_on_fp32_inputs():
    g = torch.Generator().manual_seed(1)
    v = torch.cat([
        torch.randn(200000, generator=g) * 10.0 ** torch.randint(-30, 30, (200000,), generator=g).float(),
        torch.tensor([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 3.4e38, 1e-40, -1e-40, 1e-45,
                      float("inf"), float("-inf")]),
    ])
    # exact halfway cases: 1 + 2^-8 (tie -> even 1), 1 + 3*2^-8 (tie -> up)
    v = torch.cat([v, torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130 * 1.5])])
    ref = v.to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(v.to(torch.float64).numpy())
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_ties_and_overflow():
    assert O.round_bf16(1 + 2 ** -8) == 1.0
    assert O.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6
    assert O.round_bf16(np.float64(3.4e38)) == np.inf
    assert np.isnan(O.round_bf16(np.nan))


# --------------------------------------------------------------------------- #
# stage 1: route
# --------------------------------------------------------------------------- #
def test_logits_brute_force():
    inp = make_inputs(TINY.with_(T=5, H=16, E=4), seed=3, weights=False, grad=False)
    x, W = f64(inp["x"]), f64(inp["W_r"])
    got = O.router_logits(x, W)
    for t in range(5):
        for e in range(4):
            s = 0.0
            for h in range(16):
                s += x[t, h] * W[e, h]
            assert got[t, e] == float(np.float32(s))


def _brute_topk(scores, k, allowed=None):
    # sort by (-score, expert); NaN ranks below every number
    cand = sorted(((-(s if not math.isnan(s) else -math.inf), e) for e, s in enumerate(scores)
                   if allowed is None or e in allowed))
    return [e for _, e in cand[:k]]


def _brute_route(l, cfg, bias):
    T, E = l.shape
    idx = np.zeros((T, cfg.k), dtype=np.int64)
    w = np.zeros((T, cfg.k))
    for t in range(T):
        if cfg.score_fn == SOFTMAX:
            sc = [float(np.float32(l[t, e]) + (np.float32(0) if bias is None else np.float32(bias[e])))
                  for e in range(E)]
            z = [l[t, e] + (0.0 if bias is None else float(np.float32(bias[e]))) for e in range(E)]
        else:
            s = [1.0 / (1.0 + math.exp(-l[t, e])) for e in range(E)]
            sc = [s[e] + (0.0 if bias is None else float(np.float32(bias[e]))) for e in range(E)]
        sc = [-math.inf if math.isnan(v) else v for v in sc]     # NaN ranks last
        allowed = None
        if cfg.n_groups > 1:
            per = E // cfg.n_groups
            gsc = []
            for gi in range(cfg.n_groups):
                mem = sorted(sc[gi * per:(gi + 1) * per], reverse=True)
                gsc.append(mem[0] + mem[1] if (cfg.group_score == GROUP_TOP2_SUM and per >= 2) else mem[0])
            keep = _brute_topk(gsc, cfg.topk_groups)
            allowed = {gi * per + i for gi in keep for i in range(per)}
        sel = _brute_topk(sc, cfg.k, allowed)
        idx[t] = sel
        if cfg.score_fn == SOFTMAX:
            m = z[sel[0]]
            ex = [math.exp(z[e] - m) for e in sel]
            w[t] = [v / sum(ex) for v in ex]
        else:
            ssum = sum(s[e] for e in sel)
            w[t] = [cfg.route_scale * s[e] / ssum for e in sel]
    return idx, w


@pytest.mark.parametrize("score_fn,groups,topg,gmode,bias", [
    (SOFTMAX, 1, 1, GROUP_TOP2_SUM, False),
    (SOFTMAX, 1, 1, GROUP_TOP2_SUM, True),
    (SIGMOID, 1, 1, GROUP_TOP2_SUM, True),
    (SIGMOID, 4, 2, GROUP_TOP2_SUM, True),
    (SIGMOID, 4, 2, GROUP_MAX, True),
    (SIGMOID, 8, 3, GROUP_TOP2_SUM, False),
])
def test_route_matches_brute_force_with_ties(score_fn, groups, topg, gmode, bias):
    E, k, T = 16, 3, 64
    cfg = MoEShape("t", T=T, H=8, E=E, k=k, F=8, score_fn=score_fn, n_groups=groups,
                   topk_groups=topg, group_score=gmode, route_scale=2.5 if score_fn == SIGMOID else 1.0)
    rng = np.random.default_rng(5)
    l = O.round_f32(rng.standard_normal((T, E)))
    # inject exact ties: copy columns, repeat values, a NaN
    l[:, 5] = l[:, 2]
    l[::3, 9] = l[::3, 1]
    l[7, :] = 0.25
    l[11, 4] = np.nan
    b = O.round_f32(rng.standard_normal(E) * 0.1) if bias else None
    idx, w = O.route(l, cfg, b)
    ridx, rw = _brute_route(l, cfg, b)
    np.testing.assert_array_equal(idx, ridx)
    ok = np.isfinite(rw).all(axis=1)
    np.testing.assert_allclose(w[ok], rw[ok], rtol=1e-12, atol=0)


def test_group_limited_with_one_group_is_plain_topk():
    cfg = MoEShape("t", T=40, H=8, E=12, k=4, F=8, score_fn=SIGMOID)
    rng = np.random.default_rng(0)
    l = O.round_f32(rng.standard_normal((40, 12)))
    a = O.route(l, cfg, None)
    b = O.route(l, cfg.with_(n_groups=1, topk_groups=1), None)
    np.testing.assert_array_equal(a[0], b[0])
    # G = E groups of one expert, keep k groups: also plain top-k
    c = O.route(l, cfg.with_(n_groups=12, topk_groups=4, group_score=GROUP_MAX), None)
    np.testing.assert_array_equal(a[0], c[0])


def test_softmax_weights_match_torch_softmax_and_sum_to_one():
    cfg = MoEShape("t", T=50, H=8, E=10, k=3, F=8)
    rng = np.random.default_rng(2)
    l = O.round_f32(rng.standard_normal((50, 10)) * 3)
    idx, w = O.route(l, cfg, None)
    ref = torch.softmax(torch.gather(torch.tensor(l), 1, torch.tensor(idx)), dim=1).numpy()
    np.testing.assert_allclose(w, ref, rtol=1e-13)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)
    cfg2 = cfg.with_(score_fn=SIGMOID, route_scale=1.7)
    _, w2 = O.route(l, cfg2, None)
    np.testing.assert_allclose(w2.sum(1), 1.7, rtol=1e-14)


@pytest.mark.parametrize("score_fn", [SOFTMAX, SIGMOID])
def test_route_replay_weights_match_torch_for_any_given_experts(score_fn):
    """Router Replay: the weights of recorded experts (here a seeded random
    choice of k distinct experts per token, in a random order, not the top-k)
    are torch's softmax over the chosen l + b, or route_scale * sigmoid / sum."""
    T, E, k = 40, 12, 4
    cfg = MoEShape("t", T=T, H=8, E=E, k=k, F=8, score_fn=score_fn, route_scale=2.5)
    rng = np.random.default_rng(5)
    l = O.round_f32(rng.standard_normal((T, E)) * 2)
    b = O.round_f32(0.1 * rng.standard_normal(E)).astype(np.float32)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    got_idx, w = O.route_replay(l, cfg, b, idx)
    np.testing.assert_array_equal(got_idx, idx)
    lt, it = torch.tensor(l), torch.tensor(idx)
    if score_fn == SOFTMAX:
        ref = torch.softmax(torch.gather(lt + torch.tensor(b, dtype=torch.float64), 1, it), dim=1)
    else:
        s = torch.gather(torch.sigmoid(lt), 1, it)
        ref = 2.5 * s / s.sum(dim=1, keepdim=True)
    np.testing.assert_allclose(w, ref.numpy(), rtol=1e-13)
    # replaying the router's own choice gives its own weights
    idx0, w0 = O.route(l, cfg, b)
    np.testing.assert_allclose(O.route_replay(l, cfg, b, idx0)[1], w0, rtol=0, atol=0)


# --------------------------------------------------------------------------- #
# load-balancing loss and bias update
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("score_fn", [SOFTMAX, SIGMOID])
def test_aux_loss_is_coeff_when_every_token_takes_every_expert(score_fn):
    """k = E: f_e = 1/E for every expert, so the loss is coeff * sum_e P_e,
    and the probabilities of a token sum to 1 over all experts (the sigmoid
    scores normalised over all E, not over the selected): loss = coeff for any
    logits."""
    T, E = 37, 6
    cfg = MoEShape("t", T=T, H=8, E=E, k=E, F=8, score_fn=score_fn)
    rng = np.random.default_rng(11)
    l = O.round_f32(rng.standard_normal((T, E)) * 3)
    b = O.round_f32(0.3 * rng.standard_normal(E)).astype(np.float32)
    idx = np.stack([rng.permutation(E) for _ in range(T)])
    loss, counts, P = O.aux_loss(l, cfg, b, idx, 0.125)
    np.testing.assert_array_equal(counts, np.full(E, T))
    assert abs(P.sum() - 1.0) < 1e-13
    assert abs(loss - 0.125) < 1e-13


def test_aux_loss_uniform_routing_and_full_imbalance():
    """Uniform probabilities and equal loads give coeff (the loss's minimum
    over loads for uniform P); every token sending all its weight and its one
    selection to expert 0 gives coeff * E (the maximum)."""
    T, E = 64, 8
    cfg = MoEShape("t", T=T, H=8, E=E, k=2, F=8)
    idx = np.stack([[t % E, (t + 1) % E] for t in range(T)])     # 16 selections each
    loss, counts, P = O.aux_loss(np.zeros((T, E)), cfg, None, idx, 0.01)
    np.testing.assert_array_equal(counts, np.full(E, 16))
    np.testing.assert_allclose(P, np.full(E, 1 / E), rtol=1e-15)
    assert abs(loss - 0.01) < 1e-15
    cfg1 = MoEShape("t", T=T, H=8, E=E, k=1, F=8)
    l = np.full((T, E), -800.0)
    l[:, 0] = 0.0                                   # softmax mass 1 (exp(-800) == 0)
    loss1, counts1, P1 = O.aux_loss(l, cfg1, None, np.zeros((T, 1), np.int64), 0.01)
    assert counts1[0] == T and counts1[1:].sum() == 0
    assert P1[0] == 1.0
    assert abs(loss1 - 0.01 * E) < 1e-15


def test_aux_loss_hand_computed_case():
    """T = 2, E = 3, k = 1, softmax, logits chosen so that the probabilities
    are exact fractions: token 0 (ln 1, ln 2, ln 1) -> (1/4, 1/2, 1/4), token 1
    (ln 3, ln 1, ln 0 -> -inf) -> (3/4, 1/4, 0). Selections 1 and 0:
    f = (1/2, 1/2, 0), P = (1/2, 3/8, 1/8), loss = c * 3 * (1/4 + 3/16)."""
    cfg = MoEShape("t", T=2, H=8, E=3, k=1, F=8)
    l = np.log(np.array([[1.0, 2.0, 1.0], [3.0, 1.0, 0.0]]))
    loss, counts, P = O.aux_loss(l, cfg, None, np.array([[1], [0]]), 2.0)
    np.testing.assert_array_equal(counts, [1, 1, 0])
    np.testing.assert_allclose(P, [0.5, 0.375, 0.125], rtol=1e-15)
    assert abs(loss - 2.0 * 3 * (0.25 + 0.1875)) < 1e-14


@pytest.mark.parametrize("score_fn", [SOFTMAX, SIGMOID])
def test_aux_loss_gradients_match_finite_differences(score_fn):
    """The logit gradient against central differences of aux_loss (counts
    follow idx, which is held fixed), and the x / W_r gradients against
    central differences of the loss of l = x W_r^T (no rounding)."""
    T, H, E, k = 9, 5, 7, 2
    cfg = MoEShape("t", T=T, H=H, E=E, k=k, F=8, score_fn=score_fn)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((T, H))
    W = rng.standard_normal((E, H)) * 0.7
    b = O.round_f32(0.2 * rng.standard_normal(E)).astype(np.float32)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    coeff, dloss = 0.3, 1.7
    L = lambda lg: dloss * O.aux_loss(lg, cfg, b, idx, coeff)[0]
    l = x @ W.T
    _, counts, _ = O.aux_loss(l, cfg, b, idx, coeff)
    dl = O.aux_loss_dlogits(l, cfg, b, counts, coeff, dloss)
    eps = 1e-6
    for t, e in [(0, 0), (3, 4), (8, 6), (5, 1)]:
        lp, lm = l.copy(), l.copy()
        lp[t, e] += eps
        lm[t, e] -= eps
        assert abs((L(lp) - L(lm)) / (2 * eps) - dl[t, e]) < 1e-8 * (1 + abs(dl[t, e]))
    dx0 = rng.standard_normal((T, H))
    dW0 = rng.standard_normal((E, H))
    _, dx, dW = O.aux_loss_backward(cfg, x, W, l, b, counts, coeff, dloss, dx0, dW0,
                                    rounding=False)
    for t, h in [(0, 0), (4, 3), (8, 4)]:
        xp, xm = x.copy(), x.copy()
        xp[t, h] += eps
        xm[t, h] -= eps
        fd = (L(xp @ W.T) - L(xm @ W.T)) / (2 * eps)
        assert abs(dx[t, h] - dx0[t, h] - fd) < 1e-8 * (1 + abs(fd))
    for e, h in [(0, 1), (6, 4), (3, 0)]:
        Wp, Wm = W.copy(), W.copy()
        Wp[e, h] += eps
        Wm[e, h] -= eps
        fd = (L(x @ Wp.T) - L(x @ Wm.T)) / (2 * eps)
        assert abs(dW[e, h] - dW0[e, h] - fd) < 1e-8 * (1 + abs(fd))


def test_aux_loss_dlogits_sum_to_zero_per_token_for_softmax():
    """Softmax probabilities sum to 1 whatever the logits, so shifting all of
    a token's logits by a constant changes nothing: each row of the softmax
    gradient sums to 0 (a dropped centring term would break it)."""
    T, E = 20, 16
    cfg = MoEShape("t", T=T, H=8, E=E, k=4, F=8)
    rng = np.random.default_rng(8)
    l = rng.standard_normal((T, E))
    counts = rng.integers(0, 10, E)
    dl = O.aux_loss_dlogits(l, cfg, None, counts, 0.1, 1.0)
    np.testing.assert_allclose(dl.sum(axis=1), 0.0, atol=1e-17)
    assert np.abs(dl).max() > 1e-6


def test_bias_update_moves_towards_the_mean_load():
    """T k / E = 4 * 2 / 4 = 2: loads (3, 2, 1, 2) move the biases by (-r, 0,
    +r, 0), in fp32; no bias counts as zeros."""
    cfg = MoEShape("t", T=4, H=8, E=4, k=2, F=8)
    b = np.array([0.5, -0.25, 1e-3, 0.0], np.float32)
    out = O.bias_update(b, [3, 2, 1, 2], cfg, 1e-3)
    assert out.dtype == np.float32
    np.testing.assert_array_equal(
        out, np.array([np.float32(0.5) - np.float32(1e-3), -0.25,
                       np.float32(1e-3) + np.float32(1e-3), 0.0], np.float32))
    np.testing.assert_array_equal(O.bias_update(None, [0, 4, 4, 0], cfg, 0.5),
                                  np.array([0.5, -0.5, -0.5, 0.5], np.float32))


# --------------------------------------------------------------------------- #
# stage 2: dispatch maps
# --------------------------------------------------------------------------- #
def _brute_maps(idx, cfg):
    T, k = idx.shape
    C = O.capacity(cfg)
    items = sorted((int(idx[t, j]), t, j) for t in range(T) for j in range(k))
    row_of = -np.ones((T, k), dtype=np.int64)
    off = 0
    offsets = []
    for e in range(cfg.E):
        offsets.append(off)
        mine = [(t, j) for (ee, t, j) in items if ee == e]
        kept = mine[:C] if C else mine
        for r, (t, j) in enumerate(kept):
            row_of[t, j] = off + r
        seg = C if C else int(math.ceil(len(kept) / cfg.row_align) * cfg.row_align)
        off += seg
    return row_of, offsets


@pytest.mark.parametrize("E,k,align,cf,shared", [(8, 2, 1, 0.0, 0), (8, 2, 128, 0.0, 1),
                                                  (16, 4, 8, 0.0, 0), (16, 4, 8, 1.0, 0),
                                                  (5, 5, 4, 0.0, 2), (64, 1, 16, 1.25, 0)])
def test_maps_invariants_and_brute_force(E, k, align, cf, shared):
    T = 97
    cfg = MoEShape("t", T=T, H=8, E=E, k=k, F=8, row_align=align, capacity_factor=cf, n_shared=shared)
    rng = np.random.default_rng(E * 7 + k)
    # skewed routing: distinct experts per token drawn with a hot head
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.2
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
    m = O.permutation_maps(idx, cfg)
    rrow, roff = _brute_maps(idx, cfg)
    np.testing.assert_array_equal(m["row_of"], rrow)
    np.testing.assert_array_equal(m["offsets"][:E], roff)
    kept = m["row_of"] >= 0
    # P1: kept counts sum to the kept assignments (= T*k when dropless)
    assert m["counts"][:E].sum() == kept.sum()
    if cf == 0:
        assert kept.all() and m["counts"][:E].sum() == T * k
    # every kept assignment has its own row, token_of inverts row_of
    rows = m["row_of"][kept]
    assert len(set(rows.tolist())) == rows.size
    tt = np.nonzero(kept)[0]
    np.testing.assert_array_equal(m["token_of"][rows], tt)
    # segments aligned, rows increase with t inside an expert
    assert (m["offsets"] % align == 0).all()
    for e in range(E):
        seg = m["token_of"][m["offsets"][e]:m["offsets"][e] + m["counts"][e]]
        assert (np.diff(seg) > 0).all()
        assert (m["token_of"][m["offsets"][e] + m["counts"][e]:m["offsets"][e + 1]] == -1).all()
    for s in range(shared):
        o = m["offsets"][E + s]
        np.testing.assert_array_equal(m["token_of"][o:o + T], np.arange(T))
    # selection lists hold every selecting token in token order
    for e in range(E):
        st = m["sel_tokens"][m["sel_offsets"][e]:m["sel_offsets"][e + 1]]
        np.testing.assert_array_equal(st, np.nonzero((idx == e).any(1))[0])


def _gemm_row_tiles(m):
    """128-row tiles the row-grouped GEMMs run: ceil(count / 128) per group."""
    return sum(-(-int(c) // 128) for c in m["counts"])


@pytest.mark.parametrize("E,k,cf,shared,T", [(16, 4, 0.0, 1, 700), (8, 2, 1.0, 0, 900),
                                              (64, 1, 1.25, 0, 1500), (5, 5, 0.0, 2, 97)])
def test_stash_page_table_covers_exactly_the_kept_rows(E, k, cf, shared, T):
    """Paged stash: every kept row (and every row of its 128-row block, which the
    GEMM tiles read) gets a pool row of its own inside the pages the layer took;
    the layer takes as many pages as the grouped GEMMs run 128-row tiles."""
    cfg = MoEShape("t", T=T, H=8, E=E, k=k, F=8, row_align=128, capacity_factor=cf,
                   n_shared=shared)
    rng = np.random.default_rng(T + E)
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.5
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
    m = O.permutation_maps(idx, cfg)
    rows_max = int(m["R"])
    n_tiles = _gemm_row_tiles(m)
    top = 3
    P = top + n_tiles + 5
    table, top_after, full = O.stash_page_table(m["counts"], m["offsets"], rows_max, P, top)
    assert not full and top_after == top + n_tiles
    assert table.shape == (rows_max // 128 + 2,) and table[-1] == top
    read = np.zeros(rows_max, dtype=bool)        # rows the GEMM tiles read (brute force)
    for g in range(len(m["counts"])):
        for r in range(int(m["counts"][g])):
            rr = int(m["offsets"][g]) + r
            read[rr - rr % 128: rr - rr % 128 + 128] = True
    rows = np.nonzero(read)[0]
    phys = table[rows // 128] * 128 + rows % 128
    assert len(set(phys.tolist())) == rows.size                 # no two rows share a pool row
    assert phys.min() >= top * 128 and phys.max() < top_after * 128
    assert rows.size == n_tiles * 128                           # and no page is left unused
    # every other block (and the one past the last row) is the spill page
    other = np.setdiff1d(np.arange(rows_max // 128 + 1), np.unique(rows // 128))
    assert (table[other] == P).all()
    # pages follow the block order (stable in the rows' order)
    assert (np.diff(table[np.unique(rows // 128)]) == 1).all()


def test_stash_page_table_dropless_is_the_contiguous_layout():
    """Dropless segments are padded to 128 rows, so every block below offsets[G]
    is live and the table is the identity shifted by the first page."""
    cfg = MoEShape("t", T=300, H=8, E=8, k=2, F=8)
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(8, size=2, replace=False) for _ in range(300)])
    m = O.permutation_maps(idx, cfg)
    used = int(m["offsets"][-1]) // 128
    table, top_after, full = O.stash_page_table(m["counts"], m["offsets"], int(m["R"]) + 1024,
                                                1000, 17)
    np.testing.assert_array_equal(table[:used], 17 + np.arange(used))
    assert top_after == 17 + used and not full


def test_stash_page_table_full_pool_and_stacked_layers():
    counts = np.array([130, 0, 1, 256])
    offsets = np.array([0, 256, 256, 384, 640])
    need = 2 + 0 + 1 + 2
    t, top, full = O.stash_page_table(counts, offsets, 640, need - 1, 0)
    assert full and top == 0 and (t[:-1] == need - 1).all() and t[-1] == 0
    t, top, full = O.stash_page_table(counts, offsets, 640, need, 0)
    assert not full and top == need
    # blocks 0, 1 (group 0), 2 (group 2; group 1 is empty), 3, 4 (group 3); block 5
    # is the one past the last row
    np.testing.assert_array_equal(t, [0, 1, 2, 3, 4, need, 0])
    # a second layer on the same pool takes the pages after the first's
    t2, top2, full2 = O.stash_page_table(counts, offsets, 640, 2 * need, top)
    assert not full2 and top2 == 2 * need and t2[-1] == need
    np.testing.assert_array_equal(t2[:5], need + np.arange(need))


def test_capacity_value_and_keep_first_tokens():
    cfg = MoEShape("t", T=16384, H=8, E=256, k=8, F=8, capacity_factor=1.25)
    assert O.capacity(cfg) == 640
    cfg = MoEShape("t", T=10, H=8, E=2, k=1, F=8, capacity_factor=0.5, row_align=1)
    idx = np.zeros((10, 1), dtype=np.int64)
    idx[7:] = 1
    m = O.permutation_maps(idx, cfg)
    assert O.capacity(cfg) == 3
    np.testing.assert_array_equal(m["row_of"][:, 0], [0, 1, 2, -1, -1, -1, -1, 3, 4, 5])


def test_identity_experts_round_trip():
    """P3: permute, identity experts, unpermute: out = bf16(sum_j w_j x) = x."""
    cfg = MoEShape("t", T=64, H=32, E=8, k=3, F=8)
    inp = make_inputs(cfg, seed=4, weights=False, grad=False)
    x = f64(inp["x"])
    idx, w = O.route(O.router_logits(x, f64(inp["W_r"])), cfg, None)
    m = O.permutation_maps(idx, cfg)
    xp = O.permute(x, m)
    out = np.zeros_like(x)
    for t in range(64):
        out[t] = sum(w[t, j] * xp[m["row_of"][t, j]] for j in range(3))
    np.testing.assert_array_equal(O.round_bf16(out), x)
    cfg2 = cfg.with_(score_fn=SIGMOID, route_scale=0.5)
    idx2, w2 = O.route(O.router_logits(x, f64(inp["W_r"])), cfg2, None)
    m2 = O.permutation_maps(idx2, cfg2)
    xp2 = O.permute(x, m2)
    out2 = np.stack([sum(w2[t, j] * xp2[m2["row_of"][t, j]] for j in range(3)) for t in range(64)])
    np.testing.assert_allclose(out2, 0.5 * x, rtol=1e-14)


# --------------------------------------------------------------------------- #
# stage 3 / whole layer
# --------------------------------------------------------------------------- #
def _torch_bf16(a):
    return a.to(torch.bfloat16).to(torch.float64)


def test_single_expert_layer_is_dense_swiglu_mlp():
    """P4: E=1, k=1 reduces the layer to one dense SwiGLU MLP (torch fp64)."""
    cfg = MoEShape("t", T=48, H=64, E=1, k=1, F=96)
    inp = make_inputs(cfg, seed=9)
    fwd = O.layer_forward(cfg, f64(inp["x"]), f64(inp["W_r"]), None, f64(inp["W13"]), f64(inp["W2"]))
    x = inp["x"].double()
    W13, W2 = inp["W13"][0].double(), inp["W2"][0].double()
    gu = _torch_bf16(x @ W13.T)
    h = _torch_bf16(torch.nn.functional.silu(gu[:, :96]) * gu[:, 96:])
    y = _torch_bf16(h @ W2.T)
    np.testing.assert_allclose(fwd["out"], y.numpy(), rtol=2 ** -7, atol=1e-6)
    assert np.mean(fwd["out"] == y.numpy()) > 0.99
    np.testing.assert_allclose(fwd["w"], 1.0)


def test_grouped_ffn_equals_per_token_products_and_is_equivariant():
    """P5: batched expert FFN = one row at a time; permuting tokens permutes out."""
    cfg = MoEShape("t", T=40, H=32, E=4, k=2, F=48)
    inp = make_inputs(cfg, seed=11)
    x, Wr, W13, W2 = (f64(inp[n]) for n in ("x", "W_r", "W13", "W2"))
    fwd = O.layer_forward(cfg, x, Wr, None, W13, W2)
    for t in range(0, 40, 7):
        for j in range(2):
            e = fwd["idx"][t, j]
            g = np.array([sum(x[t, hh] * W13[e, n, hh] for hh in range(32)) for n in range(96)])
            np.testing.assert_allclose(fwd["GU"][t, j], O.round_bf16(g), rtol=2 ** -7)
    perm = np.random.default_rng(0).permutation(40)
    fwd2 = O.layer_forward(cfg, x[perm], Wr, None, W13, W2)
    np.testing.assert_allclose(fwd2["out"], fwd["out"][perm], rtol=2 ** -7, atol=1e-6)
    np.testing.assert_array_equal(fwd2["idx"], fwd["idx"][perm])


def test_capacity_to_infinity_is_dropless():
    """P7: with an unreachable capacity nothing drops and values equal dropless."""
    cfg = MoEShape("t", T=32, H=32, E=4, k=2, F=32)
    inp = make_inputs(cfg, seed=12)
    args = [f64(inp[n]) for n in ("x", "W_r")] + [None] + [f64(inp[n]) for n in ("W13", "W2")]
    a = O.layer_forward(cfg, *args)
    b = O.layer_forward(cfg.with_(capacity_factor=100.0), *args)
    assert (b["maps"]["row_of"] >= 0).all()
    np.testing.assert_array_equal(a["out"], b["out"])


def _torch_layer(cfg, x, Wr, bias, W13, W2, idx, kept):
    T, H = x.shape
    l = x @ Wr.T
    it = torch.tensor(idx)
    if cfg.score_fn == SOFTMAX:
        z = l + (0.0 if bias is None else torch.tensor(bias, dtype=torch.float64))
        w = torch.softmax(torch.gather(z, 1, it), dim=1)
    else:
        s = torch.sigmoid(torch.gather(l, 1, it))
        w = cfg.route_scale * s / s.sum(1, keepdim=True)
    F = cfg.F
    outs = []
    for t in range(T):
        acc = torch.zeros(H, dtype=torch.float64)
        for j in range(cfg.k):
            if not kept[t, j]:
                continue
            e = int(idx[t, j])
            gu = W13[e] @ x[t]
            hh = torch.nn.functional.silu(gu[:F]) * gu[F:]
            acc = acc + w[t, j] * (W2[e] @ hh)
        for s_ in range(cfg.n_shared):
            gu = W13[cfg.E + s_] @ x[t]
            hh = torch.nn.functional.silu(gu[:F]) * gu[F:]
            acc = acc + W2[cfg.E + s_] @ hh
        outs.append(acc)
    return torch.stack(outs)


@pytest.mark.parametrize("cfg", [
    MoEShape("t", T=8, H=16, E=4, k=2, F=32, bias_kind="zipf"),
    MoEShape("t", T=8, H=16, E=8, k=3, F=16, n_shared=1, score_fn=SIGMOID, n_groups=4,
             topk_groups=2, bias_kind="normal", route_scale=1.5),
    MoEShape("t", T=12, H=16, E=4, k=2, F=16, capacity_factor=0.5, row_align=1,
             score_fn=SIGMOID, bias_kind="normal"),
])
def test_backward_equals_autograd_and_finite_differences(cfg):
    """P6: the oracle's backward (no rounding) = torch autograd = central FD."""
    inp = make_inputs(cfg, seed=21)
    x, Wr, W13, W2, dY = (f64(inp[n]) for n in ("x", "W_r", "W13", "W2", "dY"))
    W13 = W13 * 10.0          # make the FFN non-trivial at this size
    W2 = W2 * 10.0
    bias = None if inp["bias"] is None else f64(inp["bias"])
    fwd = O.layer_forward(cfg, x, Wr, bias, W13, W2, rounding=False)
    bwd = O.layer_backward(cfg, x, Wr, W13, W2, fwd, dY, rounding=False)
    kept = fwd["maps"]["row_of"] >= 0
    if cfg.capacity_factor > 0:
        assert (~kept).any()
    tx, tWr, tW13, tW2 = (torch.tensor(a, requires_grad=True) for a in (x, Wr, W13, W2))
    out = _torch_layer(cfg, tx, tWr, bias, tW13, tW2, fwd["idx"], kept)
    np.testing.assert_allclose(fwd["out"], out.detach().numpy(), rtol=1e-12, atol=1e-12)
    (out * torch.tensor(dY)).sum().backward()
    for name, t in (("dx", tx), ("dW_r", tWr), ("dW13", tW13), ("dW2", tW2)):
        np.testing.assert_allclose(bwd[name], t.grad.numpy(), rtol=1e-9, atol=1e-10, err_msg=name)
    # central finite differences on a few coordinates
    def loss(xx, wr, w13, w2):
        f = O.layer_forward(cfg, xx, wr, bias, w13, w2, rounding=False)
        np.testing.assert_array_equal(f["idx"], fwd["idx"])
        return float((f["out"] * dY).sum())
    eps = 1e-6
    for (arr_i, pos, gname) in ((0, (3, 5), "dx"), (1, (2, 7), "dW_r"), (2, (1, 3, 4), "dW13"),
                                (3, (0, 2, 1), "dW2")):
        args = [x.copy(), Wr.copy(), W13.copy(), W2.copy()]
        args[arr_i][pos] += eps
        lp = loss(*args)
        args[arr_i][pos] -= 2 * eps
        lm = loss(*args)
        fd = (lp - lm) / (2 * eps)
        assert abs(fd - bwd[gname][pos]) <= 1e-5 * (1 + abs(fd)), (gname, fd, bwd[gname][pos])


def test_softmax_jacobian_rows_sum_to_zero():
    cfg = MoEShape("t", T=30, H=8, E=6, k=3, F=8)
    rng = np.random.default_rng(3)
    l = rng.standard_normal((30, 6))
    idx, w = O.route(l, cfg, None)
    dl = O.router_dlogits(cfg, l, idx, w, rng.standard_normal((30, 3)))
    np.testing.assert_allclose(dl.sum(1), 0.0, atol=1e-14)
    assert (np.count_nonzero(dl, axis=1) <= 3).all()


# --------------------------------------------------------------------------- #
# FP8 (E4M3, power-of-two block scales)
# --------------------------------------------------------------------------- #
def test_round_e4m3_matches_torch_float8_in_range():
    g = torch.Generator().manual_seed(7)
    v = torch.randn(200000, generator=g) * 2.0 ** torch.randint(-12, 9, (200000,), generator=g).float()
    grid = torch.arange(0, 256, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    grid = grid[torch.isfinite(grid)]
    v = torch.cat([v, grid, -grid, torch.tensor([1 + 1 / 16, 1 + 3 / 16, 2.0 ** -10, 3 * 2.0 ** -10])])
    v = v[v.abs() <= 448]
    ref = v.to(torch.float8_e4m3fn).float().double().numpy()
    got = O.round_e4m3(v.double().numpy())
    np.testing.assert_array_equal(got, ref)


def test_round_e4m3_saturates_and_scale_closed_form():
    np.testing.assert_array_equal(O.round_e4m3([1000.0, -1e6, 448.0, 460.0]), [448, -448, 448, 448])
    amax = np.abs(np.random.default_rng(1).standard_normal(5000)) * 10.0 ** np.random.default_rng(2).integers(-8, 8, 5000)
    s = O.e4m3_scale(amax)
    k = np.log2(s)
    np.testing.assert_array_equal(k, np.round(k))              # powers of two
    r = amax / s
    assert (r > 224).all() and (r <= 448).all()                 # smallest power >= amax/448
    assert O.e4m3_scale(0.0) == 1.0
    assert O.e4m3_scale(448.0 * 2 ** -5) == 2 ** -5


def test_block_quantisers_structure():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((256, 384)) * np.repeat(10.0 ** rng.integers(-3, 3, (256, 3)), 128, axis=1)
    Q = O.quant_rows(X)
    np.testing.assert_array_equal(O.quant_rows(Q), Q)           # idempotent
    for blk in range(3):                                        # each block scaled on its own
        Bq, B = Q[:, blk * 128:(blk + 1) * 128], X[:, blk * 128:(blk + 1) * 128]
        s = O.e4m3_scale(np.abs(B).max(axis=1, keepdims=True))
        np.testing.assert_array_equal(Bq, O.round_e4m3(B / s) * s)
    np.testing.assert_array_equal(O.quant_cols(X.T).T, O.quant_rows(X))  # columns = rows of X^T
    # values already on the grid with block max 448*2^k are left unchanged
    G = O.round_e4m3(rng.uniform(-448, 448, (4, 128)))
    G[:, 0] = 448.0
    np.testing.assert_array_equal(O.quant_rows(G * 2.0 ** 5), G * 2.0 ** 5)
    # short last block of quant_cols uses its own rows
    C = rng.standard_normal((200, 8))
    C[150:] *= 1000
    Qc = O.quant_cols(C)
    s = O.e4m3_scale(np.abs(C[128:]).max(axis=0, keepdims=True))
    np.testing.assert_array_equal(Qc[128:], O.round_e4m3(C[128:] / s) * s)


def test_quant_tiles_brute_force():
    rng = np.random.default_rng(4)
    W = rng.standard_normal((256, 384)) * 0.02
    W[:128, 128:256] *= 50
    got = O.quant_tiles(W)
    for i in range(2):
        for j in range(3):
            B = W[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            amax = max(abs(float(v)) for v in B.ravel())
            k = math.ceil(math.log2(amax / 448.0))
            s = 2.0 ** k
            np.testing.assert_array_equal(got[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128],
                                          O.round_e4m3(B / s) * s)


def _torch_fq(t, dims):
    """Fake-quantise with torch's own float8 conversion; `dims` = block reduce dims."""
    amax = t.abs().amax(dim=dims, keepdim=True)
    k = torch.ceil(torch.log2(amax / 448.0))
    s = torch.where(amax > 0, torch.exp2(k), torch.ones_like(amax))
    return (t / s).to(torch.float8_e4m3fn).double() * s


def test_fp8_single_expert_layer_is_dense_fp8_mlp():
    cfg = MoEShape("t", T=256, H=256, E=1, k=1, F=256, dtype=1)
    inp = make_inputs(cfg, seed=13)
    x, Wr, W13, W2, dY = (f64(inp[n]) for n in ("x", "W_r", "W13", "W2", "dY"))
    fwd = O.layer_forward_fp8(cfg, x, Wr, None, W13, W2)
    bwd = O.layer_backward_fp8(cfg, x, Wr, W13, W2, fwd, dY)
    tx, t13, t2, tdY = (torch.tensor(a) for a in (x, W13[0], W2[0], dY))
    rows = lambda t: _torch_fq(t.view(t.shape[0], -1, 128), (2,)).view(t.shape)  # noqa: E731
    tiles = lambda t: _torch_fq(t.view(t.shape[0] // 128, 128, t.shape[1] // 128, 128), (1, 3)).reshape(t.shape)  # noqa: E731
    cols = lambda t: rows(t.T.contiguous()).T  # noqa: E731
    q13, q2 = tiles(t13), tiles(t2)
    gu = _torch_bf16(rows(tx) @ q13.T)
    h = _torch_bf16(torch.nn.functional.silu(gu[:, :256]) * gu[:, 256:])
    y = _torch_bf16(rows(h) @ q2.T)
    np.testing.assert_allclose(fwd["out"], y.numpy(), rtol=2 ** -7, atol=1e-6)
    dO = tdY                                             # weight 1
    dh = rows(dO) @ q2
    G, U = gu[:, :256], gu[:, 256:]
    sg = torch.sigmoid(G)
    dGU = _torch_bf16(torch.cat([dh * U * sg * (1 + G * (1 - sg)), dh * G * sg], dim=1))
    dX = _torch_bf16(rows(dGU) @ q13)
    np.testing.assert_allclose(bwd["dGU"][:, 0], dGU.numpy(), rtol=2 ** -6, atol=1e-5)
    np.testing.assert_allclose(bwd["dX"][:, 0], dX.numpy(), rtol=2 ** -6, atol=1e-4)
    dW2 = _torch_bf16(cols(dO).T @ cols(h))
    dW13 = _torch_bf16(cols(dGU).T @ cols(tx))
    np.testing.assert_allclose(bwd["dW2"][0], dW2.numpy(), rtol=2 ** -6, atol=1e-4)
    np.testing.assert_allclose(bwd["dW13"][0], dW13.numpy(), rtol=2 ** -6, atol=1e-4)


def test_mx_weight_forms_and_reduction_to_the_block_recipe():
    """MXFP8: the forward form quantises 1x32 along a weight's input dimension,
    the data-gradient form 32x1 along its output dimension (= 1x32 rows of the
    transpose); where every 32-long row and column piece of a 128x128 tile holds
    the tile's largest magnitude, both equal the 128x128 tile quantisation."""
    rng = np.random.default_rng(21)
    W = rng.standard_normal((256, 384)) * 0.02
    mx = MoEShape("t", T=1, H=384, E=1, k=1, F=128, dtype=O.DT_MXFP8)
    blk = MoEShape("t", T=1, H=384, E=1, k=1, F=128, dtype=O.DT_FP8_BLOCK)
    assert O.fp8_block(mx) == 32 and O.fp8_block(blk) == 128
    f, d = O.fp8_weights(mx, W)
    np.testing.assert_array_equal(f, O.quant_rows(W, 32))
    np.testing.assert_array_equal(d, O.quant_rows(W.T, 32).T)
    for r in range(0, 256, 32):                      # each 1x32 piece on its own
        s = O.e4m3_scale(np.abs(W[r, 64:96]).max())
        np.testing.assert_array_equal(f[r, 64:96], O.round_e4m3(W[r, 64:96] / s) * s)
    # the tile maximum in every 32-long piece: i % 32 == j % 32 inside each tile
    M = np.abs(W).max() * 3.0
    ii, jj = np.meshgrid(np.arange(256), np.arange(384), indexing="ij")
    W2 = np.where(ii % 32 == jj % 32, np.where((ii + jj) % 2 == 0, M, -M), W)
    f2, d2 = O.fp8_weights(mx, W2)
    t2, t2d = O.fp8_weights(blk, W2)
    np.testing.assert_array_equal(t2, t2d)
    np.testing.assert_array_equal(f2, t2)
    np.testing.assert_array_equal(d2, t2)


def test_mxfp8_single_expert_layer_is_dense_mx_mlp():
    """One expert, every token routed to it with weight 1: each stage of the
    MXFP8 layer is the dense SwiGLU MLP's on operands fake-quantised with
    torch's float8 in 32-long pieces along the GEMM's reduced dimension
    (weights: along H for FC1 and F for FC2, along 2F and H for the data
    gradients; tokens for the weight gradients). Each stage starts from the
    oracle's own bf16 inputs to it, so a one-ulp difference upstream cannot move
    a block scale downstream."""
    cfg = MoEShape("t", T=256, H=256, E=1, k=1, F=256, dtype=O.DT_MXFP8)
    inp = make_inputs(cfg, seed=17)
    x, Wr, W13, W2, dY = (f64(inp[n]) for n in ("x", "W_r", "W13", "W2", "dY"))
    # weight columns (input dimension) of magnitudes 2^0..2^7 inside every 32-long
    # piece, so the 1x32 (forward) and 32x1 (data-gradient) forms differ widely
    W13 = W13 * 2.0 ** (np.arange(256) % 8)[None, None, :]
    W2 = W2 * 2.0 ** (np.arange(256) % 8)[None, None, :]
    fwd = O.layer_forward_fp8(cfg, x, Wr, None, W13, W2)
    bwd = O.layer_backward_fp8(cfg, x, Wr, W13, W2, fwd, dY)
    T_ = lambda a: torch.tensor(np.asarray(a, np.float64))  # noqa: E731
    tx, t13, t2, dO = T_(x), T_(W13[0]), T_(W2[0]), T_(dY)   # weight 1: dO = dY
    rows = lambda t: _torch_fq(t.view(t.shape[0], -1, 32), (2,)).view(t.shape)  # noqa: E731
    cols = lambda t: rows(t.T.contiguous()).T  # noqa: E731
    GU, h, dGU = T_(fwd["GU"][:, 0]), T_(fwd["h"][:, 0]), T_(bwd["dGU"][:, 0])
    close = lambda got, ref, rt: np.testing.assert_allclose(got, ref.numpy(), rtol=rt, atol=1e-6)  # noqa: E731
    close(fwd["GU"][:, 0], _torch_bf16(rows(tx) @ rows(t13).T), 2 ** -7)
    close(fwd["h"][:, 0], _torch_bf16(torch.nn.functional.silu(GU[:, :256]) * GU[:, 256:]), 2 ** -7)
    close(fwd["out"], _torch_bf16(rows(h) @ rows(t2).T), 2 ** -7)
    dh = rows(dO) @ cols(t2)
    G, U = GU[:, :256], GU[:, 256:]
    sg = torch.sigmoid(G)
    close(bwd["dGU"][:, 0], _torch_bf16(torch.cat([dh * U * sg * (1 + G * (1 - sg)), dh * G * sg],
                                                  dim=1)), 2 ** -7)
    close(bwd["dX"][:, 0], _torch_bf16(rows(dGU) @ cols(t13)), 2 ** -7)
    close(bwd["dW2"][0], _torch_bf16(cols(dO).T @ cols(h)), 2 ** -7)
    close(bwd["dW13"][0], _torch_bf16(cols(dGU).T @ cols(tx)), 2 ** -7)
    # not the block recipe: the 1x32 pieces give a different (finer) result
    blk = O.layer_forward_fp8(cfg.with_(dtype=O.DT_FP8_BLOCK), x, Wr, None, W13, W2)
    assert not np.array_equal(blk["out"], fwd["out"])


# --------------------------------------------------------------------------- #
# the routing weight inside the expert (algebraic reordering)
# --------------------------------------------------------------------------- #
REORDER_CFGS = [
    MoEShape("t", T=8, H=16, E=4, k=2, F=32, bias_kind="zipf"),
    MoEShape("t", T=8, H=16, E=8, k=3, F=16, n_shared=1, score_fn=SIGMOID, n_groups=4,
             topk_groups=2, bias_kind="normal", route_scale=1.5),
    MoEShape("t", T=12, H=16, E=4, k=2, F=16, capacity_factor=0.5, row_align=1,
             score_fn=SIGMOID, bias_kind="normal"),
]


def _reorder_inputs(cfg, seed):
    inp = make_inputs(cfg, seed=seed)
    x, Wr, W13, W2, dY = (f64(inp[n]) for n in ("x", "W_r", "W13", "W2", "dY"))
    bias = None if inp["bias"] is None else f64(inp["bias"])
    return x, Wr, bias, W13 * 10.0, W2 * 10.0, dY


@pytest.mark.parametrize("cfg", REORDER_CFGS)
def test_reordered_layer_equals_the_layer_without_rounding(cfg):
    """w (h W2^T) = (w h) W2^T and <dY, h W2^T> = <dY W2, h>: without rounding
    the reordered forward and backward give the layer's own results."""
    x, Wr, bias, W13, W2, dY = _reorder_inputs(cfg, 31)
    a = O.layer_forward(cfg, x, Wr, bias, W13, W2, rounding=False)
    b = O.layer_forward_reordered(cfg, x, Wr, bias, W13, W2, rounding=False)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-12, atol=1e-13)
    ga = O.layer_backward(cfg, x, Wr, W13, W2, a, dY, rounding=False)
    gb = O.layer_backward_reordered(cfg, x, Wr, W13, W2, b, dY, rounding=False)
    np.testing.assert_allclose(gb["dw"], ga["dw"], rtol=1e-11, atol=1e-12)
    for n in ("dlogits", "dx", "dW_r", "dW13", "dW2"):
        np.testing.assert_allclose(gb[n], ga[n], rtol=1e-10, atol=1e-11, err_msg=n)


@pytest.mark.parametrize("cfg", REORDER_CFGS)
def test_reordered_backward_matches_finite_differences(cfg):
    x, Wr, bias, W13, W2, dY = _reorder_inputs(cfg, 32)
    fwd = O.layer_forward_reordered(cfg, x, Wr, bias, W13, W2, rounding=False)
    bwd = O.layer_backward_reordered(cfg, x, Wr, W13, W2, fwd, dY, rounding=False)

    def loss(xx, wr, w13, w2):
        f = O.layer_forward_reordered(cfg, xx, wr, bias, w13, w2, rounding=False)
        np.testing.assert_array_equal(f["idx"], fwd["idx"])
        return float((f["out"] * dY).sum())
    eps = 1e-6
    for (arr_i, pos, gname) in ((0, (3, 5), "dx"), (1, (2, 7), "dW_r"), (2, (1, 3, 4), "dW13"),
                                (3, (0, 2, 1), "dW2"), (0, (6, 11), "dx")):
        args = [x.copy(), Wr.copy(), W13.copy(), W2.copy()]
        args[arr_i][pos] += eps
        lp = loss(*args)
        args[arr_i][pos] -= 2 * eps
        lm = loss(*args)
        fd = (lp - lm) / (2 * eps)
        assert abs(fd - bwd[gname][pos]) <= 1e-5 * (1 + abs(fd)), (gname, fd, bwd[gname][pos])


def test_reordered_layer_with_rounding_stays_within_bf16_of_the_layer():
    """With bf16 rounding the two orders differ only where the roundings fall
    (h_s rounded after the weighting instead of y before it): a few bf16 ulps
    of the results' magnitudes."""
    cfg = MoEShape("t", T=64, H=64, E=8, k=2, F=64, score_fn=SIGMOID, bias_kind="normal")
    inp = make_inputs(cfg, seed=33)
    x, Wr, W13, W2, dY = (f64(inp[n]) for n in ("x", "W_r", "W13", "W2", "dY"))
    bias = f64(inp["bias"])
    a = O.layer_forward(cfg, x, Wr, bias, W13, W2)
    b = O.layer_forward_reordered(cfg, x, Wr, bias, W13, W2)
    scale = np.abs(a["out"]).max()
    assert np.abs(b["out"] - a["out"]).max() <= 4 * 2.0 ** -8 * scale
    assert (b["out"] != a["out"]).any()        # the rounding points really moved
    ga = O.layer_backward(cfg, x, Wr, W13, W2, a, dY)
    gb = O.layer_backward_reordered(cfg, x, Wr, W13, W2, b, dY)
    for n in ("dx", "dW13", "dW2"):
        assert np.abs(gb[n] - ga[n]).max() <= 4 * 2.0 ** -8 * np.abs(ga[n]).max(), n
