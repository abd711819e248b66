"""Plain CPU oracle of one Mixture-of-Experts layer, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports, links or runs this
module; only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` do. It shares no code with the CUDA path.

What it computes follows "Scalable Training of Mixture-of-Experts Models with
Megatron Core" (gist.science summaries, es: "Resumen técnico" §2.1, "Arquitectura
de la Capa MoE"): the layer is four stages in sequence --

  1. Route    -- a router assigns every token to its k best experts;
  2. Dispatch -- tokens are moved to the experts they were assigned to (on one
                 GPU this is a permutation into per-expert contiguous rows);
  3. Compute  -- every expert runs its FFN on its tokens (grouped GEMM);
  4. Combine  -- the inverse movement; results are summed with router weights.

The router stays in fp32 (same page, §2.4: router kept in high precision).
Everything the pages leave open is taken from the layer configuration and the
readings listed below; every one of them is a reading, not a quote:

  * logits l = x . W_r^T, accumulated in fp64, rounded once to fp32;
  * softmax router: selection on the fp32 value l + b (b = optional logit bias),
    ties to the lower expert index; weights = softmax over the k selected
    (renormalised top-k probabilities);
  * sigmoid router: s = sigmoid(l) in fp64, selection score s + b in fp64;
    group-limited: groups of E/G contiguous experts scored by the sum of their
    two best selection scores (or their maximum), the best topk_groups groups
    kept (ties to the lower group), then top-k inside them; weights
    route_scale * s_j / sum_sel s (bias only steers selection);
  * Router Replay (the summary's RL support, es "Soporte para RL"): the
    experts come from a recorded idx [T,k] instead of the top-k, the weights
    are the router's for those experts, in that order, from the current logits;
  * load-balancing loss (the pages fuse "aux-loss" computation with routing,
    es §2.3.C, without a formula): coeff * E * sum_e f_e P_e, f_e the share of
    the T k selections that went to e, P_e the mean over tokens of the
    router's probability of e over all experts (softmax of l + b, or the
    sigmoid scores normalised over all experts); its gradient flows into x
    and W_r through the logits. The bias update: a sign step of the selection
    bias towards the mean load (not in the pages; see bias_update);
  * capacity C = ceil(cf * T * k / E) rounded up to row_align; an expert keeps
    its first C tokens in token order, dropped assignments contribute 0 and
    the surviving weights are not renormalised;
  * permutation: stable counting sort by (expert, token); each expert's segment
    is padded to a multiple of row_align rows (padding rows are zero); shared
    experts follow the routed segments, one row per token in token order;
  * SwiGLU expert: W13[e] = [gate rows ; up rows] ([2F,H]), W2[e] is [H,F];
    G,U = X W_gate^T, X W_up^T rounded to bf16, h = bf16(silu(G) * U),
    y = bf16(h W2^T);
  * combine: out[t] = bf16(sum_j w_tj y_tj + sum_s y_shared[s,t]);
  * backward: the exact gradient of that function with the same bf16
    materialisation points (dO, dGU, dX, dx, dW13, dW2 in bf16; dlogits, dW_r
    in fp32); the router gradient flows into x and W_r.

FP8 (the FP8 configuration): E4M3 values with power-of-two block scales
(reading of the pages' MXFP8 recipe for Blackwell, es summary §2.4:
scale = 2^ceil(log2(amax/448)), 1 for an all-zero block); activations take
1x128 blocks along the reduction dimension of the GEMM that consumes them,
expert weights 128x128 blocks, weight-gradient operands 128x1 blocks along
the tokens of each expert (quantised from the bf16 tensors). The MXFP8
configuration uses 32-element blocks instead (the MX formats' block length)
for the activations (1x32) and the weight-gradient operands (32x1), and
quantises each expert weight twice: 1x32 along its input dimension for the
forward GEMM, 32x1 along its output dimension for the data gradient (the
dimension each GEMM reduces). Quantised values are exact in bf16 and in fp64,
so the GEMMs below multiply them exactly.

Rounding: ``round_bf16`` is round-to-nearest-even onto the bf16 grid, written
from the format (8 exponent bits, 7 stored fraction bits). Pass
``rounding=False`` to the layer functions for exact fp64 arithmetic (used by
the finite-difference pins).
"""
from __future__ import annotations

import math

import numpy as np

SOFTMAX = 0
SIGMOID = 1
GROUP_TOP2_SUM = 0
GROUP_MAX = 1

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
_BF16_MIN_QUANTUM_EXP = -133          # 2^(-126 - 7): the subnormal spacing


# --------------------------------------------------------------------------- #
# number formats
# --------------------------------------------------------------------------- #
def round_bf16(a) -> np.ndarray:
    """Round to the nearest bf16 value, ties to even; returns float64.

    bf16 keeps 8 significant bits: for |a| in [2^e, 2^(e+1)) the spacing is
    2^(e-7), never below the subnormal spacing 2^-133. Values whose rounded
    magnitude exceeds the largest finite bf16 become +-inf.
    """
    a = np.asarray(a, dtype=np.float64)
    out = np.array(a, copy=True)
    fin = np.isfinite(a) & (a != 0)
    if np.any(fin):
        v = a[fin]
        _, ex = np.frexp(v)                  # v = m * 2^ex, 0.5 <= |m| < 1
        qexp = np.maximum(ex - 1 - 7, _BF16_MIN_QUANTUM_EXP)
        r = np.ldexp(np.rint(np.ldexp(v, -qexp)), qexp)
        r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, v), r)
        out[fin] = r
    return out


E4M3_MAX = 448.0
_E4M3_MIN_QUANTUM_EXP = -9            # 2^(-6 - 3): the subnormal spacing


def round_e4m3(a) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to even, saturating at +-448.

    E4M3 keeps 4 significant bits: for |a| in [2^e, 2^(e+1)) the spacing is
    2^(e-3), never below the subnormal spacing 2^-9; the largest finite value
    is 1.75 * 2^8 = 448 (the format has no infinities).
    """
    a = np.asarray(a, dtype=np.float64)
    out = np.array(a, copy=True)
    fin = np.isfinite(a) & (a != 0)
    if np.any(fin):
        v = a[fin]
        _, ex = np.frexp(v)
        qexp = np.maximum(ex - 1 - 3, _E4M3_MIN_QUANTUM_EXP)
        r = np.ldexp(np.rint(np.ldexp(v, -qexp)), qexp)
        out[fin] = np.clip(r, -E4M3_MAX, E4M3_MAX)
    return out


def e4m3_scale(amax) -> np.ndarray:
    """Power-of-two block scale 2^ceil(log2(amax/448)); 1 where amax == 0."""
    amax = np.asarray(amax, dtype=np.float64)
    m, ex = np.frexp(amax / E4M3_MAX)             # amax/448 = m * 2^ex, 0.5 <= m < 1
    k = np.where(m == 0.5, ex - 1, ex)            # ceil(log2(.))
    return np.where(amax > 0, np.ldexp(1.0, k), 1.0)


def quant_rows(X, block: int = 128) -> np.ndarray:
    """Dequantised E4M3 values of X with one scale per 1 x `block` slice of a row."""
    X = np.asarray(X, np.float64)
    n, c = X.shape
    Xb = X.reshape(n, c // block, block)
    s = e4m3_scale(np.abs(Xb).max(axis=2, keepdims=True))
    return (round_e4m3(Xb / s) * s).reshape(n, c)


def quant_cols(X, block: int = 128) -> np.ndarray:
    """One scale per `block` x 1 slice of a column (consecutive rows; a short
    last block is scaled by its own rows)."""
    X = np.asarray(X, np.float64)
    out = np.empty_like(X)
    for r0 in range(0, X.shape[0], block):
        B = X[r0:r0 + block]
        s = e4m3_scale(np.abs(B).max(axis=0, keepdims=True))
        out[r0:r0 + block] = round_e4m3(B / s) * s
    return out


def quant_tiles(W, block: int = 128) -> np.ndarray:
    """One scale per `block` x `block` tile of a matrix."""
    W = np.asarray(W, np.float64)
    r, c = W.shape
    Wb = W.reshape(r // block, block, c // block, block)
    s = e4m3_scale(np.abs(Wb).max(axis=(1, 3), keepdims=True))
    return (round_e4m3(Wb / s) * s).reshape(r, c)


def round_f32(a) -> np.ndarray:
    """Round to the nearest fp32 value (IEEE cast); returns float64."""
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def _rb(a, rounding: bool):
    return round_bf16(a) if rounding else np.asarray(a, dtype=np.float64)


def _rf(a, rounding: bool):
    return round_f32(a) if rounding else np.asarray(a, dtype=np.float64)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z / (1.0 + np.exp(-z))


# --------------------------------------------------------------------------- #
# stage 1: route
# --------------------------------------------------------------------------- #
def router_logits(x, W_r, rounding: bool = True) -> np.ndarray:
    """l[t,e] = sum_h x[t,h] W_r[e,h], fp64 accumulation, one fp32 rounding."""
    x = np.asarray(x, dtype=np.float64)
    W_r = np.asarray(W_r, dtype=np.float64)
    return _rf(x @ W_r.T, rounding)


def _topk_rows(score, k, masked=None):
    """Per row: the k columns with the largest score, ties to the lower column.

    NaN scores rank below every number; masked columns rank below everything.
    """
    score = np.where(np.isnan(score), -np.inf, score)
    n, m = score.shape
    col = np.broadcast_to(np.arange(m), (n, m))
    msk = np.zeros((n, m), dtype=np.int8) if masked is None else masked.astype(np.int8)
    # lexsort: last key is primary -> (masked asc, -score asc, column asc)
    order = np.lexsort((col, -score, msk), axis=-1)
    return order[:, :k]


def capacity(cfg) -> int:
    """Rows each expert keeps in capacity mode; 0 means dropless."""
    if cfg.capacity_factor <= 0:
        return 0
    cf = float(np.float32(cfg.capacity_factor))
    c = math.ceil(cf * cfg.T * cfg.k / cfg.E)
    a = cfg.row_align
    return (c + a - 1) // a * a


def route(logits, cfg, bias=None):
    """Top-k selection and routing weights from fp32 logits.

    Returns (idx [T,k] int64, w [T,k] float64). Follows the route stage of the
    Megatron Core MoE layer (es summary, Resumen técnico §2.1, step 1: a router
    assigns each token to its k best experts).
    """
    l = np.asarray(logits, dtype=np.float64)
    T, E = l.shape
    k = cfg.k
    if cfg.score_fn == SOFTMAX:
        # selection on the fp32 sum l + b (bit-reproducible)
        l32 = l.astype(np.float32)
        if bias is not None:
            l32 = l32 + np.asarray(bias, dtype=np.float32)[None, :]
        sc = l32.astype(np.float64)
        masked = None
        if cfg.n_groups > 1:
            masked = _group_mask(sc, cfg)
        idx = _topk_rows(sc, k, masked)
        return idx, route_weights(l, cfg, bias, idx)
    if cfg.score_fn == SIGMOID:
        s = sigmoid(l)
        sc = s + (0.0 if bias is None else np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :])
        masked = _group_mask(sc, cfg) if cfg.n_groups > 1 else None
        idx = _topk_rows(sc, k, masked)
        return idx, route_weights(l, cfg, bias, idx)
    raise ValueError("score_fn")


def route_weights(logits, cfg, bias, idx):
    """Routing weights of the experts idx [T,k] (in that order) from fp32 logits.

    Softmax router: the softmax over the k chosen experts of l + b (fp64, from
    the fp32-valued logits and bias). Sigmoid router: route_scale * s_j / sum
    of s over the chosen, s = sigmoid(l) unbiased (the bias only selects).
    """
    l = np.asarray(logits, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    if cfg.score_fn == SOFTMAX:
        b64 = 0.0 if bias is None else np.asarray(bias, np.float32).astype(np.float64)[None, :]
        sel = np.take_along_axis(l + b64, idx, axis=1)
        z = np.exp(sel - sel[:, :1])
        return z / z.sum(axis=1, keepdims=True)
    if cfg.score_fn == SIGMOID:
        ssel = np.take_along_axis(sigmoid(l), idx, axis=1)
        return cfg.route_scale * ssel / ssel.sum(axis=1, keepdims=True)
    raise ValueError("score_fn")


def route_replay(logits, cfg, bias, idx):
    """Router Replay: the layer routes every token to the given experts idx
    [T,k] (decisions recorded earlier, e.g. by inference) instead of its own
    top-k; the weights are the router's, from the current logits, for those
    experts in that order. Follows the RL support of the Megatron Core MoE
    summary (es summary, Resumen técnico §2, "Soporte para RL": routing
    decisions of inference replayed in training)."""
    idx = np.asarray(idx, dtype=np.int64)
    return idx, route_weights(logits, cfg, bias, idx)


# --------------------------------------------------------------------------- #
# load-balancing auxiliary loss and the bias update
# --------------------------------------------------------------------------- #
def aux_probs(logits, cfg, bias=None):
    """Router probability of every expert [T,E] for the load-balancing loss.

    Softmax router: the softmax over all E experts of l + b. Sigmoid router:
    s_e / sum over all E of s, s = sigmoid(l) (unbiased). Each row sums to 1.
    """
    l = np.asarray(logits, dtype=np.float64)
    if cfg.score_fn == SOFTMAX:
        b64 = 0.0 if bias is None else np.asarray(bias, np.float32).astype(np.float64)[None, :]
        z = l + b64
        z = np.exp(z - z.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    if cfg.score_fn == SIGMOID:
        s = sigmoid(l)
        return s / s.sum(axis=1, keepdims=True)
    raise ValueError("score_fn")


def aux_loss(logits, cfg, bias, idx, coeff):
    """Load-balancing auxiliary loss of one batch (reading of the loss whose
    computation the pages fuse with routing and permutation, es summary
    §2.3.C "Fusión de Kernels"; the pages give no formula, so this is the
    switch-style balance loss):

      counts[e] = tokens that selected e (the router's top-k, before any
                  capacity drop),
      f_e = counts[e] / (T k),  P_e = mean over tokens of aux_probs[t, e],
      loss = coeff * E * sum_e f_e P_e.

    Returns (loss, counts [E] int64, P [E]). An empty batch gives 0, 0, 0.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, E, k = cfg.T, cfg.E, cfg.k
    counts = np.bincount(idx.reshape(-1), minlength=E)[:E].astype(np.int64)
    if T == 0:
        return 0.0, counts, np.zeros(E)
    P = aux_probs(logits, cfg, bias).mean(axis=0)
    f = counts / float(T * k)
    return float(coeff * E * np.sum(f * P)), counts, P


def aux_loss_dlogits(logits, cfg, bias, counts, coeff, dloss):
    """dloss times the gradient of aux_loss w.r.t. the logits [T,E] (counts
    are piecewise constant in the logits and carry none).

    With g_e = coeff E counts[e] / (T^2 k) = d loss / d p[t,e]:
      softmax: dl[t,e] = p[t,e] (g_e - sum_j p[t,j] g_j);
      sigmoid: p = s / S, so dl[t,e] = s_e (1 - s_e) / S (g_e - sum_j p[t,j] g_j).
    """
    l = np.asarray(logits, dtype=np.float64)
    T, E, k = cfg.T, cfg.E, cfg.k
    if T == 0:
        return np.zeros((0, E))
    g = coeff * E * np.asarray(counts, np.float64) / (float(T) * T * k)
    p = aux_probs(l, cfg, bias)
    centred = g[None, :] - (p * g[None, :]).sum(axis=1, keepdims=True)
    if cfg.score_fn == SOFTMAX:
        return dloss * p * centred
    s = sigmoid(l)
    return dloss * s * (1.0 - s) / s.sum(axis=1, keepdims=True) * centred


def aux_loss_backward(cfg, x, W_r, logits, bias, counts, coeff, dloss, dx, dW_r,
                      rounding: bool = True):
    """The loss's gradient added to the layer's input and router-weight
    gradients: dl = aux_loss_dlogits(...); dx' = bf16(dx + dl W_r) and
    dW_r' = fp32(dW_r + dl^T x) (l = x W_r^T). Returns (dl, dx', dW_r')."""
    dl = aux_loss_dlogits(logits, cfg, bias, counts, coeff, dloss)
    x = np.asarray(x, np.float64)
    W_r = np.asarray(W_r, np.float64)
    dx_new = _rb(np.asarray(dx, np.float64) + dl @ W_r, rounding)
    dW_new = _rf(np.asarray(dW_r, np.float64) + dl.T @ x, rounding)
    return dl, dx_new, dW_new


def bias_update(bias, counts, cfg, rate):
    """Auxiliary-loss-free balancing step on the per-expert selection bias.

    The pages do not describe it; it is the plain sign rule that keeps the
    selection bias of the sigmoid router with bias (the DeepSeek-V3-style
    configuration) balanced: every expert above the mean load T k / E moves
    its bias down by `rate`, every expert below it up by `rate`, an expert
    exactly at the mean keeps it. fp32, as stored."""
    b = np.zeros(cfg.E, np.float32) if bias is None else np.asarray(bias, np.float32)
    c = np.asarray(counts, np.int64)
    sign = np.sign(cfg.T * cfg.k - cfg.E * c).astype(np.float32)
    return (b + np.float32(rate) * sign).astype(np.float32)


def _group_mask(sc, cfg):
    """Mask (True = excluded) of experts outside the best topk_groups groups."""
    T, E = sc.shape
    G = cfg.n_groups
    per = E // G
    s = np.where(np.isnan(sc), -np.inf, sc).reshape(T, G, per)
    srt = -np.sort(-s, axis=2)                     # descending within group
    if cfg.group_score == GROUP_TOP2_SUM and per >= 2:
        gs = srt[:, :, 0] + srt[:, :, 1]
    else:
        gs = srt[:, :, 0]
    keep = _topk_rows(gs, cfg.topk_groups)         # [T, topk_groups]
    gmask = np.ones((T, G), dtype=bool)
    np.put_along_axis(gmask, keep, False, axis=1)
    return np.repeat(gmask, per, axis=1)


# --------------------------------------------------------------------------- #
# stage 2: dispatch (permutation maps)
# --------------------------------------------------------------------------- #
def permutation_maps(idx, cfg) -> dict:
    """Stable counting sort of the (token, slot) assignments by (expert, token).

    counts[g]      rows kept by group g (routed experts, then shared experts)
    offsets[g]     first row of group g's segment (segments padded to row_align,
                   or C rows each in capacity mode); offsets[G] = rows used
    row_of[t,j]    row of assignment (t,j), -1 if dropped by capacity
    token_of[r]    token held by row r, -1 for padding rows
    sel_offsets[e] / sel_tokens: for every routed expert, all tokens that
                   selected it (dropped or not) in increasing token order
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    E, S, a = cfg.E, cfg.n_shared, cfg.row_align
    C = capacity(cfg)
    total = np.zeros(E, dtype=np.int64)
    rank = np.zeros((T, k), dtype=np.int64)
    for t in range(T):                               # running counter per expert
        for j in range(k):
            e = int(idx[t, j])
            rank[t, j] = total[e]
            total[e] += 1
    kept = np.minimum(total, C) if C > 0 else total.copy()
    seglen = np.empty(E + S, dtype=np.int64)
    for e in range(E):
        seglen[e] = C if C > 0 else (kept[e] + a - 1) // a * a
    for s in range(S):
        seglen[E + s] = (T + a - 1) // a * a
    offsets = np.zeros(E + S + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(seglen)
    counts = np.concatenate([kept, np.full(S, T, dtype=np.int64)])
    R = int(offsets[-1])
    row_of = np.full((T, k), -1, dtype=np.int64)
    token_of = np.full(R, -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if C > 0 and rank[t, j] >= C:
                continue
            r = int(offsets[e] + rank[t, j])
            row_of[t, j] = r
            token_of[r] = t
    for s in range(S):
        token_of[offsets[E + s]: offsets[E + s] + T] = np.arange(T)
    sel_offsets = np.zeros(E + 1, dtype=np.int64)
    sel_offsets[1:] = np.cumsum(total)
    sel_tokens = np.empty(T * k, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            sel_tokens[sel_offsets[e] + rank[t, j]] = t
    return dict(counts=counts, offsets=offsets, row_of=row_of, token_of=token_of,
                sel_offsets=sel_offsets, sel_tokens=sel_tokens, R=R, C=C)


def stash_page_table(counts, offsets, rows_max: int, pool_pages: int, top: int):
    """Page table of one layer's paged stash.

    Reading of the pages' paged stashing (es summary, Resumen técnico §2.3.C:
    the dynamic buffers are managed inside the CUDA graph so that none is
    reserved for the worst case): the rows a layer keeps for its backward live
    in a pool of `pool_pages` pages of 128 rows, plus a spill page numbered
    `pool_pages`. The layer takes one page for every 128-row block of its
    permuted rows that holds a kept row -- the first ceil(counts[g] / 128)
    blocks of group g's segment, which starts at row offsets[g] -- numbered
    consecutively from `top` in block order. Every other block, and the block
    just past the last row, maps to the spill page. A layer whose blocks do not
    all fit takes no page: every block maps to the spill page and the pool is
    reported full.

    Returns (table, top_after, full): table has rows_max // 128 + 2 entries,
    table[b] the page of block b for b <= rows_max // 128 and table[-1] the
    first page taken (= top).
    """
    nblk = rows_max // 128
    live = []
    for g in range(len(counts)):
        first = int(offsets[g]) // 128
        for i in range((int(counts[g]) + 127) // 128):
            live.append(first + i)
    table = np.full(nblk + 2, pool_pages, dtype=np.int64)
    table[-1] = top
    if top + len(live) > pool_pages:
        return table, top, True
    for n, b in enumerate(live):
        table[b] = top + n
    return table, top + len(live), False


def permute(x, maps) -> np.ndarray:
    """x_perm[r] = x[token_of[r]], zero rows for padding."""
    x = np.asarray(x, dtype=np.float64)
    tok = maps["token_of"]
    out = np.zeros((tok.shape[0], x.shape[1]))
    valid = tok >= 0
    out[valid] = x[tok[valid]]
    return out


# --------------------------------------------------------------------------- #
# stage 3: compute (one SwiGLU expert)
# --------------------------------------------------------------------------- #
def expert_fc1(X, W13_e, rounding: bool = True):
    """GU = bf16(X W13_e^T) ([n,2F]: gate columns then up) and h = bf16(silu(G) U)."""
    F = W13_e.shape[0] // 2
    GU = _rb(np.asarray(X, np.float64) @ np.asarray(W13_e, np.float64).T, rounding)
    h = _rb(silu(GU[:, :F]) * GU[:, F:], rounding)
    return GU, h


def expert_fc2(h, W2_e, rounding: bool = True):
    """y = bf16(h W2_e^T)."""
    return _rb(np.asarray(h, np.float64) @ np.asarray(W2_e, np.float64).T, rounding)


def expert_fc2_dgrad_swiglu(dO, W2_e, GU, rounding: bool = True):
    """dh = dO W2_e (kept in full precision), then the SwiGLU backward.

    dG = dh * U * sig(G) * (1 + G (1 - sig(G))), dU = dh * silu(G); both bf16.
    """
    F = W2_e.shape[1]
    dh = np.asarray(dO, np.float64) @ np.asarray(W2_e, np.float64)
    G, U = GU[:, :F], GU[:, F:]
    sg = sigmoid(G)
    dG = dh * U * sg * (1.0 + G * (1.0 - sg))
    dU = dh * silu(G)
    return _rb(np.concatenate([dG, dU], axis=1), rounding)


def expert_fc1_dgrad(dGU, W13_e, rounding: bool = True):
    """dX = bf16(dGU W13_e)."""
    return _rb(np.asarray(dGU, np.float64) @ np.asarray(W13_e, np.float64), rounding)


def wgrad(A, B, rounding: bool = True):
    """dW = bf16(A^T B): the weight gradient summed over an expert's rows."""
    return _rb(np.asarray(A, np.float64).T @ np.asarray(B, np.float64), rounding)


# --------------------------------------------------------------------------- #
# the whole layer, token by token (the plain definition)
# --------------------------------------------------------------------------- #
def layer_forward(cfg, x, W_r, bias, W13, W2, logits=None, rounding: bool = True):
    """One MoE layer forward; returns a dict of every intermediate.

    out[t] = sum over kept slots j of w_tj * FFN_{e_tj}(x_t), plus every shared
    expert's FFN(x_t) with weight 1. Per-assignment values are stored per
    (t, j) so that they can be compared against any row layout.
    """
    x = np.asarray(x, np.float64)
    T, H = x.shape
    E, k, F, S = cfg.E, cfg.k, cfg.F, cfg.n_shared
    if logits is None:
        logits = router_logits(x, W_r, rounding)
    logits = np.asarray(logits, np.float64)
    idx, w = route(logits, cfg, bias)
    maps = permutation_maps(idx, cfg)
    kept = maps["row_of"] >= 0
    GU = np.zeros((T, k, 2 * F))
    h = np.zeros((T, k, F))
    y = np.zeros((T, k, H))
    for e in range(E):
        tt, jj = np.nonzero((idx == e) & kept)
        if tt.size == 0:
            continue
        g, hh = expert_fc1(x[tt], W13[e], rounding)
        GU[tt, jj], h[tt, jj] = g, hh
        y[tt, jj] = expert_fc2(hh, W2[e], rounding)
    GU_s = np.zeros((S, T, 2 * F))
    h_s = np.zeros((S, T, F))
    y_s = np.zeros((S, T, H))
    for s in range(S):
        GU_s[s], h_s[s] = expert_fc1(x, W13[E + s], rounding)
        y_s[s] = expert_fc2(h_s[s], W2[E + s], rounding)
    acc = np.einsum("tj,tjh->th", np.where(kept, w, 0.0), y) + y_s.sum(axis=0)
    out = _rb(acc, rounding)
    return dict(logits=logits, idx=idx, w=w, maps=maps, GU=GU, h=h, y=y,
                GU_s=GU_s, h_s=h_s, y_s=y_s, out=out)


def router_dlogits(cfg, logits, idx, w, dw):
    """Gradient of the routing weights w.r.t. the fp32 logits (dense [T,E]).

    softmax renormalised top-k: dl_{e_j} = w_j (dw_j - sum_i w_i dw_i);
    sigmoid normalised: ds_i = (r/S)(dw_i - sum_j (s_j/S) dw_j) on the selected
    experts, dl_i = ds_i s_i (1 - s_i); every other entry is 0 (selection,
    grouping and biases carry no gradient).
    """
    logits = np.asarray(logits, np.float64)
    T, E = logits.shape
    dl = np.zeros((T, E))
    if cfg.score_fn == SOFTMAX:
        inner = (w * dw).sum(axis=1, keepdims=True)
        vals = w * (dw - inner)
    else:
        s = sigmoid(np.take_along_axis(logits, idx, axis=1))
        Ssum = s.sum(axis=1, keepdims=True)
        r = cfg.route_scale
        ds = (r / Ssum) * (dw - ((s / Ssum) * dw).sum(axis=1, keepdims=True))
        vals = ds * s * (1.0 - s)
    np.put_along_axis(dl, idx, vals, axis=1)
    return dl


def layer_backward(cfg, x, W_r, W13, W2, fwd, dY, rounding: bool = True):
    """Gradient of sum(out * dY) w.r.t. x, W_r, W13, W2, with the layer's
    bf16 materialisation points. Returns a dict of every intermediate."""
    x = np.asarray(x, np.float64)
    dY = np.asarray(dY, np.float64)
    T, H = x.shape
    E, k, F, S = cfg.E, cfg.k, cfg.F, cfg.n_shared
    idx, w, maps = fwd["idx"], fwd["w"], fwd["maps"]
    kept = maps["row_of"] >= 0
    # combine backward
    dO = _rb(np.where(kept, w, 0.0)[:, :, None] * dY[:, None, :], rounding)
    dw = np.where(kept, np.einsum("th,tjh->tj", dY, fwd["y"]), 0.0)
    dGU = np.zeros((T, k, 2 * F))
    dX = np.zeros((T, k, H))
    dW13 = np.zeros((E + S, 2 * F, H))
    dW2 = np.zeros((E + S, H, F))
    for e in range(E):
        tt, jj = np.nonzero((idx == e) & kept)
        if tt.size == 0:
            dW13[e] = 0.0
            dW2[e] = 0.0
            continue
        d = expert_fc2_dgrad_swiglu(dO[tt, jj], W2[e], fwd["GU"][tt, jj], rounding)
        dGU[tt, jj] = d
        dX[tt, jj] = expert_fc1_dgrad(d, W13[e], rounding)
        dW2[e] = wgrad(dO[tt, jj], fwd["h"][tt, jj], rounding)
        dW13[e] = wgrad(d, x[tt], rounding)
    dGU_s = np.zeros((S, T, 2 * F))
    dX_s = np.zeros((S, T, H))
    dYb = _rb(dY, rounding)
    for s in range(S):
        dGU_s[s] = expert_fc2_dgrad_swiglu(dYb, W2[E + s], fwd["GU_s"][s], rounding)
        dX_s[s] = expert_fc1_dgrad(dGU_s[s], W13[E + s], rounding)
        dW2[E + s] = wgrad(dYb, fwd["h_s"][s], rounding)
        dW13[E + s] = wgrad(dGU_s[s], x, rounding)
    dlogits = router_dlogits(cfg, fwd["logits"], idx, w, dw)
    dx_router = dlogits @ np.asarray(W_r, np.float64)
    dx = _rb(dX.sum(axis=1) + dX_s.sum(axis=0) + dx_router, rounding)
    dW_r = _rf(dlogits.T @ x, rounding)
    return dict(dO=dO, dw=dw, dGU=dGU, dX=dX, dGU_s=dGU_s, dX_s=dX_s,
                dlogits=dlogits, dx=dx, dW_r=dW_r, dW13=dW13, dW2=dW2)


def to_rows(per_slot, per_shared, maps, cfg, width):
    """Place per-(t,j) and per-shared-expert values at their permuted rows."""
    R = maps["R"]
    out = np.zeros((R, width))
    r = maps["row_of"]
    ok = r >= 0
    out[r[ok]] = per_slot[ok]
    T = r.shape[0]
    for s in range(cfg.n_shared):
        o = maps["offsets"][cfg.E + s]
        out[o:o + T] = per_shared[s]
    return out


# --------------------------------------------------------------------------- #
# the layer with the routing weight inside the expert
# --------------------------------------------------------------------------- #
def layer_forward_reordered(cfg, x, W_r, bias, W13, W2, logits=None, rounding: bool = True):
    """The layer with the routing weight moved into the expert, before FC2.

    "Scalable Training of Mixture-of-Experts Models with Megatron Core" (es
    summary, Resumen técnico §2.3.A, memory: an algebraic reordering of the
    routing weights so the permuted expert outputs need not be kept for the
    backward). Since y = h W2^T is linear in h, w y = (w h) W2^T: each
    assignment's expert scales its own SwiGLU output,
        h_s = bf16(w_tj silu(G) U),   y_s = bf16(h_s W2^T),
    and the combine is an unweighted sum, out[t] = bf16(sum_j y_s + shared).
    Shared experts have weight 1 (h_s = h). Without rounding this is
    layer_forward exactly; with rounding only the bf16 rounding points move.
    """
    x = np.asarray(x, np.float64)
    T, H = x.shape
    E, k, F, S = cfg.E, cfg.k, cfg.F, cfg.n_shared
    if logits is None:
        logits = router_logits(x, W_r, rounding)
    logits = np.asarray(logits, np.float64)
    idx, w = route(logits, cfg, bias)
    maps = permutation_maps(idx, cfg)
    kept = maps["row_of"] >= 0
    GU = np.zeros((T, k, 2 * F))
    hs = np.zeros((T, k, F))
    y = np.zeros((T, k, H))
    for e in range(E):
        tt, jj = np.nonzero((idx == e) & kept)
        if tt.size == 0:
            continue
        g = _rb(x[tt] @ np.asarray(W13[e], np.float64).T, rounding)
        GU[tt, jj] = g
        hs[tt, jj] = _rb(w[tt, jj][:, None] * silu(g[:, :F]) * g[:, F:], rounding)
        y[tt, jj] = expert_fc2(hs[tt, jj], W2[e], rounding)
    GU_s = np.zeros((S, T, 2 * F))
    h_s = np.zeros((S, T, F))
    y_s = np.zeros((S, T, H))
    for s in range(S):
        GU_s[s], h_s[s] = expert_fc1(x, W13[E + s], rounding)
        y_s[s] = expert_fc2(h_s[s], W2[E + s], rounding)
    acc = np.where(kept[:, :, None], y, 0.0).sum(axis=1) + y_s.sum(axis=0)
    return dict(logits=logits, idx=idx, w=w, maps=maps, GU=GU, hs=hs, y=y, GU_s=GU_s,
                h_s=h_s, y_s=y_s, out=_rb(acc, rounding))


def expert_fc2_dgrad_swiglu_weighted(dY, W2_e, GU, w, rounding: bool = True):
    """The FC2 data gradient of one expert with the routing weight inside it:
    dh_s = dY W2_e (full precision), dw = <dh_s, silu(G) U> per row (G, U the
    stored bf16 values), dh = w dh_s, then the SwiGLU backward of
    expert_fc2_dgrad_swiglu. Returns (dGU in bf16, dw)."""
    F = W2_e.shape[1]
    dhs = np.asarray(dY, np.float64) @ np.asarray(W2_e, np.float64)
    G, U = GU[:, :F], GU[:, F:]
    dw = (dhs * (silu(G) * U)).sum(axis=1)
    dh = np.asarray(w, np.float64)[:, None] * dhs
    sg = sigmoid(G)
    d = _rb(np.concatenate([dh * U * sg * (1.0 + G * (1.0 - sg)), dh * silu(G)], axis=1),
            rounding)
    return d, dw


def layer_backward_reordered(cfg, x, W_r, W13, W2, fwd, dY, rounding: bool = True):
    """Backward of layer_forward_reordered (same page and section).

    The expert's output gradient is dY itself (no weighting on the way in):
        dh_s = dY W2 (full precision),
        dw_tj = <dh_s, h> with h = silu(G) U recomputed from the stored bf16
                G, U (the routing weight's gradient, taken here instead of from
                the expert outputs y, which therefore need not be kept),
        dh = w_tj dh_s, then the SwiGLU backward as in layer_backward,
        dW2 = sum over rows of dY^T h_s, dW13 and dX as in layer_backward.
    The router gradient, dx and dW_r follow from dw exactly as in layer_backward.
    """
    x = np.asarray(x, np.float64)
    dY = np.asarray(dY, np.float64)
    T, H = x.shape
    E, k, F, S = cfg.E, cfg.k, cfg.F, cfg.n_shared
    idx, w, maps = fwd["idx"], fwd["w"], fwd["maps"]
    kept = maps["row_of"] >= 0
    dYb = _rb(dY, rounding)
    dw = np.zeros((T, k))
    dGU = np.zeros((T, k, 2 * F))
    dX = np.zeros((T, k, H))
    dW13 = np.zeros((E + S, 2 * F, H))
    dW2 = np.zeros((E + S, H, F))
    for e in range(E):
        tt, jj = np.nonzero((idx == e) & kept)
        if tt.size == 0:
            continue
        d, dw[tt, jj] = expert_fc2_dgrad_swiglu_weighted(dYb[tt], W2[e], fwd["GU"][tt, jj],
                                                         w[tt, jj], rounding)
        dGU[tt, jj] = d
        dX[tt, jj] = expert_fc1_dgrad(d, W13[e], rounding)
        dW2[e] = wgrad(dYb[tt], fwd["hs"][tt, jj], rounding)
        dW13[e] = wgrad(d, x[tt], rounding)
    dGU_s = np.zeros((S, T, 2 * F))
    dX_s = np.zeros((S, T, H))
    for s in range(S):
        dGU_s[s] = expert_fc2_dgrad_swiglu(dYb, W2[E + s], fwd["GU_s"][s], rounding)
        dX_s[s] = expert_fc1_dgrad(dGU_s[s], W13[E + s], rounding)
        dW2[E + s] = wgrad(dYb, fwd["h_s"][s], rounding)
        dW13[E + s] = wgrad(dGU_s[s], x, rounding)
    dlogits = router_dlogits(cfg, fwd["logits"], idx, w, dw)
    dx = _rb(dX.sum(axis=1) + dX_s.sum(axis=0) + dlogits @ np.asarray(W_r, np.float64), rounding)
    dW_r = _rf(dlogits.T @ x, rounding)
    return dict(dw=dw, dGU=dGU, dX=dX, dGU_s=dGU_s, dX_s=dX_s, dlogits=dlogits, dx=dx,
                dW_r=dW_r, dW13=dW13, dW2=dW2)


# --------------------------------------------------------------------------- #
# the FP8 layer (E4M3 with power-of-two block scales)
# --------------------------------------------------------------------------- #
DT_FP8_BLOCK = 1      # 128-element blocks, 128x128 weight tiles
DT_MXFP8 = 2          # 32-element blocks along the reduced dimension (MX)


def fp8_block(cfg) -> int:
    """Quantisation block length of an FP8 configuration: 32 for MXFP8 (the MX
    formats share one scale per 32 consecutive elements), else 128."""
    return 32 if getattr(cfg, "dtype", DT_FP8_BLOCK) == DT_MXFP8 else 128


def fp8_weights(cfg, W):
    """The two E4M3 forms of one expert weight W [out, in]: the forward GEMM's
    (reduces over `in`) and the data gradient's (reduces over `out`). Block
    recipe: one 128x128 tile quantisation serves both. MXFP8: 1x32 blocks
    along `in` for the forward, 32x1 blocks along `out` for the data gradient."""
    if fp8_block(cfg) == 128:
        q = quant_tiles(W)
        return q, q
    return quant_rows(W, 32), quant_cols(W, 32)


def layer_forward_fp8(cfg, x, W_r, bias, W13, W2, logits=None):
    """The layer with its expert GEMMs on E4M3-quantised operands.

    Routing stays in fp32 (es summary §2.4: the router keeps high precision).
    Per expert, with b = fp8_block(cfg): X_q = quant_rows(X, b) (1 x b along
    H), the weights' forward forms (fp8_weights), GU = bf16(X_q W13_q^T),
    h = bf16(silu(G) U), y = bf16(quant_rows(h, b) W2_q^T) (1 x b along F);
    combine as in bf16. The data-gradient forms of the weights are kept for
    the backward (Wd13, Wd2).
    """
    x = np.asarray(x, np.float64)
    T, H = x.shape
    E, k, F = cfg.E, cfg.k, cfg.F
    if logits is None:
        logits = router_logits(x, W_r)
    logits = np.asarray(logits, np.float64)
    idx, w = route(logits, cfg, bias)
    maps = permutation_maps(idx, cfg)
    kept = maps["row_of"] >= 0
    GU = np.zeros((T, k, 2 * F))
    h = np.zeros((T, k, F))
    y = np.zeros((T, k, H))
    b = fp8_block(cfg)
    Wq13, Wq2, Wd13, Wd2 = {}, {}, {}, {}
    for e in range(E):
        tt, jj = np.nonzero((idx == e) & kept)
        if tt.size == 0:
            continue
        order = np.argsort(tt, kind="stable")            # rows in token order
        tt, jj = tt[order], jj[order]
        Wq13[e], Wd13[e] = fp8_weights(cfg, W13[e])
        Wq2[e], Wd2[e] = fp8_weights(cfg, W2[e])
        g, hh = expert_fc1(quant_rows(x[tt], b), Wq13[e])
        GU[tt, jj], h[tt, jj] = g, hh
        y[tt, jj] = expert_fc2(quant_rows(hh, b), Wq2[e])
    acc = np.einsum("tj,tjh->th", np.where(kept, w, 0.0), y)
    return dict(logits=logits, idx=idx, w=w, maps=maps, GU=GU, h=h, y=y, out=round_bf16(acc),
                Wq13=Wq13, Wq2=Wq2, Wd13=Wd13, Wd2=Wd2)


def layer_backward_fp8(cfg, x, W_r, W13, W2, fwd, dY):
    """Backward of layer_forward_fp8, with b = fp8_block(cfg). Data gradients:
    dO and dGU quantised in 1 x b slices along the dimension their GEMM reduces
    (H, 2F), the weights in their data-gradient forms; weight gradients: both
    operands quantised in b x 1 slices along the expert's tokens (in token
    order)."""
    x = np.asarray(x, np.float64)
    dY = np.asarray(dY, np.float64)
    T, H = x.shape
    E, k, F = cfg.E, cfg.k, cfg.F
    idx, w, maps = fwd["idx"], fwd["w"], fwd["maps"]
    kept = maps["row_of"] >= 0
    b = fp8_block(cfg)
    dO = round_bf16(np.where(kept, w, 0.0)[:, :, None] * dY[:, None, :])
    dw = np.where(kept, np.einsum("th,tjh->tj", dY, fwd["y"]), 0.0)
    dGU = np.zeros((T, k, 2 * F))
    dX = np.zeros((T, k, H))
    dW13 = np.zeros((E, 2 * F, H))
    dW2 = np.zeros((E, H, F))
    for e in range(E):
        tt, jj = np.nonzero((idx == e) & kept)
        if tt.size == 0:
            continue
        order = np.argsort(tt, kind="stable")
        tt, jj = tt[order], jj[order]
        Wd13, Wd2 = fwd["Wd13"][e], fwd["Wd2"][e]
        dOe = dO[tt, jj]
        d = expert_fc2_dgrad_swiglu(quant_rows(dOe, b), Wd2, fwd["GU"][tt, jj])
        dGU[tt, jj] = d
        dX[tt, jj] = expert_fc1_dgrad(quant_rows(d, b), Wd13)
        dW2[e] = wgrad(quant_cols(dOe, b), quant_cols(fwd["h"][tt, jj], b))
        dW13[e] = wgrad(quant_cols(d, b), quant_cols(x[tt], b))
    dlogits = router_dlogits(cfg, fwd["logits"], idx, w, dw)
    dx = round_bf16(dX.sum(axis=1) + dlogits @ np.asarray(W_r, np.float64))
    dW_r = round_f32(dlogits.T @ x)
    return dict(dO=dO, dw=dw, dGU=dGU, dX=dX, dlogits=dlogits, dx=dx, dW_r=dW_r, dW13=dW13,
                dW2=dW2)
