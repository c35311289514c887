"""CPU oracle for the block-local tail of the DFlash2 drafter (float64, numpy).

TEST INFRASTRUCTURE ONLY. This module states what the hot path computes, as
plainly as possible, so that the CUDA library can be checked against it. Only
the test suite, the smoke check and the benchmark's CPU-baseline / reference
leg may import it. It shares no code with the CUDA path and imports nothing
from it; the product path never calls it.

Sources (web pages; cited by title and section below):

* [ts]  "@mlx-bun/inference 0.0.0-stage -> 1.0.0", diff of
        package/src/models/speculative/dflash2.ts: the header comment
        ("layer", "output", "selector" paragraphs), ``#rms``,
        ``#coefficients``, ``#conv``, ``#block`` and ``#select``.
* [max] "max.pipelines.architectures.dflash2_qwen3_5" (Modular MAX Python API):
        ``DFlash2GroupedConv`` (+ ``prepare`` / ``finish``),
        ``DFlash2CandidateSelector`` (+ ``score_edges`` / ``select_path``),
        ``DFlash2Qwen3_5.compute_candidates``, ``DFlash2TransformerBlock``.

Every input arrives as float64 holding the exact values the GPU is given
(bf16- or f32-representable); every computation is float64 with no rounding
to the storage dtype. Readings taken where the pages are silent:

* D's column order is (side, tap, group), side-major ([ts] ``#coefficients``
  reshapes the projection to [B, G, stage, tap, groups, 1]).
* ``finish`` receives side 1's deltas *without* the base kernel; the base is
  added again when side 1 is applied ([max] ``prepare`` returns the
  [tokens, taps, groups] coefficients; [ts] adds base once per site).
* top-K order: value descending, equal values by lower vocabulary id first;
  the same rule decides membership at the K-th place ([ts] ``#select`` uses an
  unordered partition, [max] is silent).
* the walk's argmax takes the lowest candidate position on a tie (first
  maximum, as an argmax over the candidate axis returns it).
* slot 0's predecessor is the anchor for every predecessor index p.

Parity pins: every function here is pinned by tests that do not re-derive it
(closed forms, special cases reducing to textbook routines, invariants stated
on the pages, brute force on tiny inputs). ``block_tail`` composes pinned
functions; the composition itself has no worked example on the pages.
"""
from __future__ import annotations

import numpy as np

SLAB_ROWS = 16384  # vocabulary rows per head slab (bounds host memory only)


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------- the grouped dynamic conv

def rms_norm(x, w, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w.

    [ts] ``#rms`` (an RMS norm with the layer's gain and the config's eps),
    applied to the sublayer input before ``kernel_projection`` ([ts] header,
    "layer" paragraph: n = rms(x)).
    """
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(w)


def kernel_projection(n, w_kp) -> np.ndarray:
    """D = n @ W_kpᵀ, W_kp stored [out, in] with out = 2 sides * 2 taps * groups.

    [ts] ``#coefficients`` (the BF16 projection of n) and [max]
    ``DFlash2GroupedConv`` (one projection per sublayer emits both sides,
    width 2 * taps * num_groups).
    Returns D with its last axis split as [side, tap, group].
    """
    n = _f64(n)
    w = _f64(w_kp)
    d = n @ w.T
    groups = w.shape[0] // 4
    return d.reshape(n.shape[:-1] + (2, 2, groups))


def coefficients(D, base, group_size: int) -> np.ndarray:
    """Per-channel coefficients coef[..., side, tap, c] = base[side, tap, c] + D[..., side, tap, c // group_size].

    [ts] ``#coefficients`` (broadcast each group's delta across its
    ``convGroupSize`` channels, then add the per-channel base kernel) and
    [max] ``DFlash2GroupedConv`` (base per channel, delta per group).
    """
    D = _f64(D)
    wide = np.repeat(D, group_size, axis=-1)
    return wide + _f64(base)


def conv_apply(y, c_tap0, c_tap1) -> np.ndarray:
    """Two-tap block-local conv: out[b, t] = c_tap0[b, t] * y[b, t] + c_tap1[b, t] * y[b, t-1], y[b, -1] = 0.

    [ts] header formula Conv(y)[t,c] = sum over tau of (base + D)[t,tau,c] * y[t-tau, c]
    with y[-1] = 0, and ``#conv`` (prev = zero row followed by rows 0..G-2);
    [max] ``DFlash2GroupedConv``: t is block-local, so taps before the block
    start read zero and nothing crosses a block boundary.
    y: [B, G, H]; c_tap0, c_tap1: [B, G, H].
    """
    y = _f64(y)
    prev = np.zeros_like(y)
    prev[:, 1:, :] = y[:, :-1, :]
    return _f64(c_tap0) * y + _f64(c_tap1) * prev


def conv_prepare(x, norm_w, eps: float, w_kp, base, group_size: int):
    """The pre-sublayer half of one conv site.

    [max] ``DFlash2GroupedConv.prepare`` and ``DFlash2TransformerBlock``
    (h = norm(r); h = conv.prepare(h)); [ts] ``#block`` (n = rms(x);
    coef = #coefficients(n); a = #conv(n, coef, 0)).
    ``norm_w`` None means x is already normalised (n = x).
    Returns (out [B,G,H] = side-0 conv of n, d_side1 [B,G,2,groups] = side 1's
    deltas without base, n).
    """
    n = _f64(x) if norm_w is None else rms_norm(x, norm_w, eps)
    D = kernel_projection(n, w_kp)                      # [B, G, 2, 2, groups]
    coef0 = coefficients(D[..., 0, :, :], base[0], group_size)   # [B, G, 2, H]
    out = conv_apply(n, coef0[..., 0, :], coef0[..., 1, :])
    return out, D[..., 1, :, :].copy(), n


def conv_finish(y, d_side1, base, group_size: int, residual=None) -> np.ndarray:
    """The post-sublayer half: side 1 applied to the sublayer output y, added to the residual stream.

    [max] ``DFlash2GroupedConv.finish`` (reuses prepare's coefficients) and
    ``DFlash2TransformerBlock`` (r += conv.finish(h)); [ts] ``#block``
    (x = x + #conv(out, coef, 1), the add in f32).
    ``residual`` None returns the conv output alone.
    """
    coef1 = coefficients(d_side1, base[1], group_size)  # [B, G, 2, H]
    out = conv_apply(y, coef1[..., 0, :], coef1[..., 1, :])
    if residual is None:
        return out
    return _f64(residual) + out


# --------------------------------------------------------------------------- the candidate-path selector

def head_logits(h, w_head, bias=None, rows_per_slab: int = SLAB_ROWS) -> np.ndarray:
    """logits[m, v] = sum_k h[m, k] * W[v, k] (+ bias[v]); W stored [V, H].

    [ts] ``#block`` (rows 1..G-1, normed, through the target's lm_head) and
    [max] ``compute_candidates`` (float32 logits [batch, steps, vocab]).
    ``w_head`` may be any object whose row slices give float64 arrays; it is
    read in slabs of ``rows_per_slab`` rows to bound host memory.
    """
    h = _f64(h)
    V = w_head.shape[0]
    out = np.empty(h.shape[:-1] + (V,), dtype=np.float64)
    for v0 in range(0, V, rows_per_slab):
        v1 = min(V, v0 + rows_per_slab)
        out[..., v0:v1] = h @ _f64(w_head[v0:v1]).T
    if bias is not None:
        out += _f64(bias)
    return out


def top_k(logits, K: int):
    """The K largest logits of each row, ordered value descending then id ascending.

    [ts] ``#select`` (top-K candidates per position from one partition over
    all positions) and [max] ``compute_candidates`` ((candidate_ids,
    unary_logits), both [batch, steps, top_k]). A full stable sort of each row
    by descending value keeps equal values in id order.
    Returns (ids int64 [..., K], values float64 [..., K]).
    """
    L = _f64(logits)
    flat = L.reshape(-1, L.shape[-1])
    ids = np.empty((flat.shape[0], K), dtype=np.int64)
    for i, row in enumerate(flat):
        order = np.argsort(-row, kind="stable")
        ids[i] = order[:K]
    vals = np.take_along_axis(flat, ids, axis=1)
    return ids.reshape(L.shape[:-1] + (K,)), vals.reshape(L.shape[:-1] + (K,))


def listed_candidates(cols, ids) -> np.ndarray:
    """Token ids of top-K columns taken over a draft vocabulary: ids[cols].

    [ts] ``#block`` (a target that declares a draft vocabulary projects the head onto those rows
    only) and ``#select`` (``ids`` maps the columns of logits over the draft vocabulary to token
    ids before the codebook gathers). The top-K itself runs over the listed columns with the same
    rule as ``top_k`` (equal values: lower column, i.e. earlier listed row, first).
    """
    return np.asarray(ids, dtype=np.int64)[np.asarray(cols, dtype=np.int64)]


def kth_margin(logits, K: int) -> np.ndarray:
    """Per row: (K-th largest) - ((K+1)-th largest) logit; the gap that decides top-K membership."""
    L = _f64(logits)
    s = -np.sort(-L.reshape(-1, L.shape[-1]), axis=1)
    return (s[:, K - 1] - s[:, K]).reshape(L.shape[:-1])


def hidden_projection(h, w_proj) -> np.ndarray:
    """z = h @ Pᵀ, P stored [R, H]. [ts] ``#block`` (z = selProj(h), on the normed drafter hidden)
    and [max] ``DFlash2CandidateSelector`` (proj(h_l))."""
    return _f64(h) @ _f64(w_proj).T


def score_edges(cand, unary, z, anchors, pred_book, succ_book) -> np.ndarray:
    """S[b, l, p, c] = unary[b,l,c] + sum_r pred_book[pid(b,l,p), r] * z[b,l,r] * succ_book[cand[b,l,c], r].

    pid(b, 0, p) = anchors[b] for every p; pid(b, l, p) = cand[b, l-1, p].
    [max] ``DFlash2CandidateSelector`` formula and ``score_edges`` (output
    [batch, steps, top_k, top_k] indexed [b, l, p, c]); [ts] ``#select``
    (predecessor rows gathered by the previous token, successor rows by the
    candidate, weighted by z).
    cand: [B, steps, K] int; unary: [B, steps, K]; z: [B, steps, R]; anchors: [B].
    """
    cand = np.asarray(cand, dtype=np.int64)
    B, steps, K = cand.shape
    pred = _f64(pred_book)
    succ = _f64(succ_book)
    pid = np.empty((B, steps, K), dtype=np.int64)
    pid[:, 0, :] = np.asarray(anchors, dtype=np.int64)[:, None]
    pid[:, 1:, :] = cand[:, :-1, :]
    P = pred[pid]                                   # [B, steps, K(p), R]
    C = succ[cand]                                  # [B, steps, K(c), R]
    edge = np.einsum("blpr,blr,blcr->blpc", P, _f64(z), C)
    return _f64(unary)[:, :, None, :] + edge


def select_path(S, cand, seed_index: int = 0):
    """Greedy left-to-right walk over S, following the best successor.

    [max] ``select_path`` (a single greedy pass, no beam, no Viterbi; slot 0's
    rows are all the anchor's, so index 0 seeds it) and [ts] ``#select``
    (argmax of unary + edge per position; the chosen token becomes the next
    predecessor). Ties go to the lowest candidate position. ``seed_index`` is
    the predecessor position read at slot 0 (any value gives the same walk
    when slot 0's rows are identical, as ``score_edges`` makes them).
    Returns (path ids [B, steps], chosen positions [B, steps]).
    """
    S = _f64(S)
    cand = np.asarray(cand)
    B, steps, K, _ = S.shape
    pos = np.zeros((B, steps), dtype=np.int64)
    path = np.zeros((B, steps), dtype=np.int64)
    for b in range(B):
        p = seed_index
        for l in range(steps):
            c = int(np.argmax(S[b, l, p, :]))
            pos[b, l] = c
            path[b, l] = cand[b, l, c]
            p = c
    return path, pos


def block_columns(depth: int, G: int) -> int:
    """Rows a block drafting ``depth`` tokens runs over: min(G, max(1, depth) + 1).

    [ts] ``blockColumns`` (the anchor and up to ``depth`` mask positions, never fewer than one);
    [max] ``DFlash2Qwen3_5.supports_zero_draft_rows`` is False (no block drafts nothing).
    A block over ``columns`` rows drafts ``columns - 1`` tokens.
    """
    return min(int(G), max(1, int(depth)) + 1)


def select_path_depths(S, cand, depths):
    """The greedy walk of blocks that draft different numbers of tokens in one batch.

    [ts] ``blockColumns`` / ``#block``: a block asked to draft ``depth`` tokens runs over
    ``block_columns(depth, steps + 1)`` rows (the anchor and its mask rows) and drafts one token
    per mask row, so block b walks its first ``min(steps, max(1, depths[b]))`` slots; every
    value of ``depths`` is accepted, as ``blockColumns`` accepts it. The slots after them hold -1
    (no token). Rows past a block's depth are padding in a dense [B, G, ...] batch.
    Returns (path ids [B, steps] with -1 padding, chosen positions [B, steps] with -1 padding).
    """
    S = _f64(S)
    cand = np.asarray(cand)
    B, steps, K, _ = S.shape
    pos = np.full((B, steps), -1, dtype=np.int64)
    path = np.full((B, steps), -1, dtype=np.int64)
    for b in range(B):
        d = block_columns(depths[b], steps + 1) - 1
        p = 0
        for l in range(d):
            c = int(np.argmax(S[b, l, p, :]))
            pos[b, l] = c
            path[b, l] = cand[b, l, c]
            p = c
    return path, pos


def walk_margins(S, pos) -> np.ndarray:
    """Per (b, l): best minus second-best of the row the walk read at slot l (its tie margin)."""
    S = _f64(S)
    B, steps, K, _ = S.shape
    m = np.empty((B, steps))
    for b in range(B):
        p = 0
        for l in range(steps):
            row = np.sort(S[b, l, p, :])[::-1]
            m[b, l] = row[0] - row[1] if K > 1 else np.inf
            p = int(pos[b, l])
    return m


# --------------------------------------------------------------------------- composition

def conv_chain(x0, sites, eps: float, group_size: int, norm_inputs: bool = True):
    """Run the conv sites in order: per site n = rms(x); a = prepare(n); x += finish(y_site).

    The sublayer between prepare and finish is replaced by the site's seeded
    output ``y`` (its input ``a`` is produced but not consumed).
    [max] ``DFlash2TransformerBlock`` (norm -> prepare -> sublayer -> finish ->
    residual, twice per layer); [ts] ``#block`` (the same per layer).
    ``sites``: sequence of objects with w_kp, base, norm_w, y.
    Returns (x_final, list of per-site (a, d_side1, n)).
    """
    x = _f64(x0)
    trace = []
    for s in sites:
        a, d1, n = conv_prepare(x, s.norm_w if norm_inputs else None, eps, s.w_kp, s.base, group_size)
        x = conv_finish(s.y, d1, s.base, group_size, residual=x)
        trace.append((a, d1, n))
    return x, trace


def block_tail(x0, sites, final_norm_w, eps, group_size, w_head, bias, w_proj,
               pred_book, succ_book, anchors, K: int):
    """The whole block tail: conv chain -> rows 1..G-1 -> final norm -> head -> top-K -> z -> S -> walk.

    [ts] ``#block`` (rows 1..G-1 go through the final norm and the head;
    z = hidden_projection(h); ``#select``) and [max] ``DFlash2Qwen3_5``.
    Returns a dict of every intermediate.
    """
    x, trace = conv_chain(x0, sites, eps, group_size)
    h = rms_norm(x[:, 1:, :], final_norm_w, eps)
    logits = head_logits(h, w_head, bias)
    cand, unary = top_k(logits, K)
    z = hidden_projection(h, w_proj)
    S = score_edges(cand, unary, z, anchors, pred_book, succ_book)
    path, pos = select_path(S, cand)
    return dict(x=x, trace=trace, h=h, logits=logits, cand=cand, unary=unary, z=z, S=S,
                path=path, pos=pos)


def block_tail_ragged(x0, sites, final_norm_w, eps, group_size, w_head, bias, w_proj,
                      pred_book, succ_book, anchors, K: int, depths):
    """The block tail of a batch whose blocks draft different numbers of tokens, with only the
    drafted rows going through the head and the selector.

    [ts] ``blockColumns`` / ``#block``: block b runs over ``block_columns(depths[b], G)`` rows, so
    rows 1..d_b (d_b = that minus one) go through the final norm, the head, top-K, z and
    ``#select``, whose walk has d_b slots. The conv sites run over the whole dense block (rows past
    d_b + 1 are padding that no earlier row reads). Rows of all blocks are packed in block order.
    Returns a dict: offsets [B + 1]; h, logits, cand, unary, z, S over the packed rows; path and
    pos [B, G - 1] with -1 past each block's d_b.
    """
    x, _ = conv_chain(x0, sites, eps, group_size)
    B, G, _ = x.shape
    steps = G - 1
    offsets = [0]
    hs, logits, cands, unaries, zs, Ss = [], [], [], [], [], []
    path = np.full((B, steps), -1, dtype=np.int64)
    pos = np.full((B, steps), -1, dtype=np.int64)
    for b in range(B):
        d = block_columns(depths[b], G) - 1
        offsets.append(offsets[-1] + d)
        h = rms_norm(x[b, 1:1 + d, :], final_norm_w, eps)           # [d, H]
        lg = head_logits(h, w_head, bias)
        c, u = top_k(lg, K)
        zz = hidden_projection(h, w_proj)
        S = score_edges(c[None], u[None], zz[None], np.asarray(anchors)[b:b + 1], pred_book, succ_book)
        pth, ps = select_path(S, c[None])
        path[b, :d], pos[b, :d] = pth[0], ps[0]
        hs.append(h); logits.append(lg); cands.append(c); unaries.append(u); zs.append(zz); Ss.append(S[0])
    return dict(offsets=np.asarray(offsets), h=np.concatenate(hs), logits=np.concatenate(logits),
                cand=np.concatenate(cands), unary=np.concatenate(unaries), z=np.concatenate(zs),
                S=np.concatenate(Ss), path=path, pos=pos)


# --------------------------------------------------------------------------- sublayer projections

def affine_dequantize(q, scales, biases, group: int = 64) -> np.ndarray:
    """W[n, k] = scales[n, k // group] * q[n, k] + biases[n, k // group] (affine quantisation).

    [ts] ``quantizedWeight`` (``quantize(source, 64, bits)``, ``QuantizedLinear`` with
    ``groupSize: 64, mode: "affine"``): a 4-bit code per weight and one scale and bias per row and
    group of 64 input channels. q: [N, K] integer codes; scales, biases: [N, K // group].
    """
    q = _f64(q)
    return q * np.repeat(_f64(scales), group, axis=1) + np.repeat(_f64(biases), group, axis=1)


def projection(a, W) -> np.ndarray:
    """y = a @ Wᵀ, W stored [out, in]. [ts] ``Bf16Projection.forward`` (a matmul against the stored
    transpose) and the sublayers' q/k/v/o and gate/up/down projections."""
    return _f64(a) @ _f64(W).T


def sublayer_in(n, d_side0, base, group_size: int, W) -> np.ndarray:
    """An input projection of the sublayer applied to prepare's output: Conv_0(n) @ Wᵀ.

    [ts] ``#block`` (a = #conv(n, coef, 0), then q/k/v = projection(a) or gate/up = projection(m's
    conv)); [max] ``DFlash2TransformerBlock`` (h = conv.prepare(norm(r)); h feeds the sublayer).
    n: [B, G, H]; d_side0: [B, G, 2, groups] (side 0's deltas); base [2, 2, H]; W [N, H].
    """
    coef0 = coefficients(d_side0, base[0], group_size)                   # [B, G, 2, H]
    a = conv_apply(n, coef0[..., 0, :], coef0[..., 1, :])
    return projection(a, W)


def sublayer_out(a, W, d_side1, base, group_size: int, residual=None) -> np.ndarray:
    """The sublayer's output projection followed by finish: residual + Conv_1(a @ Wᵀ).

    [ts] ``#block`` (out = o.forward(attn) or down.forward(prod); x = x + #conv(out, coef, 1));
    [max] ``DFlash2TransformerBlock`` (r += conv.finish(sublayer output)).
    a: [B, G, K]; W: [H, K]; d_side1: [B, G, 2, groups].
    """
    return conv_finish(projection(a, W), d_side1, base, group_size, residual=residual)
