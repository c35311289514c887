"""Pins for the CPU oracle: facts fixed by the pages and by mathematics, not by the oracle itself.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, a swapped side/tap, an off-by-one at the
block boundary, a wrong tie rule) fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import dflash2_oracle as O
from tests.conftest import load_golden

RNG = np.random.default_rng(12345)


def _rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# ----------------------------------------------------------------------------- RMSNorm

def test_rms_norm_closed_forms():
    # a 3-4-0-0 row: mean square 25/4, so n = x / 2.5 (eps = 0)
    x = np.array([[3.0, 4.0, 0.0, 0.0]])
    np.testing.assert_allclose(O.rms_norm(x, np.ones(4), 0.0), x / 2.5, rtol=0, atol=1e-15)
    # constant row c: n = c / sqrt(c^2 + eps) * w
    c, eps = -0.3, 1e-2
    w = np.array([1.0, 2.0, -1.0, 0.5])
    np.testing.assert_allclose(O.rms_norm(np.full((1, 4), c), w, eps)[0], c / math.sqrt(c * c + eps) * w, rtol=1e-14)
    # each row is normalised on its own (not over the whole tensor)
    x = np.array([[1.0, 1.0], [10.0, 10.0]])
    np.testing.assert_allclose(O.rms_norm(x, np.ones(2), 0.0), np.ones((2, 2)), rtol=1e-15)


def test_rms_norm_scale_invariance():
    x = _rand(3, 5, 64)
    np.testing.assert_allclose(O.rms_norm(7.5 * x, np.ones(64), 0.0), O.rms_norm(x, np.ones(64), 0.0), rtol=1e-12)


# ----------------------------------------------------------------------------- the two-tap conv

def test_conv_golden_hand_example():
    g = load_golden("conv_two_tap_hand.txt")
    n = np.array(g["n"]).reshape(1, 3, 2)
    w_kp = np.array(g["w_kp"]).reshape(4, 2)
    base = np.array(g["base"]).reshape(2, 2, 2)
    out, d1, n_out = O.conv_prepare(n, None, 0.0, w_kp, base, group_size=2)
    np.testing.assert_allclose(out.ravel(), g["prepare"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(d1.ravel(), g["d_side1"], rtol=0, atol=1e-12)
    y = np.array(g["y"]).reshape(1, 3, 2)
    fin = O.conv_finish(y, d1, base, 2, residual=np.zeros((1, 3, 2)))
    np.testing.assert_allclose(fin.ravel(), g["finish"], rtol=0, atol=1e-12)


def _identity_base(H):
    base = np.zeros((2, 2, H))
    base[:, 0, :] = 1.0
    return base


def test_conv_identity():
    # D = 0 (zero projection) and base = [1, 0] on both sides: prepare returns n, finish adds y
    B, G, H, gs = 3, 5, 32, 16
    x = _rand(B, G, H)
    y = _rand(B, G, H)
    out, d1, n = O.conv_prepare(x, None, 0.0, np.zeros((4 * H // gs, H)), _identity_base(H), gs)
    assert np.array_equal(out, x)
    assert np.array_equal(d1, np.zeros((B, G, 2, H // gs)))
    assert np.array_equal(O.conv_finish(y, d1, _identity_base(H), gs, residual=x), x + y)


def test_conv_shift_pins_block_boundary():
    # base = [0, 1]: out[t] = in[t-1] inside each block and out[0] = 0 for every block
    B, G, H, gs = 4, 6, 16, 16
    x = _rand(B, G, H)
    base = np.zeros((2, 2, H))
    base[:, 1, :] = 1.0
    out, d1, _ = O.conv_prepare(x, None, 0.0, np.zeros((4, H)), base, gs)
    assert np.array_equal(out[:, 0, :], np.zeros((B, H)))
    assert np.array_equal(out[:, 1:, :], x[:, :-1, :])
    fin = O.conv_finish(x, d1, base, gs)
    assert np.array_equal(fin[:, 0, :], np.zeros((B, H)))
    assert np.array_equal(fin[:, 1:, :], x[:, :-1, :])


def test_conv_static_base_equals_textbook_causal_conv1d():
    # D = 0 and an arbitrary base: each (block, channel) is the causal 2-tap FIR
    # given by numpy's full linear convolution, truncated to the block length.
    B, G, H, gs = 2, 7, 32, 16
    x = _rand(B, G, H)
    base = _rand(2, 2, H)
    out, d1, _ = O.conv_prepare(x, None, 0.0, np.zeros((4 * H // gs, H)), base, gs)
    fin = O.conv_finish(x, d1, base, gs)
    for b in range(B):
        for c in range(H):
            np.testing.assert_allclose(out[b, :, c], np.convolve(x[b, :, c], base[0, :, c])[:G], atol=1e-13)
            np.testing.assert_allclose(fin[b, :, c], np.convolve(x[b, :, c], base[1, :, c])[:G], atol=1e-13)


@pytest.mark.parametrize("side,tap", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_conv_projection_column_order(side, tap):
    # One non-zero kernel_projection row, row (side*2 + tap)*groups + g = alpha*e_k, so
    # D[t, side, tap, g] = alpha * n[t, k] and every other delta is 0. With base = [1, 0]
    # the closed forms below follow from Conv(y)[t,c] = sum_tau (base + D)[t,tau,c] y[t-tau,c].
    B, G, H, gs = 2, 5, 64, 16
    groups = H // gs
    g, k, alpha = 2, 5, 0.75
    n = _rand(B, G, H)
    y = _rand(B, G, H)
    w = np.zeros((4 * groups, H))
    w[(side * 2 + tap) * groups + g, k] = alpha
    base = _identity_base(H)
    out, d1, _ = O.conv_prepare(n, None, 0.0, w, base, gs)
    fin = O.conv_finish(y, d1, base, gs)
    in_g = np.zeros(H, dtype=bool)
    in_g[g * gs:(g + 1) * gs] = True
    d = alpha * n[:, :, k][:, :, None]          # the one delta, per (b, t)
    y_prev = np.concatenate([np.zeros((B, 1, H)), y[:, :-1]], axis=1)
    n_prev = np.concatenate([np.zeros((B, 1, H)), n[:, :-1]], axis=1)
    if side == 0:
        exp = n.copy()
        if tap == 0:
            exp[:, :, in_g] = (1 + d) * n[:, :, in_g]
        else:
            exp[:, :, in_g] = n[:, :, in_g] + d * n_prev[:, :, in_g]
        np.testing.assert_allclose(out, exp, atol=1e-13)
        np.testing.assert_array_equal(fin, y)
    else:
        np.testing.assert_array_equal(out, n)
        exp = y.copy()
        if tap == 0:
            exp[:, :, in_g] = (1 + d) * y[:, :, in_g]
        else:
            exp[:, :, in_g] = y[:, :, in_g] + d * y_prev[:, :, in_g]
        np.testing.assert_allclose(fin, exp, atol=1e-13)
        expected_d1 = np.zeros((B, G, 2, groups))
        expected_d1[:, :, tap, g] = d[:, :, 0]
        np.testing.assert_allclose(d1, expected_d1, atol=1e-15)


def test_conv_block_isolation():
    # Perturbing one block leaves every other block's prepare/finish outputs bit-identical.
    B, G, H, gs = 4, 8, 32, 16
    x = _rand(B, G, H)
    y = _rand(B, G, H)
    w = _rand(4 * H // gs, H, scale=0.2)
    base = _rand(2, 2, H)
    ref_out, ref_d1, _ = O.conv_prepare(x, np.ones(H), 1e-6, w, base, gs)
    ref_fin = O.conv_finish(y, ref_d1, base, gs, residual=x)
    x2, y2 = x.copy(), y.copy()
    x2[2] += _rand(G, H)
    y2[2] += _rand(G, H)
    out, d1, _ = O.conv_prepare(x2, np.ones(H), 1e-6, w, base, gs)
    fin = O.conv_finish(y2, d1, base, gs, residual=x2)
    keep = [0, 1, 3]
    assert np.array_equal(out[keep], ref_out[keep])
    assert np.array_equal(fin[keep], ref_fin[keep])
    assert not np.array_equal(out[2], ref_out[2])


def test_conv_first_row_uses_tap0_only():
    # t = 0 of a block has no predecessor: changing tap 1's base leaves row 0 unchanged.
    B, G, H, gs = 2, 4, 16, 16
    n = _rand(B, G, H)
    w = _rand(4, H, scale=0.3)
    base = _rand(2, 2, H)
    a, _, _ = O.conv_prepare(n, None, 0.0, w, base, gs)
    base2 = base.copy()
    base2[0, 1] += 3.0
    b, _, _ = O.conv_prepare(n, None, 0.0, w, base2, gs)
    assert np.array_equal(a[:, 0], b[:, 0])
    assert not np.allclose(a[:, 1:], b[:, 1:])


def test_conv_chain_identity_sites_sum_residuals():
    # every site with a zero projection and base [1,0]: x_final = x0 + sum of the sublayer outputs
    class Site:
        pass
    B, G, H, gs = 2, 4, 32, 16
    x0 = _rand(B, G, H)
    sites = []
    for _ in range(3):
        s = Site()
        s.w_kp = np.zeros((4 * H // gs, H))
        s.base = _identity_base(H)
        s.norm_w = np.ones(H)
        s.y = _rand(B, G, H)
        sites.append(s)
    x, trace = O.conv_chain(x0, sites, 1e-6, gs)
    np.testing.assert_allclose(x, x0 + sites[0].y + sites[1].y + sites[2].y, atol=1e-13)
    # the first site's prepare output is rms(x0) (identity conv of the normed input)
    np.testing.assert_allclose(trace[0][0], O.rms_norm(x0, np.ones(H), 1e-6), atol=1e-15)


# ----------------------------------------------------------------------------- head, top-K, z

def test_head_logits_selection_matrix():
    # W[v] = e_{v mod H}: logit[m, v] = h[m, v mod H] + bias[v]; small slabs exercise the slab loop
    M, H, V = 5, 8, 37
    h = _rand(M, H)
    W = np.zeros((V, H))
    W[np.arange(V), np.arange(V) % H] = 1.0
    bias = _rand(V)
    L = O.head_logits(h, W, bias, rows_per_slab=10)
    np.testing.assert_allclose(L, h[:, np.arange(V) % H] + bias[None, :], atol=1e-15)
    L2 = O.head_logits(h, 2.0 * W, None, rows_per_slab=7)
    np.testing.assert_allclose(L2, 2.0 * h[:, np.arange(V) % H], atol=1e-15)


def test_topk_all_equal_logits_tie_rule():
    L = np.zeros((3, 100))
    ids, vals = O.top_k(L, 16)
    assert np.array_equal(ids, np.tile(np.arange(16), (3, 1)))
    assert np.array_equal(vals, np.zeros((3, 16)))


def test_topk_k1_is_first_argmax():
    L = RNG.integers(-3, 4, size=(50, 40)).astype(np.float64)   # many ties
    ids, vals = O.top_k(L, 1)
    assert np.array_equal(ids[:, 0], np.argmax(L, axis=1))


def test_topk_brute_force_rank_counting():
    # v is in the top-K iff fewer than K entries beat it under (greater value, or equal value and lower id);
    # its position in the list is exactly that count.
    L = RNG.integers(-4, 5, size=(20, 30)).astype(np.float64)
    K = 7
    ids, vals = O.top_k(L, K)
    for r in range(L.shape[0]):
        for v in range(L.shape[1]):
            beats = sum(1 for u in range(L.shape[1]) if L[r, u] > L[r, v] or (L[r, u] == L[r, v] and u < v))
            if beats < K:
                assert ids[r, beats] == v
                assert vals[r, beats] == L[r, v]
            else:
                assert v not in ids[r]


def test_kth_margin():
    L = np.array([[5.0, 1.0, 3.0, 2.0]])
    assert O.kth_margin(L, 2)[0] == 1.0   # 3 - 2
    assert O.kth_margin(L, 1)[0] == 2.0   # 5 - 3


def test_hidden_projection_selection_rows():
    M, H, R = 4, 10, 3
    h = _rand(M, H)
    P = np.zeros((R, H))
    P[0, 7] = 1.0
    P[1, 2] = -2.0
    P[2, 0] = 0.5
    z = O.hidden_projection(h, P)
    np.testing.assert_allclose(z, np.stack([h[:, 7], -2.0 * h[:, 2], 0.5 * h[:, 0]], axis=1), atol=1e-15)


# ----------------------------------------------------------------------------- edge scores and the walk

def _golden_selector():
    g = load_golden("selector_hand.txt")
    pred = np.array(g["pred_book"]).reshape(4, 1)
    succ = np.array(g["succ_book"]).reshape(4, 1)
    cand = np.array(g["cand"], dtype=np.int64).reshape(1, 2, 2)
    unary = np.array(g["unary"]).reshape(1, 2, 2)
    z = np.array(g["z"]).reshape(1, 2, 1)
    anchors = np.array([int(g["anchor"][0])])
    return g, pred, succ, cand, unary, z, anchors


def test_selector_golden_hand_example():
    g, pred, succ, cand, unary, z, anchors = _golden_selector()
    S = O.score_edges(cand, unary, z, anchors, pred, succ)
    np.testing.assert_allclose(S.ravel(), g["S"], atol=1e-12)
    path, pos = O.select_path(S, cand)
    assert path.ravel().tolist() == [int(v) for v in g["path"]]


def test_score_edges_brute_force_loops():
    B, steps, K, R, V = 2, 4, 3, 5, 11
    cand = RNG.integers(0, V, size=(B, steps, K))
    unary = _rand(B, steps, K)
    z = _rand(B, steps, R)
    anchors = RNG.integers(0, V, size=B)
    pred, succ = _rand(V, R), _rand(V, R)
    S = O.score_edges(cand, unary, z, anchors, pred, succ)
    for b in range(B):
        for l in range(steps):
            for p in range(K):
                prev = anchors[b] if l == 0 else cand[b, l - 1, p]
                for c in range(K):
                    acc = unary[b, l, c]
                    for r in range(R):
                        acc += pred[prev, r] * z[b, l, r] * succ[cand[b, l, c], r]
                    assert abs(S[b, l, p, c] - acc) < 1e-12


def test_score_edges_slot0_rows_identical_and_zero_pred():
    B, steps, K, R, V = 3, 5, 4, 8, 50
    cand = RNG.integers(0, V, size=(B, steps, K))
    unary = _rand(B, steps, K)
    z = _rand(B, steps, R)
    anchors = RNG.integers(0, V, size=B)
    pred, succ = _rand(V, R), _rand(V, R)
    S = O.score_edges(cand, unary, z, anchors, pred, succ)
    for p in range(1, K):
        assert np.array_equal(S[:, 0, p, :], S[:, 0, 0, :])
    S0 = O.score_edges(cand, unary, z, anchors, np.zeros((V, R)), succ)
    np.testing.assert_array_equal(S0, np.broadcast_to(unary[:, :, None, :], S0.shape))


def test_walk_seed_invariance():
    B, steps, K, R, V = 4, 6, 5, 8, 40
    cand = RNG.integers(0, V, size=(B, steps, K))
    unary = _rand(B, steps, K)
    z = _rand(B, steps, R)
    anchors = RNG.integers(0, V, size=B)
    S = O.score_edges(cand, unary, z, anchors, _rand(V, R), _rand(V, R))
    ref, _ = O.select_path(S, cand)
    for seed in range(K):
        path, _ = O.select_path(S, cand, seed_index=seed)
        assert np.array_equal(path, ref)


def test_walk_zero_codebooks_is_per_slot_argmax():
    B, steps, K, R, V = 3, 7, 16, 4, 300
    logits = _rand(B, steps, V)
    cand, unary = O.top_k(logits, K)
    z = _rand(B, steps, R)
    anchors = RNG.integers(0, V, size=B)
    S = O.score_edges(cand, unary, z, anchors, np.zeros((V, R)), np.zeros((V, R)))
    path, pos = O.select_path(S, cand)
    assert np.array_equal(pos, np.zeros((B, steps), dtype=np.int64))
    assert np.array_equal(path, np.argmax(logits, axis=-1))


def test_walk_exhaustive_unique_locally_optimal_path():
    # Enumerate all K^steps position sequences: exactly one is step-wise locally optimal from
    # the anchor (each choice the first maximum of the row its predecessor selects), and it is the walk.
    for trial in range(20):
        K, steps = 3, 4
        S = RNG.integers(-2, 3, size=(1, steps, K, K)).astype(np.float64)   # ties on purpose
        S[:, 0, 1:, :] = S[:, 0, :1, :]
        cand = np.arange(steps * K).reshape(1, steps, K)
        _, pos = O.select_path(S, cand)
        found = []
        for seq in itertools.product(range(K), repeat=steps):
            p, ok = 0, True
            for l, c in enumerate(seq):
                row = S[0, l, p]
                if not (row[c] == row.max() and all(row[j] < row[c] for j in range(c))):
                    ok = False
                    break
                p = c
            if ok:
                found.append(seq)
        assert len(found) == 1
        assert tuple(pos[0]) == found[0]


def test_walk_score_below_viterbi_optimum():
    K, steps = 4, 5
    for trial in range(10):
        S = _rand(1, steps, K, K)
        S[:, 0, 1:, :] = S[:, 0, :1, :]
        cand = np.arange(steps * K).reshape(1, steps, K)
        _, pos = O.select_path(S, cand)
        greedy = S[0, 0, 0, pos[0, 0]] + sum(S[0, l, pos[0, l - 1], pos[0, l]] for l in range(1, steps))
        best = max(S[0, 0, 0, seq[0]] + sum(S[0, l, seq[l - 1], seq[l]] for l in range(1, steps))
                   for seq in itertools.product(range(K), repeat=steps))
        assert greedy <= best + 1e-12


def test_walk_margins():
    S = np.zeros((1, 2, 2, 2))
    S[0, 0, :, :] = [3.0, 1.0]
    S[0, 1, 0, :] = [0.0, 0.5]
    S[0, 1, 1, :] = [2.0, 0.0]
    _, pos = O.select_path(S, np.zeros((1, 2, 2), dtype=np.int64))
    np.testing.assert_allclose(O.walk_margins(S, pos), [[2.0, 0.5]])


def test_block_tail_composition_shapes_and_zero_codebooks():
    # With zero codebooks the tail's path is the per-row argmax of h @ Wᵀ + bias on rows 1..G-1
    # of the normed final residual.
    class Site:
        pass
    B, G, H, gs, V, K, R = 2, 5, 32, 16, 64, 4, 8
    x0 = _rand(B, G, H)
    s = Site()
    s.w_kp = _rand(4 * H // gs, H, scale=0.1)
    s.base = _rand(2, 2, H, scale=0.5)
    s.norm_w = np.ones(H)
    s.y = _rand(B, G, H)
    W = _rand(V, H)
    bias = _rand(V)
    out = O.block_tail(x0, [s], np.ones(H), 1e-6, gs, W, bias, _rand(R, H), np.zeros((V, R)),
                       np.zeros((V, R)), RNG.integers(0, V, size=B), K)
    assert out["S"].shape == (B, G - 1, K, K)
    h = O.rms_norm(out["x"][:, 1:], np.ones(H), 1e-6)
    assert np.array_equal(out["path"], np.argmax(h @ W.T + bias, axis=-1))


def test_block_tail_predecessor_free_codebooks_reduce_to_per_slot_choice():
    # End to end with hand-computed intermediates: identity conv sites make x = x0 + sum of the
    # sublayer outputs; the final norm, head, top-K and z are written out in plain numpy; and with
    # every predecessor codebook row equal, S no longer depends on the previous choice, so the walk
    # picks, slot by slot, the candidate maximising logit + sum_r pred_r z_r succ[cand, r].
    class Site:
        pass
    B, G, H, gs, V, K, R, eps = 4, 9, 32, 16, 64, 4, 8, 1e-6
    ident = np.zeros((2, 2, H))
    ident[:, 0] = 1.0
    sites = []
    for _ in range(2):
        st = Site()
        st.w_kp = np.zeros((4 * H // gs, H))
        st.base = ident
        st.norm_w = np.ones(H)
        st.y = _rand(B, G, H)
        sites.append(st)
    x0 = _rand(B, G, H)
    g = 0.5 + RNG.random(H)
    W, bias, P = _rand(V, H), _rand(V), _rand(R, H)
    p_row = _rand(R)
    pred = np.tile(p_row, (V, 1))
    succ = _rand(V, R, scale=0.05)  # the pairwise term on the scale of the logit gaps
    anchors = RNG.integers(0, V, size=B)
    out = O.block_tail(x0, sites, g, eps, gs, W, bias, P, pred, succ, anchors, K)

    x = x0 + sites[0].y + sites[1].y
    xr = x[:, 1:]
    h = xr / np.sqrt((xr * xr).mean(axis=-1, keepdims=True) + eps) * g
    logits = h @ W.T + bias
    z = h @ P.T
    assert np.allclose(out["x"], x) and np.allclose(out["h"], h) and np.allclose(out["z"], z)
    want = np.empty((B, G - 1), dtype=np.int64)
    unary_only = np.empty_like(want)
    pair_only = np.empty_like(want)
    for b in range(B):
        for l in range(G - 1):
            cand = np.argsort(-logits[b, l], kind="stable")[:K]
            pair = (succ[cand] * (p_row * z[b, l])).sum(axis=-1)
            want[b, l] = cand[int(np.argmax(logits[b, l, cand] + pair))]
            unary_only[b, l] = cand[0]
            pair_only[b, l] = cand[int(np.argmax(pair))]
    # both terms decide some slots, so dropping either one would change the path
    assert not np.array_equal(want, unary_only) and not np.array_equal(want, pair_only)
    assert np.array_equal(out["path"], want)


def test_listed_vocabulary_equals_masked_full_head():
    # Top-K over a sorted draft vocabulary S (head rows W[S]) mapped through ids equals the full
    # head's top-K with every unlisted logit removed (same tie rule: the listed order is id order).
    M, H, V, K = 6, 12, 200, 8
    h = _rand(M, H)
    W = _rand(V, H)
    bias = RNG.integers(-2, 3, size=V).astype(np.float64)   # integer bias makes ties likely
    W[5] = W[7]                                             # two identical rows: an exact tie
    S = np.sort(RNG.choice(V, size=60, replace=False))
    S = np.union1d(S, [5, 7])
    cols, vals = O.top_k(O.head_logits(h, W[S], bias[S]), K)
    got = O.listed_candidates(cols, S)
    full = O.head_logits(h, W, bias)
    masked = np.full_like(full, -np.inf)
    masked[:, S] = full[:, S]
    ref_ids, ref_vals = O.top_k(masked, K)
    assert np.array_equal(got, ref_ids)
    np.testing.assert_array_equal(vals, ref_vals)


def test_listed_vocabulary_identity_map():
    M, H, V, K = 4, 8, 50, 5
    h = _rand(M, H)
    W = _rand(V, H)
    cols, _ = O.top_k(O.head_logits(h, W), K)
    assert np.array_equal(O.listed_candidates(cols, np.arange(V)), cols)


def test_mixed_depth_walk_is_prefix_of_full_walk():
    # The walk is causal: a block that drafts d tokens chooses exactly the first d tokens of the
    # full-depth walk, followed by -1 padding; d = steps reproduces the full walk. Depths outside
    # [1, steps] draft min(steps, max(1, d)) tokens (dflash2.ts blockColumns clamps both ends).
    B, steps, K, R, V = 8, 7, 5, 8, 60
    cand = RNG.integers(0, V, size=(B, steps, K))
    unary = _rand(B, steps, K)
    z = _rand(B, steps, R)
    anchors = RNG.integers(0, V, size=B)
    S = O.score_edges(cand, unary, z, anchors, _rand(V, R), _rand(V, R))
    full, full_pos = O.select_path(S, cand)
    depths = np.array([1, 7, 3, 0, 5, 2, -4, 11])
    drafted = [1, 7, 3, 1, 5, 2, 1, 7]
    path, pos = O.select_path_depths(S, cand, depths)
    for b in range(B):
        d = drafted[b]
        assert np.array_equal(path[b, :d], full[b, :d])
        assert np.array_equal(pos[b, :d], full_pos[b, :d])
        assert np.all(path[b, d:] == -1) and np.all(pos[b, d:] == -1)
    p2, _ = O.select_path_depths(S, cand, np.full(B, steps))
    assert np.array_equal(p2, full)


def test_block_columns_never_drafts_nothing():
    # dflash2.ts blockColumns: the anchor plus max(1, depth) mask rows, at most the block size;
    # MAX DFlash2Qwen3_5.supports_zero_draft_rows is False. Values worked by hand for G = 16.
    G = 16
    for depth, columns in [(0, 2), (-3, 2), (1, 2), (2, 3), (8, 9), (15, 16), (16, 16), (40, 16)]:
        assert O.block_columns(depth, G) == columns, (depth, columns)


def test_conv_rows_past_depth_do_not_reach_earlier_rows():
    # A block of G rows whose rows past d+1 are arbitrary padding gives, on its first d+1 rows,
    # exactly the conv of the (d+1)-row block: the conv only looks back one row.
    B, G, H, gs, d = 3, 9, 32, 16, 4
    x = _rand(B, G, H)
    y = _rand(B, G, H)
    w = _rand(4 * H // gs, H, scale=0.2)
    base = _rand(2, 2, H)
    out, d1, _ = O.conv_prepare(x, np.ones(H), 1e-6, w, base, gs)
    fin = O.conv_finish(y, d1, base, gs, residual=x)
    out_s, d1_s, _ = O.conv_prepare(x[:, :d + 1], np.ones(H), 1e-6, w, base, gs)
    fin_s = O.conv_finish(y[:, :d + 1], d1_s, base, gs, residual=x[:, :d + 1])
    assert np.array_equal(out[:, :d + 1], out_s)
    assert np.array_equal(fin[:, :d + 1], fin_s)


def test_ragged_tail_is_the_dense_tail_restricted_to_the_drafted_rows():
    # Rows never interact in the head, top-K and z, and a block's walk is causal, so the ragged
    # tail equals the dense tail's rows 1..d_b of each block and select_path_depths' walk.
    B, G, H, gs, V, K, R = 4, 6, 32, 16, 40, 4, 8
    x0 = _rand(B, G, H)

    class Site:
        pass
    s = Site()
    s.w_kp, s.base, s.norm_w, s.y = _rand(4 * H // gs, H, scale=0.2), _rand(2, 2, H), np.ones(H), _rand(B, G, H)
    w_head, w_proj = _rand(V, H), _rand(R, H)
    pred, succ = _rand(V, R), _rand(V, R)
    anchors = RNG.integers(0, V, size=B)
    depths = np.array([5, 0, 2, 9])
    dense = O.block_tail(x0, [s], np.ones(H), 1e-6, gs, w_head, None, w_proj, pred, succ, anchors, K)
    rag = O.block_tail_ragged(x0, [s], np.ones(H), 1e-6, gs, w_head, None, w_proj, pred, succ, anchors, K, depths)
    d = [5, 1, 2, 5]
    assert list(rag["offsets"]) == [0, 5, 6, 8, 13]
    rows = [(b, l) for b in range(B) for l in range(d[b])]
    for i, (b, l) in enumerate(rows):
        np.testing.assert_allclose(rag["h"][i], dense["h"][b, l], rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(rag["cand"][i], dense["cand"][b, l])
        np.testing.assert_allclose(rag["S"][i], dense["S"][b, l], rtol=1e-12, atol=1e-12)
    want, _ = O.select_path_depths(dense["S"], dense["cand"], depths)
    np.testing.assert_array_equal(rag["path"], want)


def test_affine_dequantize_closed_forms():
    # q = 0 gives the bias, q = 15 gives 15 * scale + bias, per row and per group of 64 channels;
    # values worked by hand
    q = np.zeros((2, 128), dtype=np.int64)
    q[0, :64] = 15
    q[1, 64:] = 3
    scales = np.array([[0.5, 2.0], [0.25, 1.5]])
    biases = np.array([[-1.0, 0.25], [0.0, -2.0]])
    W = O.affine_dequantize(q, scales, biases)
    assert np.all(W[0, :64] == 6.5) and np.all(W[0, 64:] == 0.25)
    assert np.all(W[1, :64] == 0.0) and np.all(W[1, 64:] == 2.5)


def test_int4_storage_roundtrip():
    from synth import inputs as I
    q = RNG.integers(0, 16, size=(5, 64))
    w = I.pack_int4(q)
    assert w.shape == (5, 8) and w.dtype == np.uint32
    # code k of a row lives in bits 4 (k % 8) of word k / 8
    assert (w[2, 3] >> 4 * 5) & 15 == q[2, 8 * 3 + 5]
    np.testing.assert_array_equal(I.unpack_int4(w, 64), q)


def test_sublayer_in_identity_and_shift_conv():
    B, G, H, gs, N = 3, 4, 32, 16, 12
    n = _rand(B, G, H)
    W = _rand(N, H)
    d0 = np.zeros((B, G, 2, H // gs))
    ident = np.stack([np.stack([np.ones(H), np.zeros(H)]), np.zeros((2, H))])
    np.testing.assert_allclose(O.sublayer_in(n, d0, ident, gs, W), n @ W.T, rtol=1e-13, atol=1e-13)
    shift = np.stack([np.stack([np.zeros(H), np.ones(H)]), np.zeros((2, H))])
    prev = np.zeros_like(n)
    for b in range(B):             # the previous row of each block, a zero row before the block
        for t in range(1, G):
            prev[b, t] = n[b, t - 1]
    np.testing.assert_allclose(O.sublayer_in(n, d0, shift, gs, W), prev @ W.T, rtol=1e-13, atol=1e-13)


def test_sublayer_out_applies_the_projection_before_the_conv():
    # With W a permutation of the channels, the conv acts on the permuted channels (the projection
    # comes first); a zero W leaves the residual.
    B, G, H, gs = 2, 5, 32, 16
    a = _rand(B, G, H)
    d1 = _rand(B, G, 2, H // gs, scale=0.3)
    base = _rand(2, 2, H)
    perm = RNG.permutation(H)
    P = np.eye(H)[perm]            # (a @ P.T)[..., j] = a[..., perm[j]]
    got = O.sublayer_out(a, P, d1, base, gs)
    np.testing.assert_allclose(got, O.conv_finish(a[..., perm], d1, base, gs), rtol=1e-12, atol=1e-12)
    res = _rand(B, G, H)
    np.testing.assert_array_equal(O.sublayer_out(a, np.zeros((H, H)), d1, base, gs, residual=res), res)
