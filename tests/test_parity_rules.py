"""The comparison rules of the GPU parity tests, checked on the CPU: the oracle's own results
pass them, and planted mistakes (a wrong id at a decided slot, an invalid near-tie choice) fail."""
import numpy as np
import pytest

from oracle import dflash2_oracle as O
from tests.parity import compare_walk, path_parity, scale_of

RNG = np.random.default_rng(11)


def _selector(B=6, steps=5, K=4, R=8, V=40):
    cand = np.stack([np.stack([RNG.choice(V, size=K, replace=False) for _ in range(steps)]) for _ in range(B)])
    unary = -np.sort(-RNG.standard_normal((B, steps, K)), axis=-1)
    z = RNG.standard_normal((B, steps, R))
    anchors = RNG.integers(0, V, size=B)
    S = O.score_edges(cand, unary, z, anchors, RNG.standard_normal((V, R)), RNG.standard_normal((V, R)))
    return cand, S


def test_compare_walk_accepts_the_oracle_and_rejects_a_wrong_decided_id():
    cand, S = _selector()
    path, pos = O.select_path(S, cand)
    tol = 1e-6 * scale_of(S)
    near, checked = compare_walk(path, S, pos, cand, tol)
    assert near == 0 and checked == path.size
    bad = path.copy()
    bad[2, 3] = cand[2, 3, (pos[2, 3] + 1) % cand.shape[2]]
    with pytest.raises(AssertionError):
        compare_walk(bad, S, pos, cand, tol)


def test_compare_walk_near_tie_choice_must_be_near_maximal():
    cand, S = _selector(B=1, steps=3, K=4)
    S = S.copy()
    S[0, 0, 0, :] = [1.0, 0.99995, -5.0, 0.2]   # slot 0: positions 0 and 1 tie within 4 * tol
    path, pos = O.select_path(S, cand)
    tol = 1e-4
    alt = path.copy()
    alt[0, 0] = cand[0, 0, 1]                   # the other near-maximal candidate: valid
    near, checked = compare_walk(alt, S, pos, cand, tol)
    assert near == 1 and checked == 0
    alt[0, 0] = cand[0, 0, 2]                   # far below the best: invalid
    with pytest.raises(AssertionError):
        compare_walk(alt, S, pos, cand, tol)


def test_end_to_end_rule_on_the_oracle_tail():
    B, steps, K, R, V, H = 3, 4, 3, 8, 30, 16
    h = RNG.standard_normal((B, steps, H))
    W = RNG.standard_normal((V, H))
    logits = O.head_logits(h, W)
    cand, unary = O.top_k(logits, K)
    z = RNG.standard_normal((B, steps, R))
    anchors = RNG.integers(0, V, size=B)
    pred, succ = RNG.standard_normal((V, R)), RNG.standard_normal((V, R))
    S = O.score_edges(cand, unary, z, anchors, pred, succ)
    path, pos = O.select_path(S, cand)
    ref = dict(cand=cand, S=S, pos=pos, logits=logits, path=path, z=z)
    r = path_parity(path, ref, anchors, pred, succ, 1e-9, 1e-9)
    assert r["near_tie_blocks"] == 0 and r["strict_slots"] == path.size and r["mismatches"] == 0
    bad = path.copy()
    others = np.setdiff1d(np.arange(V), cand[1, 2])
    bad[1, 2] = others[0]                       # an id outside a decided candidate set
    with pytest.raises(AssertionError):
        path_parity(bad, ref, anchors, pred, succ, 1e-9, 1e-9)
    assert path_parity(bad, ref, anchors, pred, succ, 1e-9, 1e-9, strict=False)["mismatches"] == 1
    # with a tolerance wider than every gap no slot is decided: the first slot of each block is
    # checked for validity only (the oracle's own choice is valid)
    r = path_parity(path, ref, anchors, pred, succ, 1e9, 1e9)
    assert r["near_tie_blocks"] == B and r["strict_slots"] == 0 and r["mismatches"] == 0
