"""Comparison rules of the GPU-vs-oracle parity tests.

* Floating-point outputs: max |gpu - oracle| <= REL_TOL * max |oracle| over the tensor
  (REL_TOL = 2e-2, "within max-abs 2e-2 relative to the output scale").
* Top-K candidate ids: for each row, if the oracle's K-th minus (K+1)-th logit exceeds
  4 * tol the GPU's id set must equal the oracle's exactly; adjacent positions i, i+1 must be
  in the oracle's order where their gap exceeds 4 * tol. Rows under the margin are near-ties:
  counted, and checked for validity only (every GPU id's oracle logit is within 4 * tol of the
  oracle's K-th value, and the GPU's values equal the oracle's logits at the GPU's ids).
* The walk: slot by slot, while the oracle's best-minus-second margin of the row it reads
  exceeds 4 * tol the chosen id must match. At the first near-tie slot of a block the GPU's
  choice must be one of the near-maximal candidates (its oracle score within 4 * tol of the
  best); that slot ends the strict comparison for the block (counted).
* End to end (the GPU's whole tail against the oracle's own walk, each on its own candidates):
  the same, with a slot also ending the strict comparison when its head row is a near-tie.
* Counts of near-tie rows, blocks and strictly compared slots are recorded with ``record`` and
  printed at the end of the test session.
"""
from __future__ import annotations

import numpy as np

REL_TOL = 2e-2


def scale_of(ref) -> float:
    return float(np.max(np.abs(ref))) if np.size(ref) else 1.0


def assert_close_scaled(got, ref, rel=REL_TOL, what="tensor"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    s = scale_of(ref)
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err <= rel * s, f"{what}: max abs err {err:.4g} > {rel} * scale {s:.4g}"
    return err / s if s else err


def compare_topk(gpu_ids, gpu_vals, ref_logits, K, tol):
    """Check per-row top-K ids/values against the oracle's logits. Returns the number of near-tie rows."""
    gpu_ids = np.asarray(gpu_ids).reshape(-1, K)
    gpu_vals = np.asarray(gpu_vals, dtype=np.float64).reshape(-1, K)
    L = np.asarray(ref_logits, dtype=np.float64).reshape(gpu_ids.shape[0], -1)
    near = 0
    for r in range(L.shape[0]):
        row = L[r]
        order = np.argsort(-row, kind="stable")
        ref_ids = order[:K]
        vk = row[order[K - 1]]
        margin = vk - row[order[K]] if row.size > K else np.inf
        ids = gpu_ids[r]
        assert np.all((ids >= 0) & (ids < row.size)), f"row {r}: id out of range {ids}"
        assert len(set(ids.tolist())) == K, f"row {r}: duplicate ids {ids}"
        # values are the logits of the ids the GPU chose
        assert np.max(np.abs(gpu_vals[r] - row[ids])) <= tol, f"row {r}: unary differs from the logits at its ids"
        # descending order of the GPU's own values
        assert np.all(np.diff(gpu_vals[r]) <= 0), f"row {r}: values not descending {gpu_vals[r]}"
        if margin > 4 * tol:
            assert set(ids.tolist()) == set(ref_ids.tolist()), f"row {r}: id set differs (margin {margin:.3g})"
            for i in range(K - 1):
                gap = row[ref_ids[i]] - row[ref_ids[i + 1]]
                if gap > 4 * tol:
                    pos_a = int(np.where(ids == ref_ids[i])[0][0])
                    pos_b = int(np.where(ids == ref_ids[i + 1])[0][0])
                    assert pos_a < pos_b, f"row {r}: order of ids {ref_ids[i]}, {ref_ids[i + 1]}"
        else:
            near += 1
            assert np.all(row[ids] >= vk - 4 * tol), f"row {r}: near-tie row holds an id far below the K-th value"
    return near


def compare_walk(gpu_path, ref_S, ref_pos, cand, tol):
    """Strict slot-by-slot comparison of a walk over the same candidates (cand [B, steps, K]) as
    the oracle's S, until the first near-tie of each block, where the GPU's choice must score
    within 4 * tol of the row's best. Returns (near_tie_blocks, slots_checked)."""
    gpu_path = np.asarray(gpu_path)
    S = np.asarray(ref_S, dtype=np.float64)
    cand = np.asarray(cand)
    B, steps, K, _ = S.shape
    near, checked = 0, 0
    for b in range(B):
        p = 0
        for l in range(steps):
            row = S[b, l, p]
            best = int(ref_pos[b, l])
            second = np.max(np.delete(row, best)) if K > 1 else -np.inf
            g = int(gpu_path[b, l])
            if row[best] - second <= 4 * tol:
                near += 1
                hit = np.flatnonzero(cand[b, l] == g)
                assert hit.size == 1, f"block {b} slot {l}: GPU id {g} is not a candidate"
                assert row[hit[0]] >= row[best] - 4 * tol, \
                    f"block {b} slot {l}: near-tie choice {g} scores {row[hit[0]]:.4g}, best {row[best]:.4g}"
                break
            assert g == int(cand[b, l, best]), f"block {b} slot {l}: {g} != {int(cand[b, l, best])}"
            checked += 1
            p = best
    return near, checked


def _edge_scores(ids, prev_id, z_row, pred_book, succ_book):
    """Oracle edge term sum_r pred[prev, r] * z[r] * succ[u, r] for each id u (float64)."""
    w = np.asarray(pred_book[int(prev_id)], dtype=np.float64) * np.asarray(z_row, dtype=np.float64)
    rows = np.stack([np.asarray(succ_book[int(u)], dtype=np.float64) for u in ids])
    return rows @ w


def path_parity(gpu_path, ref, anchors, pred_book, succ_book, logits_tol, S_tol, strict=True):
    """The GPU's path against the oracle's own walk (``ref`` = the oracle's block_tail dict), each
    on its own candidates, under the stated margins.

    A slot is decided when the oracle's choice c* is certainly in any top-K the tolerance allows
    (its logit exceeds the (K+1)-th by more than 4 * logits_tol) and its oracle score
    unary + edge beats, by more than 4 * S_tol, every other id that may be a candidate (logit at
    least the K-th minus 4 * logits_tol), scored with the same predecessor. Decided slots must give
    the oracle's id; the first undecided slot of a block must give a valid choice (an id that may
    be a candidate, scoring within 4 * S_tol of c*) and ends the block's comparison (predecessors
    may differ after it). Returns dict(near_tie_blocks, strict_slots, mismatches); with
    strict=True a mismatch raises instead of being counted."""
    gpu_path = np.asarray(gpu_path)
    logits, z, path = ref["logits"], ref["z"], ref["path"]
    B, steps = path.shape
    K = ref["cand"].shape[-1]
    out = dict(near_tie_blocks=0, strict_slots=0, mismatches=0)
    for b in range(B):
        prev = int(anchors[b])
        for l in range(steps):
            L = np.asarray(logits[b, l], dtype=np.float64)
            srt = -np.sort(-L)
            vK, vK1 = srt[K - 1], (srt[K] if L.size > K else -np.inf)
            possible = np.flatnonzero(L >= vK - 4 * logits_tol)
            score = L[possible] + _edge_scores(possible, prev, z[b, l], pred_book, succ_book)
            best_id = int(path[b, l])
            best = float(score[possible == best_id][0])
            others = score[possible != best_id]
            runner_up = float(np.max(others)) if others.size else -np.inf
            g = int(gpu_path[b, l])
            decided = L[best_id] > vK1 + 4 * logits_tol and best - runner_up > 4 * S_tol
            if not decided:
                out["near_tie_blocks"] += 1
                ok = g in set(possible.tolist()) and float(score[possible == g][0]) >= best - 4 * S_tol
                if not ok:
                    out["mismatches"] += 1
                    assert not strict, f"block {b} slot {l}: near-tie choice {g} is not a valid candidate/score"
                break
            if g != best_id:
                out["mismatches"] += 1
                assert not strict, f"block {b} slot {l}: {g} != {best_id} (end to end, decided slot)"
                break
            out["strict_slots"] += 1
            prev = best_id
    return out


REPORT = []


def record(name, **counts):
    """Keep a test's near-tie counts; conftest prints them when the session ends."""
    REPORT.append((name, counts))
