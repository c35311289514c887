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


def compare_path_end_to_end(gpu_path, ref, logits_tol, S_tol):
    """The GPU's path against the oracle's own walk (``ref`` = the oracle's block_tail dict), each
    on its own candidates. Slot by slot the ids must match while the oracle's head row of that
    slot has a K-th margin above 4 * logits_tol and its walk margin exceeds 4 * S_tol. At the
    first slot that is a near-tie either way, the GPU's id g must be a valid choice: if g is an
    oracle candidate, its oracle score is within 4 * S_tol of the best; otherwise the row must be
    a head near-tie (only then may the candidate sets differ). That slot ends the block's strict
    comparison. Returns (near_tie_blocks, slots_checked)."""
    gpu_path = np.asarray(gpu_path)
    cand, S, pos, logits = ref["cand"], ref["S"], ref["pos"], ref["logits"]
    B, steps, K = cand.shape
    near, checked = 0, 0
    for b in range(B):
        p = 0
        for l in range(steps):
            row_logits = logits[b, l]
            srt = -np.sort(-row_logits)
            head_margin = srt[K - 1] - srt[K] if row_logits.size > K else np.inf
            row = S[b, l, p]
            best = int(pos[b, l])
            second = np.max(np.delete(row, best)) if K > 1 else -np.inf
            g = int(gpu_path[b, l])
            if head_margin <= 4 * logits_tol or row[best] - second <= 4 * S_tol:
                near += 1
                hit = np.flatnonzero(cand[b, l] == g)
                if hit.size:
                    assert row[hit[0]] >= row[best] - 4 * S_tol, \
                        f"block {b} slot {l}: near-tie choice {g} scores {row[hit[0]]:.4g}, best {row[best]:.4g}"
                else:
                    assert head_margin <= 4 * logits_tol, \
                        f"block {b} slot {l}: GPU id {g} is not an oracle candidate of a decided row"
                    assert row_logits[g] >= srt[K - 1] - 4 * logits_tol, \
                        f"block {b} slot {l}: GPU id {g} lies far below the oracle's K-th logit"
                break
            assert g == int(ref["path"][b, l]), f"block {b} slot {l}: {g} != {int(ref['path'][b, l])} (end to end)"
            checked += 1
            p = best
    return near, checked


REPORT = []


def record(name, **counts):
    """Keep a test's near-tie counts; conftest prints them when the session ends."""
    REPORT.append((name, counts))
