"""Comparison rules of the GPU-vs-oracle parity tests.

* Floating-point outputs: max |gpu - oracle| <= REL_TOL * max |oracle| over the tensor
  (REL_TOL = 2e-2, "within max-abs 2e-2 relative to the output scale").
* Top-K candidate ids: for each row, if the oracle's K-th minus (K+1)-th logit exceeds
  4 * tol the GPU's id set must equal the oracle's exactly; adjacent positions i, i+1 must be
  in the oracle's order where their gap exceeds 4 * tol. Rows under the margin are near-ties:
  counted, and checked for validity only (every GPU id's oracle logit is within 4 * tol of the
  oracle's K-th value, and the GPU's values equal the oracle's logits at the GPU's ids).
* The walk: slot by slot, while the oracle's best-minus-second margin of the row it reads
  exceeds 4 * tol the chosen id must match; the first near-tie ends the strict comparison for
  that block (counted).
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


def compare_walk(gpu_path, ref_path, ref_margins, tol):
    """Strict slot-by-slot comparison until the first near-tie of each block. Returns (near_tie_blocks, slots_checked)."""
    gpu_path = np.asarray(gpu_path)
    ref_path = np.asarray(ref_path)
    near, checked = 0, 0
    for b in range(ref_path.shape[0]):
        for l in range(ref_path.shape[1]):
            if ref_margins[b, l] <= 4 * tol:
                near += 1
                break
            assert gpu_path[b, l] == ref_path[b, l], f"block {b} slot {l}: {gpu_path[b, l]} != {ref_path[b, l]}"
            checked += 1
    return near, checked
