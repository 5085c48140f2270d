"""Comparison rules shared by the parity tests (no layer arithmetic here).

Tolerances (stated once, used everywhere):
  * expert IDs: exact, in rank order, for every token whose oracle decision
    gap (10th minus 11th logit) exceeds GAP_TOL = 1e-3; tokens at or below it
    are counted and reported, not failed.  Inside the route, two adjacent ranks
    may swap only if their oracle logits are within GAP_TOL.
  * route weights: |w_gpu - w_ref| <= W_ATOL = 1e-5 where IDs match.
  * layer / expert outputs: max|gpu - ref| <= 1e-2 * max|ref| and
    mean|gpu - ref| / mean|ref| <= 5e-3.
  * integer outputs (counts, offsets, permutations, masks, U, bytes): exact.
"""
from __future__ import annotations

import numpy as np

GAP_TOL = 1e-3
W_ATOL = 1e-5
MAX_ABS_FRAC = 1e-2
MEAN_REL = 5e-3


def compare_routes(ids_gpu, w_gpu, ids_ref, w_ref, gap_ref, logits_ref):
    """Returns a report dict; raises AssertionError on a real mismatch."""
    ids_gpu = np.asarray(ids_gpu)
    ids_ref = np.asarray(ids_ref)
    T, k = ids_ref.shape
    near_tie = 0
    rank_swaps = 0
    checked = 0
    match_rows = []
    for t in range(T):
        if not gap_ref[t] > GAP_TOL:
            near_tie += 1
            continue
        checked += 1
        g, r = list(ids_gpu[t]), list(ids_ref[t])
        assert set(g) == set(r), f"token {t}: expert set differs (gap {gap_ref[t]:.3e}): {g} vs {r}"
        if g != r:
            # every displaced expert must be within GAP_TOL of the one in its place
            for j in range(k):
                if g[j] != r[j]:
                    d = abs(float(logits_ref[t, g[j]]) - float(logits_ref[t, r[j]]))
                    assert d <= GAP_TOL, f"token {t}: rank {j} swap with logit gap {d:.3e}"
            rank_swaps += 1
            continue
        match_rows.append(t)
        dw = np.abs(np.asarray(w_gpu[t], np.float64) - np.asarray(w_ref[t], np.float64)).max()
        assert dw <= W_ATOL, f"token {t}: weight error {dw:.3e}"
    return {"checked": checked, "near_tie": near_tie, "rank_swaps": rank_swaps, "exact_rows": match_rows}


def compare_route_ids(ids_gpu, ids_ref, gap_ref, logits_ref):
    """compare_routes for a route whose weights are not kept (IDs only)."""
    w = np.zeros(np.asarray(ids_ref).shape, np.float32)
    return compare_routes(ids_gpu, w, ids_ref, w, gap_ref, logits_ref)


def output_errors(out, ref):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = np.abs(out - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    ref_max = float(np.abs(ref).max()) if ref.size else 0.0
    mean_rel = float(diff.mean() / np.abs(ref).mean()) if ref.size else 0.0
    return max_abs, ref_max, mean_rel


def assert_output_close(out, ref, what="output"):
    max_abs, ref_max, mean_rel = output_errors(out, ref)
    assert max_abs <= MAX_ABS_FRAC * ref_max, f"{what}: max|err| {max_abs:.3e} > 1e-2 * max|ref| {ref_max:.3e}"
    assert mean_rel <= MEAN_REL, f"{what}: mean relative error {mean_rel:.3e} > 5e-3"
    return max_abs / max(ref_max, 1e-30), mean_rel
