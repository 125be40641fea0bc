"""Shared test helpers: closed forms and the GPU-vs-oracle comparison rule.

Nothing here calls the CUDA library; nothing here is imported by the product.
"""
from __future__ import annotations

import math

import numpy as np


def n_visible_closed_form(t: int, ratio: int, S_kv: int) -> int:
    """Number of compressed keys visible at position t.

    Key j is visible iff (j+1)*r - 1 <= t, i.e. j < floor((t+1)/r); the
    count is clamped to [0, S_kv].
    """
    if t < 0:
        return 0
    return max(0, min(S_kv, (t + 1) // ratio))


def score_tol(o):
    """Score tolerance: |gpu - oracle| <= 1e-3 + 2e-3 * |oracle|."""
    return 1e-3 + 2e-3 * np.abs(o)


def compare_topk_row(g_idx, g_sc, o_idx, o_sc64, o_next, logits64,
                     extra=None):
    """Compare one row of GPU top-k output with the oracle's.

    g_idx/g_sc: GPU indices (int32) and scores (fp32) for the row.
    o_idx/o_sc64: oracle indices and fp64 scores; o_next: the oracle's
    (topk+1)-th visible score (-inf if there is none).  logits64: the
    oracle's full fp64 row (-inf where invisible), used to look up the
    oracle score of every GPU index.  extra: None, or an allowance per key
    of the row (same shape as logits64) added to the tolerance of that key's
    score, for inputs the two sides may legitimately round differently; the
    largest allowance over the row widens the slot-by-slot and near-tie
    margins.

    Returns None when the row matches, else a message.
    Rule: the -1 slots match exactly; scores agree slot by slot within the
    tolerance; every returned score is the oracle score of the index
    returned in the same slot, within the tolerance (so an output whose
    indices are permuted against its scores fails); index sets are equal
    when the oracle's k-th and (k+1)-th scores are at least a tolerance
    apart, otherwise every oracle index scored clearly above the k-th is
    kept and every GPU index scores at least the k-th minus the tolerance.
    """
    g_idx = np.asarray(g_idx)
    g_sc = np.asarray(g_sc, dtype=np.float64)
    o_idx = np.asarray(o_idx)
    o_sc = np.asarray(o_sc64, dtype=np.float64)
    if not np.array_equal(g_idx == -1, o_idx == -1):
        return f"-1 slots differ: gpu {np.sum(g_idx == -1)} oracle {np.sum(o_idx == -1)}"
    valid = o_idx != -1
    L = np.asarray(logits64, dtype=np.float64)
    E = np.zeros_like(L) if extra is None else np.asarray(extra, np.float64)
    fin = np.isfinite(L)
    emax = float(E[fin].max()) if np.any(fin) else 0.0
    if not np.all(np.isneginf(g_sc[~valid])):
        return "padded slot score is not -inf"
    if np.any(~np.isfinite(g_sc[valid])):
        return "non-finite score in a valid slot"
    err = np.abs(g_sc[valid] - o_sc[valid])
    bad = err > score_tol(o_sc[valid]) + emax
    if np.any(bad):
        i = int(np.flatnonzero(bad)[0])
        return f"score slot {i}: gpu {g_sc[valid][i]!r} oracle {o_sc[valid][i]!r}"
    gv = g_idx[valid]
    if len(set(gv.tolist())) != gv.size:
        return "duplicate indices"
    if gv.size and (gv.min() < 0 or gv.max() >= L.size):
        return "index outside the row"
    own = L[gv]
    pair_bad = ~(np.abs(g_sc[valid] - own) <= score_tol(own) + E[gv])
    if np.any(pair_bad):
        i = int(np.flatnonzero(pair_bad)[0])
        return (f"slot {i}: score {g_sc[valid][i]!r} is not the score of its "
                f"index {int(gv[i])} (oracle {own[i]!r})")
    ov = o_idx[valid]
    if ov.size == 0:
        return None
    kth = o_sc[valid][-1]
    tol = score_tol(kth) + 2.0 * emax
    if math.isinf(o_next) or kth - o_next >= tol:
        if set(gv.tolist()) != set(ov.tolist()):
            return "index sets differ away from a near-tie"
        return None
    must = set(ov[o_sc[valid] > kth + tol].tolist())
    if not must.issubset(set(gv.tolist())):
        return "near-tie row dropped a clearly larger index"
    if np.any(L[gv] < kth - tol):
        return "near-tie row kept an index scored clearly below the k-th"
    return None
