"""The GPU-vs-oracle comparison rule itself (tests/helpers.py), on the CPU.

Each case starts from the oracle's own answer for a small random problem,
which must pass, then plants one mistake a kernel could make and checks
that the rule rejects it: indices permuted against their scores, a score
off by more than the tolerance, a padded slot in the wrong place, a
duplicated index, and an index swapped for a clearly smaller one.  A
swap across a genuine near-tie (the k-th and (k+1)-th oracle scores closer
than the tolerance) must still pass.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dsa_inputs import Workload, make_inputs
from tests.helpers import compare_topk_row, score_tol


def _case(topk=12, S=40, S_kv=40):
    wl = Workload("t", B=1, S=S, S_kv=S_kv, H=8, D=32, compress_ratio=1,
                  topk=topk, w_scale=8 ** -0.5, seed=123)
    q, k, w, _ = make_inputs(wl)
    ref = oracle.indexer_fwd(q, k, w, 1, topk, want_logits=True)
    return ref


def _row(ref, r):
    return (ref["idx"][r].copy(), ref["scores"][r].astype(np.float32).copy(),
            ref["idx"][r], ref["scores64"][r], ref["next"][r],
            ref["logits"][r])


def test_oracle_answer_passes():
    ref = _case()
    for r in range(ref["idx"].shape[0]):
        gi, gs, oi, os_, on, L = _row(ref, r)
        assert compare_topk_row(gi, gs, oi, os_, on, L) is None


def test_indices_permuted_against_scores_fail():
    ref = _case()
    r = 39  # 40 visible keys, 12 kept
    gi, gs, oi, os_, on, L = _row(ref, r)
    # same index set, same sorted scores, but the first two indices swapped
    gi[[0, 1]] = gi[[1, 0]]
    assert abs(L[gi[0]] - L[gi[1]]) > score_tol(L[gi[0]])
    msg = compare_topk_row(gi, gs, oi, os_, on, L)
    assert msg is not None and "not the score of its index" in msg
    # a rotation of all kept indices fails the same way
    gi, gs, oi, os_, on, L = _row(ref, r)
    gi[:12] = np.roll(gi[:12], 1)
    assert compare_topk_row(gi, gs, oi, os_, on, L) is not None


def test_score_outside_tolerance_fails():
    ref = _case()
    gi, gs, oi, os_, on, L = _row(ref, 39)
    gs[3] = np.float32(gs[3] + 2 * score_tol(gs[3]))
    assert compare_topk_row(gi, gs, oi, os_, on, L) is not None


def test_padding_and_duplicates_fail():
    ref = _case()
    # row 5 sees 6 keys: slots 6.. are padded
    gi, gs, oi, os_, on, L = _row(ref, 5)
    gi[6] = 0
    assert compare_topk_row(gi, gs, oi, os_, on, L) is not None
    gi, gs, oi, os_, on, L = _row(ref, 39)
    gi[1] = gi[0]
    gs[1] = gs[0]
    assert compare_topk_row(gi, gs, oi, os_, on, L) is not None


def test_clearly_smaller_index_fails_near_tie_swap_passes():
    ref = _case()
    gi, gs, oi, os_, on, L = _row(ref, 39)
    # replace the k-th index by the smallest visible key, with its own score
    worst = int(np.argmin(np.where(np.isfinite(L), L, np.inf)))
    gi[11] = worst
    gs[11] = np.float32(L[worst])
    assert compare_topk_row(gi, gs, oi, os_, on, L) is not None
    # a near-tie: the (k+1)-th oracle key moved to within the tolerance of
    # the k-th; swapping the two is then allowed
    gi, gs, oi, os_, on, L = _row(ref, 39)
    L = L.copy()
    order = np.argsort(-L, kind="stable")
    kth, nxt = int(order[11]), int(order[12])
    L[nxt] = L[kth] - 0.25 * score_tol(L[kth])
    gi[11] = nxt
    gs[11] = np.float32(L[nxt])
    assert compare_topk_row(gi, gs, oi, os_, L[nxt], L) is None


def test_rule_helpers_agree_with_torch_topk_on_distinct_scores():
    """Independent cross-check of the oracle's selection on one row: the
    order of the kept scores equals torch.topk over the row's visible
    logits (all distinct on random inputs)."""
    ref = _case()
    L = torch.from_numpy(ref["logits"][39])
    vals, ids = torch.topk(L, 12)
    np.testing.assert_array_equal(ids.numpy(), ref["idx"][39])
    np.testing.assert_allclose(vals.numpy(), ref["scores64"][39])
