"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: a hand-worked
example, a library routine that the definition reduces to in a special case,
exact rational brute force, closed forms and invariants.  The plausible
mistakes each one catches are named in its docstring.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dsa_inputs import WORKLOADS, Workload, make_given_indices, make_inputs
from tests.helpers import n_visible_closed_form

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example.txt")


def _f(s: str) -> float:
    return -math.inf if s == "-inf" else float(s)


def load_hand_example():
    q = np.zeros((5, 1, 2, 2), np.float32)
    k = np.zeros((4, 1, 2), np.float32)
    w = np.zeros((5, 1, 2), np.float32)
    topk, gather = [], []
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *v = line.split()
            if tag == "q":
                t, h, a, b = v
                q[int(t), 0, int(h)] = (float(a), float(b))
            elif tag == "k":
                j, a, b = v
                k[int(j), 0] = (float(a), float(b))
            elif tag == "w":
                t, a, b = v
                w[int(t), 0] = (float(a), float(b))
            elif tag == "topk":
                r, t, i0, i1, s0, s1 = v
                topk.append((int(r), int(t), [int(i0), int(i1)], [_f(s0), _f(s1)]))
            elif tag == "gather":
                t, i0, i1, s0, s1 = v
                gather.append((int(t), [int(i0), int(i1)], [_f(s0), _f(s1)]))
    to_bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    return to_bf(q), to_bf(k), torch.from_numpy(w), topk, gather


def test_hand_example_topk():
    """Hand-derived values: pins the head sum, ReLU, w multiply, the causal
    rule at r = 1, 2, 4, the tie order (three-way tie at t=3) and padding."""
    q, k, w, topk, _ = load_hand_example()
    for r in (1, 2, 4):
        out = oracle.indexer_fwd(q, k, w, r, 2)
        for rr, t, idx, sc in topk:
            if rr != r:
                continue
            assert out["idx"][t].tolist() == idx, (r, t, out["idx"][t])
            assert out["scores"][t].tolist() == sc, (r, t, out["scores"][t])


def test_hand_example_gather():
    """Hand-derived given-indices values: -1, invisible and out-of-range
    indices give -inf; indices are returned unchanged."""
    q, k, w, _, gather = load_hand_example()
    in_idx = torch.tensor([[g[1] for g in gather]], dtype=torch.int32)
    out = oracle.indexer_fwd(q, k, w, 1, 2, in_idx=in_idx)
    for t, idx, sc in gather:
        assert out["idx"][t].tolist() == idx
        assert out["scores"][t].tolist() == sc


def _rand_problem(S, B, H, D, S_kv, seed, w_scale=0.5):
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=1,
                  topk=4, w_scale=w_scale, seed=seed)
    q, k, w, _ = make_inputs(wl)
    return q, k, w


def test_single_head_unit_weight_is_relu_of_matmul():
    """H=1, w=1, r=1: I = ReLU(Q K^T) under a lower-triangular mask.  Checked
    against numpy's matmul; catches a transposed operand, a wrong q or k
    stride, or a wrong mask direction."""
    S, B, H, D = 40, 2, 1, 24
    q, k, _ = _rand_problem(S, B, H, D, S, seed=7)
    w = torch.ones((S, B, H), dtype=torch.float32)
    out = oracle.indexer_fwd(q, k, w, 1, 4, want_logits=True)
    L = out["logits"].reshape(B, S, S)
    qd = q.float().double().numpy()
    kd = k.float().double().numpy()
    for b in range(B):
        ref = np.maximum(qd[:, b, 0, :] @ kd[:, b, :].T, 0.0)
        mask = np.tril(np.ones((S, S), bool))
        ref = np.where(mask, ref, -np.inf)
        np.testing.assert_allclose(L[b], ref, rtol=1e-12, atol=1e-12)


def test_relu_odd_part_is_linear():
    """ReLU(x) - ReLU(-x) = x, so I(q) - I(-q) = (sum_h w_h q_h) . k_j, a
    plain matmul.  Catches a dropped head, a wrong w index, a sign error and
    a wrong batch stride (B=2, H=3)."""
    S, B, H, D = 24, 2, 3, 16
    q, k, w = _rand_problem(S, B, H, D, S, seed=8)
    a = oracle.indexer_fwd(q, k, w, 1, 4, want_logits=True)["logits"]
    b_ = oracle.indexer_fwd(-q, k, w, 1, 4, want_logits=True)["logits"]
    with np.errstate(invalid="ignore"):
        diff = (a - b_).reshape(B, S, S)
    qd = q.float().double().numpy()
    kd = k.float().double().numpy()
    wd = w.double().numpy()
    for b in range(B):
        qbar = np.einsum("sh,shd->sd", wd[:, b, :], qd[:, b, :, :])
        ref = qbar @ kd[:, b, :].T
        mask = np.tril(np.ones((S, S), bool))
        np.testing.assert_allclose(diff[b][mask], ref[mask], rtol=1e-10,
                                   atol=1e-10)


def test_batches_are_independent():
    """The oracle on a B=2 problem equals the oracle on each batch alone.
    Catches a batch/sequence stride mix-up in the SBHD layouts."""
    S, B, H, D = 20, 2, 4, 8
    q, k, w = _rand_problem(S, B, H, D, S, seed=9)
    both = oracle.indexer_fwd(q, k, w, 1, 5, want_logits=True)
    for b in range(B):
        one = oracle.indexer_fwd(q[:, b:b + 1].contiguous(),
                                 k[:, b:b + 1].contiguous(),
                                 w[:, b:b + 1].contiguous(), 1, 5,
                                 want_logits=True)
        sl = slice(b * S, (b + 1) * S)
        np.testing.assert_array_equal(both["logits"][sl], one["logits"])
        np.testing.assert_array_equal(both["idx"][sl], one["idx"])


def test_head_permutation_invariance():
    """Permuting heads of q and w together leaves I unchanged; permuting
    only w changes it (so w really is indexed per head)."""
    S, B, H, D = 16, 1, 6, 8
    q, k, w = _rand_problem(S, B, H, D, S, seed=10)
    perm = torch.tensor([3, 0, 5, 1, 4, 2])
    L0 = oracle.indexer_fwd(q, k, w, 1, 3, want_logits=True)["logits"]
    L1 = oracle.indexer_fwd(q[:, :, perm].contiguous(), k,
                            w[:, :, perm].contiguous(), 1, 3,
                            want_logits=True)["logits"]
    L2 = oracle.indexer_fwd(q, k, w[:, :, perm].contiguous(), 1, 3,
                            want_logits=True)["logits"]
    fin = np.isfinite(L0)
    np.testing.assert_allclose(L1[fin], L0[fin], rtol=1e-12, atol=1e-12)
    assert not np.allclose(L2[fin], L0[fin])


@pytest.mark.parametrize("ratio", [1, 2, 3, 4, 7])
def test_visible_counts_closed_form(ratio):
    """Visible-key count and -1 padding count follow the closed forms
    n_vis = clamp(floor((t+1)/r), 0, S_kv), pad = max(0, topk - n_vis)."""
    S, B, H, D, S_kv, topk = 50, 1, 2, 8, 9, 5
    q, k, w = _rand_problem(S, B, H, D, S_kv, seed=11)
    out = oracle.indexer_fwd(q, k, w, ratio, topk, want_logits=True)
    for t in range(S):
        n = n_visible_closed_form(t, ratio, S_kv)
        assert out["nvis"][t] == n
        assert np.sum(np.isfinite(out["logits"][t])) == n
        assert np.all(np.isfinite(out["logits"][t][:n]))
        assert np.sum(out["idx"][t] == -1) == max(0, topk - n)
        for j in range(S_kv):
            assert oracle.key_visible(j, t, ratio) == (j < n)


def test_decode_position_matches_prefill_row():
    """A decode row at q_pos = p scores like prefill row p of the same
    query: pins the q_pos reading pos = q_pos[b] + s."""
    S, B, H, D, S_kv, r = 37, 1, 4, 16, 9, 4
    q, k, w = _rand_problem(S, B, H, D, S_kv, seed=12)
    pre = oracle.indexer_fwd(q, k, w, r, 6, want_logits=True)
    for p in (0, 3, 4, 18, 36):
        dec = oracle.indexer_fwd(q[p:p + 1].contiguous(), k,
                                 w[p:p + 1].contiguous(), r, 6,
                                 q_pos=torch.tensor([p], dtype=torch.int32),
                                 want_logits=True)
        np.testing.assert_array_equal(dec["logits"][0], pre["logits"][p])
        np.testing.assert_array_equal(dec["idx"][0], pre["idx"][p])


def _exact_scores(qi, ki, wi, ratio, b, s, t):
    """Exact rational I[t, j] for integer q, k and dyadic w, by brute force."""
    S, B, H, D = qi.shape
    S_kv = ki.shape[0]
    out = {}
    for j in range(S_kv):
        if (j + 1) * ratio - 1 > t:
            continue
        tot = Fraction(0)
        for h in range(H):
            dot = sum(int(qi[s, b, h, d]) * int(ki[j, b, d]) for d in range(D))
            tot += Fraction(wi[s, b, h]) * max(dot, 0)
        out[j] = tot
    return out


@pytest.mark.parametrize("ratio,topk", [(1, 6), (2, 4), (4, 3), (1, 40)])
def test_integer_inputs_match_exact_brute_force(ratio, topk):
    """Integer q, k in [-3, 3] and w in {+-1, +-1/2, +-1/4}: every score is
    exact, ties are frequent.  The oracle must equal exact rational brute
    force with k rounds of argmax (lowest j wins a tie), bit for bit."""
    rng = np.random.default_rng(123 + ratio)
    S, B, H, D, S_kv = 30, 2, 3, 5, 12
    qi = rng.integers(-3, 4, size=(S, B, H, D))
    ki = rng.integers(-3, 4, size=(S_kv, B, D))
    wi = rng.choice([1, -1, 0.5, -0.5, 0.25, -0.25], size=(S, B, H))
    q = torch.from_numpy(qi.astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(ki.astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy(wi.astype(np.float32))
    out = oracle.indexer_fwd(q, k, w, ratio, topk)
    for b in range(B):
        for s in range(S):
            sc = _exact_scores(qi, ki, wi, ratio, b, s, s)
            left = dict(sc)
            want_i, want_s = [], []
            for _ in range(topk):
                if not left:
                    want_i.append(-1)
                    want_s.append(-math.inf)
                    continue
                best = max(left.values())
                j = min(jj for jj, v in left.items() if v == best)
                want_i.append(j)
                want_s.append(float(best))
                del left[j]
            r = b * S + s
            assert out["idx"][r].tolist() == want_i, (b, s)
            assert out["scores"][r].tolist() == want_s, (b, s)


def test_topk_invariants_random():
    """On random bf16 inputs: kept indices are visible and distinct, scores
    non-increasing, every kept score >= every dropped visible score, and the
    (k+1)-th score reported equals the largest dropped one."""
    S, B, H, D, S_kv, r, topk = 64, 2, 4, 32, 32, 2, 7
    q, k, w = _rand_problem(S, B, H, D, S_kv, seed=13)
    out = oracle.indexer_fwd(q, k, w, r, topk, want_logits=True)
    for row in range(B * S):
        s = row % S
        L = out["logits"][row]
        idx = out["idx"][row]
        sc = out["scores64"][row]
        valid = idx >= 0
        n = n_visible_closed_form(s, r, S_kv)
        assert valid.sum() == min(topk, n)
        assert np.all(idx[valid] < n)
        assert len(set(idx[valid].tolist())) == valid.sum()
        assert np.all(np.diff(sc[valid]) <= 0)
        np.testing.assert_array_equal(sc[valid], L[idx[valid]])
        dropped = np.setdiff1d(np.arange(n), idx[valid])
        if dropped.size:
            assert sc[valid].min() >= L[dropped].max()
            assert out["next"][row] == L[dropped].max()
        else:
            assert out["next"][row] == -np.inf


def test_topk_at_least_visible_returns_all():
    """topk >= n_vis returns every visible key, sorted."""
    S, B, H, D, S_kv = 12, 1, 2, 8, 12
    q, k, w = _rand_problem(S, B, H, D, S_kv, seed=14)
    out = oracle.indexer_fwd(q, k, w, 1, S_kv + 3, want_logits=True)
    for t in range(S):
        idx = out["idx"][t]
        assert sorted(idx[idx >= 0].tolist()) == list(range(t + 1))


def test_gather_reproduces_topk_scores():
    """Feeding the oracle's own top-k indices back through the given-indices
    path reproduces its scores exactly; -1 slots give -inf."""
    S, B, H, D, S_kv, r, topk = 40, 2, 4, 16, 20, 2, 6
    q, k, w = _rand_problem(S, B, H, D, S_kv, seed=15)
    top = oracle.indexer_fwd(q, k, w, r, topk)
    in_idx = torch.from_numpy(top["idx"].reshape(B, S, topk))
    g = oracle.indexer_fwd(q, k, w, r, topk, in_idx=in_idx)
    np.testing.assert_array_equal(g["idx"], top["idx"])
    np.testing.assert_array_equal(g["scores"], top["scores"])


def test_gather_random_valid_indices():
    """Random valid indices (the input generator's recipe) gather the same
    values as the full logit row."""
    S, B, H, D, S_kv, r, topk = 30, 2, 2, 8, 16, 2, 5
    q, k, w = _rand_problem(S, B, H, D, S_kv, seed=16)
    lim = np.array([[n_visible_closed_form(s, r, S_kv) for s in range(S)]
                    for _ in range(B)])
    in_idx = make_given_indices(B, S, topk, lim, seed=3)
    full = oracle.indexer_fwd(q, k, w, r, topk, want_logits=True)
    g = oracle.indexer_fwd(q, k, w, r, topk, in_idx=in_idx)
    gi = in_idx.numpy().reshape(B * S, topk)
    for row in range(B * S):
        for i in range(topk):
            j = gi[row, i]
            want = -np.inf if j < 0 else full["logits"][row, j]
            assert g["scores64"][row, i] == want


def test_workload_recipes_have_stated_shapes():
    """The synthetic recipes keep the shapes and scales they are named for."""
    wl = WORKLOADS["tiny"]
    q, k, w, pos = make_inputs(wl)
    assert q.shape == (128, 1, 4, 32) and q.dtype == torch.bfloat16
    assert k.shape == (128, 1, 32) and w.shape == (128, 1, 4)
    assert pos is None
    dec = WORKLOADS["decode"]
    assert dec.S_kv * dec.compress_ratio >= dec.pos_range[1]
    g = torch.Generator().manual_seed(0)
    assert abs(float(torch.randn(10000, generator=g).std()) - 1.0) < 0.05


# ---------------------------------------------------------------------------
# the backward: pinned to finite differences of the forward oracle


def _bwd_case(seed, ratio):
    rng = np.random.default_rng(seed)
    S, B, H, D, S_kv, topk = 6, 2, 3, 5, 8, 5
    q = rng.integers(-3, 4, size=(S, B, H, D)).astype(np.float32)
    k = rng.integers(-3, 4, size=(S_kv, B, D)).astype(np.float32)
    w = rng.choice([1.0, -1.0, 0.5, -0.5, 0.25], size=(S, B, H))
    idx = rng.integers(-1, S_kv, size=(B, S, topk)).astype(np.int32)
    idx[0, 3, 1] = idx[0, 3, 0]          # a repeated slot counts twice
    idx[1, 0, 2] = S_kv - 1              # not visible at position 0
    g = rng.choice([1.0, -2.0, 0.5, 3.0, -0.25], size=(B, S, topk))
    return q, k, w.astype(np.float32), idx, g.astype(np.float32), ratio


def _loss(q, k, w, ratio, idx, g):
    import torch
    out = oracle.indexer_fwd(torch.from_numpy(q).to(torch.bfloat16),
                             torch.from_numpy(k).to(torch.bfloat16),
                             torch.from_numpy(w), ratio, idx.shape[-1],
                             in_idx=idx)
    sc = out["scores64"].reshape(g.shape)
    fin = np.isfinite(sc)
    return float((g.astype(np.float64)[fin] * sc[fin]).sum())


@pytest.mark.parametrize("seed,ratio", [(1, 1), (2, 2), (3, 1)])
def test_backward_matches_finite_differences(seed, ratio):
    import torch
    q, k, w, idx, g, ratio = _bwd_case(seed, ratio)
    bwd = oracle.indexer_bwd(torch.from_numpy(q).to(torch.bfloat16),
                             torch.from_numpy(k).to(torch.bfloat16),
                             torch.from_numpy(w), ratio, idx, g)
    base = _loss(q, k, w, ratio, idx, g)
    # w: the loss is linear in w, so a central difference is exact
    eps = 2.0 ** -6
    for pos in np.ndindex(w.shape):
        wp, wm = w.copy(), w.copy()
        wp[pos] += eps
        wm[pos] -= eps
        fd = (_loss(q, k, wp, ratio, idx, g) - _loss(q, k, wm, ratio, idx, g))
        assert fd / (2 * eps) == pytest.approx(bwd["grad_w"][pos], abs=1e-9)
    # q and k: piecewise linear in each entry.  A step of 2^-6 is exact in
    # bf16 for |x| <= 3 and moves an integer dot product by at most 3/64, so
    # only a dot that is exactly 0 can change sign.  ReLU has no derivative
    # there, so entries that feed a zero dot of a scored slot are skipped
    # (found by listing the dots; the expected value itself still comes only
    # from the forward's differences).
    B, S, topk = idx.shape
    zero_q, zero_k = set(), set()
    for b in range(B):
        for s in range(S):
            for i in range(topk):
                j = int(idx[b, s, i])
                if j < 0 or j >= k.shape[0] or not oracle.key_visible(j, s,
                                                                      ratio):
                    continue
                for h in range(q.shape[2]):
                    if float(q[s, b, h] @ k[j, b]) == 0.0:
                        zero_q.add((s, b, h))
                        zero_k.add((j, b))
    for name, arr, grad in (("q", q, bwd["grad_q"]), ("k", k, bwd["grad_k"])):
        checked = total = 0
        for pos in np.ndindex(arr.shape):
            total += 1
            if (name == "q" and pos[:3] in zero_q) or \
                    (name == "k" and pos[:2] in zero_k):
                continue
            ap, am = arr.copy(), arr.copy()
            ap[pos] += eps
            am[pos] -= eps
            args_p = (ap, k) if name == "q" else (q, ap)
            args_m = (am, k) if name == "q" else (q, am)
            fp = (_loss(*args_p, w, ratio, idx, g) - base) / eps
            fm = (base - _loss(*args_m, w, ratio, idx, g)) / eps
            assert fp == pytest.approx(fm, abs=1e-9), (name, pos)
            checked += 1
            assert fp == pytest.approx(grad[pos], abs=1e-9), (name, pos)
        assert checked >= total // 3, (name, checked, total)


def test_backward_ignores_invalid_slots():
    import torch
    q, k, w, idx, g, ratio = _bwd_case(4, 1)
    idx[:] = -1
    bwd = oracle.indexer_bwd(torch.from_numpy(q).to(torch.bfloat16),
                             torch.from_numpy(k).to(torch.bfloat16),
                             torch.from_numpy(w), ratio, idx, g)
    for n in ("grad_q", "grad_k", "grad_w"):
        assert not bwd[n].any()


def test_backward_closed_form_and_relu_convention():
    """One slot, one head: a positive dot gives grad_q = g*w*k,
    grad_k = g*w*q and grad_w = g*dot; a dot of exactly 0 contributes
    nothing (the convention ReLU'(0) = 0)."""
    import torch
    k = np.array([[[1.0, 2.0, 0.0, -1.0]], [[1.0, 1.0, 1.0, 1.0]]],
                 np.float32)                          # [S_kv=2, B=1, D=4]
    q = np.array([[[[1.0, 1.0, 3.0, 0.0]]],           # dot with k0 = 3
                  [[[1.0, -1.0, 0.0, 0.0]]]],         # dot with k1 = 0
                 np.float32)                          # [S=2, B=1, H=1, D=4]
    w = np.array([[[0.5]], [[-2.0]]], np.float32)
    idx = np.array([[[0], [1]]], np.int32)            # [B, S, topk=1]
    g = np.array([[[3.0], [5.0]]], np.float32)
    bwd = oracle.indexer_bwd(torch.from_numpy(q).to(torch.bfloat16),
                             torch.from_numpy(k).to(torch.bfloat16),
                             torch.from_numpy(w), 1, idx, g)
    np.testing.assert_array_equal(bwd["grad_q"][0, 0, 0], 3.0 * 0.5 * k[0, 0])
    np.testing.assert_array_equal(bwd["grad_q"][1], 0.0)
    np.testing.assert_array_equal(bwd["grad_k"][0, 0], 3.0 * 0.5 * q[0, 0, 0])
    np.testing.assert_array_equal(bwd["grad_k"][1], 0.0)
    assert bwd["grad_w"][0, 0, 0] == 3.0 * 3.0
    assert bwd["grad_w"][1, 0, 0] == 0.0


# ---- the pool variant: key validity, pool compression, expansion ----------

@pytest.mark.parametrize("ratio,topk", [(1, 6), (2, 4), (1, 40)])
def test_key_valid_mask_matches_exact_brute_force(ratio, topk):
    """A key whose valid flag is 0 is not a candidate: exact rational brute
    force over the valid visible keys only (integer inputs, frequent ties),
    -inf logits and -inf given-index scores for the masked keys."""
    rng = np.random.default_rng(77 + ratio)
    S, B, H, D, S_kv = 24, 2, 3, 5, 12
    qi = rng.integers(-3, 4, size=(S, B, H, D))
    ki = rng.integers(-3, 4, size=(S_kv, B, D))
    wi = rng.choice([1, -1, 0.5, -0.5, 0.25], size=(S, B, H))
    kv = (rng.random((S_kv, B)) > 0.3).astype(np.uint8)
    q = torch.from_numpy(qi.astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(ki.astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy(wi.astype(np.float32))
    out = oracle.indexer_fwd(q, k, w, ratio, topk, key_valid=kv,
                             want_logits=True)
    for b in range(B):
        for s in range(S):
            sc = {j: v for j, v in _exact_scores(qi, ki, wi, ratio, b, s,
                                                 s).items() if kv[j, b]}
            r = b * S + s
            assert out["nvis"][r] == len(sc)
            for j in range(S_kv):
                if j not in sc:
                    assert out["logits"][r, j] == -math.inf
            left = dict(sc)
            want = []
            for _ in range(topk):
                if not left:
                    want.append(-1)
                    continue
                best = max(left.values())
                j = min(jj for jj, v in left.items() if v == best)
                want.append(j)
                del left[j]
            assert out["idx"][r].tolist() == want, (b, s)
    # given indices: a masked key scores -inf, its index is copied through
    gi = torch.from_numpy(rng.integers(0, S_kv, size=(B, S, 4)).astype(
        np.int32))
    g = oracle.indexer_fwd(q, k, w, ratio, 4, in_idx=gi, key_valid=kv)
    for b in range(B):
        for s in range(S):
            for i in range(4):
                j = int(gi[b, s, i])
                val = g["scores64"][b * S + s, i]
                if not kv[j, b] or (j + 1) * ratio - 1 > s:
                    assert val == -math.inf
                else:
                    assert val == float(_exact_scores(qi, ki, wi, ratio, b, s,
                                                      s)[j])


def _pool_inputs(T, B, D, kpool, seed):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn((T, B, D), generator=g).to(torch.bfloat16)
    gate = torch.randn((T, B, D), generator=g)
    ape = torch.randn((kpool, D), generator=g) * 0.5
    return k, gate, ape


def test_kpool_single_slot_is_the_key():
    """kpool = 1: the softmax over one slot is 1, the pooled key is the
    token's key exactly."""
    k, gate, ape = _pool_inputs(11, 2, 16, 1, 1)
    c = oracle.kpool_compress(k, gate, ape, None, 1, 0)
    assert c["P"] == 11
    np.testing.assert_array_equal(c["keys"], k.float().numpy())


def test_kpool_hand_example():
    """kpool = 2, gate 0 on both slots, position embedding (0, ln 3): the
    weights are 1/4 and 3/4 in every channel, so the pooled key is
    k0/4 + 3*k1/4 (integer keys, exact up to the exponential's rounding)."""
    D = 6
    k = torch.tensor([[[1, -2, 3, 0, 5, -7]], [[3, 2, -1, 4, 1, 1]]],
                     dtype=torch.float32).to(torch.bfloat16)
    gate = torch.zeros((2, 1, D))
    ape = torch.tensor([[0.0] * D, [math.log(3.0)] * D])
    c = oracle.kpool_compress(k, gate, ape, None, 2, 0)
    want = np.array([1, -2, 3, 0, 5, -7]) / 4 + 3 * np.array(
        [3, 2, -1, 4, 1, 1]) / 4
    # ape is fp32: ln 3 rounded to fp32 shifts the weights by < 1e-7
    np.testing.assert_allclose(c["keys"][0, 0], want, rtol=0, atol=1e-6)


def test_kpool_equal_logits_give_the_mean_per_channel():
    """Slot logits equal across the slots (varying across channels and
    pools): every channel's pooled value is the plain mean of its slots.
    A softmax taken over channels instead of slots fails this."""
    T, B, D, kp = 24, 2, 16, 4
    k, _, _ = _pool_inputs(T, B, D, kp, 2)
    rng = np.random.default_rng(3)
    per_pool = rng.normal(size=(T // kp, B, D)).astype(np.float32)
    gate = torch.from_numpy(np.repeat(per_pool, kp, axis=0))
    ape = torch.zeros((kp, D))
    c = oracle.kpool_compress(k, gate, ape, None, kp, 0)
    want = k.float().numpy().reshape(T // kp, kp, B, D).mean(axis=1)
    np.testing.assert_allclose(c["keys"], want, rtol=0, atol=1e-12)


def test_kpool_shift_invariance_and_dominant_slot():
    """Adding one constant per (pool, channel) to every slot's logit leaves
    the pooled key unchanged; a slot whose logit is 60 above the others
    gives (nearly) that slot's key."""
    T, B, D, kp = 16, 1, 8, 4
    k, gate, ape = _pool_inputs(T, B, D, kp, 4)
    c0 = oracle.kpool_compress(k, gate, ape, None, kp, 0)
    shift = np.repeat(np.random.default_rng(5).normal(
        size=(T // kp, B, D)).astype(np.float32) * 3, kp, axis=0)
    c1 = oracle.kpool_compress(k, gate + torch.from_numpy(shift), ape, None,
                               kp, 0)
    np.testing.assert_allclose(c1["keys"], c0["keys"], rtol=0, atol=1e-6)
    g2 = torch.zeros((T, B, D))
    g2[2::kp] = 60.0  # slot 2 of every pool dominates
    c2 = oracle.kpool_compress(k, g2, torch.zeros((kp, D)), None, kp, 0)
    np.testing.assert_allclose(c2["keys"], k.float().numpy()[2::kp],
                               rtol=0, atol=1e-20 + 1e-24)


def test_kpool_first_key_count_and_validity():
    """Pools start at first_key and only whole pools count; a pool is valid
    iff each of its tokens is."""
    T, B, D, kp, fk = 37, 2, 8, 4, 5
    k, gate, ape = _pool_inputs(T, B, D, kp, 6)
    valid = (np.random.default_rng(7).random((T, B)) > 0.1).astype(np.uint8)
    c = oracle.kpool_compress(k, gate, ape, valid, kp, fk)
    assert c["P"] == (T - fk) // kp == 8
    # the same pools from the tokens after first_key with first_key = 0
    c0 = oracle.kpool_compress(k[fk:], gate[fk:], ape, valid[fk:], kp, 0)
    np.testing.assert_array_equal(c["keys"], c0["keys"])
    want_valid = valid[fk:fk + 8 * kp].reshape(8, kp, B).all(axis=1)
    np.testing.assert_array_equal(c["valid"], want_valid.astype(np.uint8))
    assert oracle.kpool_compress(k[:4], gate[:4], ape, None, kp, 1)["P"] == 0


def test_expand_selection_closed_form():
    pools = np.array([[[3, -1, 0]], [[-1, -1, 7]]], np.int32)  # [2, 1, 3]
    t = oracle.expand_selection(pools, 4, 10)
    assert t.shape == (2, 1, 12)
    assert t[0, 0].tolist() == [22, 23, 24, 25, -1, -1, -1, -1,
                                10, 11, 12, 13]
    assert t[1, 0].tolist() == [-1] * 8 + [38, 39, 40, 41]


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9,
                  -(1.0 + 2.0 ** -8 + 2.0 ** -30), 0.0, -0.0, 2.0 ** -126])
    bits = oracle.round_bf16(x).tolist()
    assert bits == [0x3F80, 0x3F82, 0x3F80, 0xBF81, 0x0000, 0x8000, 0x0080]


def test_pooled_forward_with_one_slot_pools_is_the_plain_forward():
    """kpool = 1, first_key = 0, every token valid: pools are the tokens and
    the pool variant is the plain top-k forward (tokens = indices)."""
    S, B, H, D = 40, 2, 4, 16
    q, k, w = _rand_problem(S, B, H, D, S, 8)
    gate = torch.randn((S, B, D))
    ape = torch.zeros((1, D))
    pooled = oracle.indexer_pooled_fwd(q, k, gate, ape, None, w, 1, 0, 9)
    plain = oracle.indexer_fwd(q, k, w, 1, 9)
    np.testing.assert_array_equal(pooled["tokens"].reshape(B * S, 9),
                                  plain["idx"])
    np.testing.assert_array_equal(pooled["scores"], plain["scores"])


# ---- sparse MLA forward over selected tokens ------------------------------

def _mla_inputs(S, B, H, Dc, T, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((S, B, H, Dc), generator=g).to(torch.bfloat16)
    c = torch.randn((T, B, Dc), generator=g).to(torch.bfloat16)
    return q, c


def test_mla_single_slot_and_repeated_token():
    """One valid slot: the output is that token's latent row and lse its
    scaled score; the same token in n slots: the same output, lse + log n."""
    S, B, H, Dc, T = 3, 2, 4, 16, 9
    q, c = _mla_inputs(S, B, H, Dc, T, 1)
    qf, cf = q.double().numpy(), c.double().numpy()
    idx = np.full((B, S, 5), -1, np.int32)
    idx[:, :, 2] = 4
    r = oracle.sparse_mla_fwd(q, c, idx, 0.125)
    for s in range(S):
        for b in range(B):
            for h in range(H):
                np.testing.assert_array_equal(r["o"][s, b, h], cf[4, b])
                x = 0.125 * float(qf[s, b, h] @ cf[4, b])
                assert abs(r["lse"][s, b, h] - x) <= 1e-12 * (1 + abs(x))
    idx[:, :, :] = 4
    r3 = oracle.sparse_mla_fwd(q, c, idx, 0.125)
    np.testing.assert_allclose(r3["o"], r["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r3["lse"], r["lse"] + math.log(5), rtol=0,
                               atol=1e-12)


def test_mla_two_slot_closed_form():
    """Two tokens whose scaled scores differ by ln 3: weights 1/4 and 3/4."""
    Dc = 8
    q = torch.zeros((1, 1, 1, Dc))
    q[0, 0, 0, 0] = 1.0
    c = torch.zeros((2, 1, Dc))
    c[0, 0] = torch.tensor([0.0, 1, 2, 3, 4, 5, 6, 7])
    c[1, 0] = torch.tensor([2.0, -1, 0, 1, 8, 0, 2, 2])
    # scores (scale 1): c[0,0,0] = 0 and c[1,0,0] = 2; choose scale so that
    # scale * 2 = ln 3
    scale = math.log(3.0) / 2.0
    r = oracle.sparse_mla_fwd(q.to(torch.bfloat16), c.to(torch.bfloat16),
                              np.array([[[0, 1]]], np.int32), scale)
    want = 0.25 * c[0, 0].numpy() + 0.75 * c[1, 0].numpy()
    np.testing.assert_allclose(r["o"][0, 0, 0], want, rtol=0, atol=1e-12)
    assert abs(r["lse"][0, 0, 0] - math.log(4.0)) <= 1e-12


def test_mla_invalid_slots_permutation_and_shift():
    """-1 and out-of-range slots are skipped; permuting the slots changes
    nothing; an empty row gives o = 0 and lse = -inf."""
    S, B, H, Dc, T, k = 5, 2, 3, 32, 20, 12
    q, c = _mla_inputs(S, B, H, Dc, T, 2)
    rng = np.random.default_rng(3)
    idx = rng.integers(0, T, size=(B, S, k)).astype(np.int32)
    idx[:, :, ::4] = -1
    r = oracle.sparse_mla_fwd(q, c, idx, 0.1)
    bad = idx.copy()
    bad[:, :, ::4] = T + 3  # out of range: skipped like -1
    rb = oracle.sparse_mla_fwd(q, c, bad, 0.1)
    np.testing.assert_array_equal(rb["o"], r["o"])
    perm = rng.permutation(k)
    rp = oracle.sparse_mla_fwd(q, c, idx[:, :, perm], 0.1)
    np.testing.assert_allclose(rp["o"], r["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(rp["lse"], r["lse"], rtol=0, atol=1e-12)
    empty = np.full((B, S, k), -1, np.int32)
    re_ = oracle.sparse_mla_fwd(q, c, empty, 0.1)
    assert np.all(re_["o"] == 0) and np.all(np.isneginf(re_["lse"]))


def test_mla_convex_combination_and_head_independence():
    """Each output is a convex combination of the selected rows (inside
    their per-channel range), and a head's output depends on its own query
    only (heads permute with the queries)."""
    S, B, H, Dc, T, k = 4, 1, 6, 16, 30, 9
    q, c = _mla_inputs(S, B, H, Dc, T, 4)
    idx = np.random.default_rng(5).integers(0, T, size=(B, S, k)).astype(
        np.int32)
    r = oracle.sparse_mla_fwd(q, c, idx, 0.2)
    cf = c.double().numpy()
    for s in range(S):
        rows = cf[idx[0, s], 0]
        lo, hi = rows.min(axis=0), rows.max(axis=0)
        assert np.all(r["o"][s, 0] >= lo - 1e-12)
        assert np.all(r["o"][s, 0] <= hi + 1e-12)
    perm = np.random.default_rng(6).permutation(H)
    rp = oracle.sparse_mla_fwd(q[:, :, perm].contiguous(), c, idx, 0.2)
    np.testing.assert_array_equal(rp["o"], r["o"][:, :, perm])
