"""GPU parity of the indexer backward (dsa_indexer_bwd) against the fp64
CPU oracle's backward, through the C ABI.

Rule, element by element: |gpu - oracle| <= 2^-7 * A + 1e-6 (+ X), where A
is the oracle's sum of the absolute values of the element's terms (the
kernel rounds g * w to bf16, a relative error of at most 2^-9 per term, and
accumulates in fp32) and X covers the ReLU' decisions floating point cannot
settle: a (slot, head) whose fp64 dot product is within 1e-4 of the sum of
|q_d k_d| of zero may fall on either side of 0 in the kernel's fp32, so its
whole term is allowed on the elements it feeds.

At the prefill size (S = S_kv = 4096, topk = 2048), sampled rows are
checked against the oracle run on those rows alone (a row's grad_q and
grad_w depend only on its own slots), grad_k against the oracle with the
upstream gradient kept on the sampled rows only, and the whole result
against the homogeneity identity
    <grad_q, q> = <grad_k, k> = sum_{t,h} w[t,h] grad_w[t,h]
(each side equals sum over slots of g * sum_h w * ReLU(s_h)).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dsa_inputs import make_given_indices

pytestmark = pytest.mark.gpu

RANGE_STATUS = 6  # DSA_ERR_INDEX_RANGE
REL = 2.0 ** -7
ABS = 1e-6
AMBIG = 1e-4


@pytest.fixture(scope="module")
def dsa():
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    return m


def make_problem(S, B, H, D, S_kv, ratio, topk, seed, q_pos=None,
                 limit="all"):
    """Seeded q, k, w (the workloads' distributions), indices and upstream
    gradients.  limit="all" draws indices over every key (invisible ones
    included, which the backward must skip), "visible" over the row's
    visible keys only."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((S, B, H, D), generator=g).to(torch.bfloat16)
    k = torch.randn((S_kv, B, D), generator=g).to(torch.bfloat16)
    w = torch.randn((S, B, H), generator=g) * H ** -0.5
    gs = torch.randn((B, S, topk), generator=g)
    if limit == "all":
        lim = np.full((B, S), S_kv)
    else:
        base = (np.zeros(B, np.int64) if q_pos is None
                else q_pos.numpy().astype(np.int64))
        pos = base[:, None] + np.arange(S)[None, :]
        lim = np.clip((pos + 1) // ratio, 0, S_kv)
    idx = make_given_indices(B, S, topk, lim, seed + 1000)
    return q, k, w, idx, gs


def run_gpu(dsa, q, k, w, ratio, idx, gs, q_pos=None):
    d = torch.device("cuda")
    S, B, H, D = q.shape
    S_kv = k.shape[0]
    nan = dict(dtype=torch.float32, device=d)
    # outputs start as NaN: every element must be written
    gq = torch.full((S, B, H, D), float("nan"), **nan)
    gk = torch.full((S_kv, B, D), float("nan"), **nan)
    gw = torch.full((S, B, H), float("nan"), **nan)
    gq, gk, gw, ws = dsa.dsa_indexer_bwd(
        q.to(d), k.to(d), w.to(d), ratio, idx.to(d), gs.to(d),
        q_pos=None if q_pos is None else q_pos.to(d), grad_q=gq, grad_k=gk,
        grad_w=gw)
    st = dsa.dsa_indexer_check(ws)
    return (gq.cpu().numpy().astype(np.float64),
            gk.cpu().numpy().astype(np.float64),
            gw.cpu().numpy().astype(np.float64), st)


def ambiguity(q, k, w, ratio, idx, gs, q_pos=None, rows=None):
    """Allowances (X above) for grad_q [S,B,H,D], grad_k [S_kv,B,D] and
    grad_w [S,B,H], from the fp64 dot products of every valid slot."""
    qf = q.float().numpy().astype(np.float64)
    kf = k.float().numpy().astype(np.float64)
    wf = w.numpy().astype(np.float64)
    ix = idx.numpy()
    gf = gs.numpy().astype(np.float64)
    S, B, H, D = qf.shape
    S_kv = kf.shape[0]
    xq, xk, xw = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(wf)
    n_amb = 0
    for b in range(B):
        base = 0 if q_pos is None else int(q_pos[b])
        for s in (range(S) if rows is None else rows):
            pos = base + s
            nv = 0 if pos < 0 else min(S_kv, (pos + 1) // ratio)
            js = ix[b, s]
            sel = np.nonzero((js >= 0) & (js < nv))[0]
            if sel.size == 0:
                continue
            kj = kf[js[sel], b]                     # [n, D]
            dots = kj @ qf[s, b].T                  # [n, H]
            mag = np.abs(kj) @ np.abs(qf[s, b]).T
            amb = np.abs(dots) <= AMBIG * mag
            if not amb.any():
                continue
            for ii, h in zip(*np.nonzero(amb)):
                n_amb += 1
                c = abs(gf[b, s, sel[ii]] * wf[s, b, h])
                xq[s, b, h] += c * np.abs(kj[ii])
                xk[js[sel[ii]], b] += c * np.abs(qf[s, b, h])
                xw[s, b, h] += abs(gf[b, s, sel[ii]]) * AMBIG * mag[ii, h]
    return xq, xk, xw, n_amb


def assert_close(name, got, ref, absum, extra):
    err = np.abs(got - ref)
    tol = REL * absum + ABS + extra
    bad = ~(err <= tol)  # NaN counts as bad
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {bad.size} outside tolerance; "
            f"first {i.tolist()}: got {got[bad][:5]}, want {ref[bad][:5]}, "
            f"tol {tol[bad][:5]}")


def check_all(dsa, q, k, w, ratio, idx, gs, q_pos=None, want_status=0):
    gq, gk, gw, st = run_gpu(dsa, q, k, w, ratio, idx, gs, q_pos)
    assert st == want_status
    ref = oracle.indexer_bwd(q, k, w, ratio, idx, gs, q_pos=q_pos)
    xq, xk, xw, _ = ambiguity(q, k, w, ratio, idx, gs, q_pos)
    assert_close("grad_q", gq, ref["grad_q"], ref["abs_q"], xq)
    assert_close("grad_k", gk, ref["grad_k"], ref["abs_k"], xk)
    assert_close("grad_w", gw, ref["grad_w"], ref["abs_w"], xw)
    return gq, gk, gw


@pytest.mark.parametrize("S,B,D,S_kv,ratio,topk,with_pos,limit", [
    # two tiles with a ragged tail; invisible keys among the indices
    (257, 2, 128, 257, 1, 200, False, "all"),
    # C4-style positions, D = 64 (the second d-chunk is zero padding)
    (130, 1, 64, 40, 4, 64, True, "all"),
    # D = 96 (a partial second chunk), three tiles with a 44-slot tail
    (64, 3, 96, 300, 1, 300, True, "visible"),
    # many rows per CTA, four full tiles per row
    (512, 1, 128, 512, 1, 512, False, "visible"),
    # one tile per row (the row's first tile is also its last)
    (1024, 2, 128, 1024, 1, 128, False, "all"),
])
def test_bwd_matches_oracle(dsa, S, B, D, S_kv, ratio, topk, with_pos,
                            limit):
    pos = None
    if with_pos:
        pos = torch.from_numpy(
            np.random.default_rng(S + B).integers(0, 4 * S_kv, size=B)
            .astype(np.int32))
    q, k, w, idx, gs = make_problem(S, B, 64, D, S_kv, ratio, topk,
                                    seed=S + D + topk, q_pos=pos, limit=limit)
    check_all(dsa, q, k, w, ratio, idx, gs, q_pos=pos)


def test_bwd_padding_duplicates_and_range(dsa):
    """-1 slots, repeated keys in a row (each slot counts), a zero upstream
    gradient, and indices outside [-1, S_kv) (skipped, status raised)."""
    S, B, D, S_kv, topk = 200, 2, 128, 200, 160
    q, k, w, idx, gs = make_problem(S, B, 64, D, S_kv, 1, topk, seed=77)
    idx = idx.clone()
    idx[0, 150, 10:40] = -1
    idx[1, 199, 5] = idx[1, 199, 6] = idx[1, 199, 7] = 3
    idx[0, 100, :] = 17  # one key in every slot of a row
    gs[1, 50, :] = 0.0
    check_all(dsa, q, k, w, 1, idx, gs)
    bad = idx.clone()
    bad[0, 120, 3] = S_kv
    bad[1, 7, 0] = -5
    check_all(dsa, q, k, w, 1, bad, gs, want_status=RANGE_STATUS)


def test_bwd_rows_without_valid_slots(dsa):
    """Rows whose slots are all -1 or invisible get zero grad_q and grad_w
    (written, not left untouched), and grad_k stays zero."""
    S, B, D, S_kv, topk = 40, 1, 128, 64, 128
    q, k, w, idx, gs = make_problem(S, B, 64, D, S_kv, 4, topk, seed=5)
    idx = torch.full_like(idx, -1)
    idx[0, :, :4] = 63  # never visible to rows at positions < 255
    gq, gk, gw, st = run_gpu(dsa, q, k, w, 4, idx, gs)
    assert st == 0
    assert np.all(gq == 0) and np.all(gk == 0) and np.all(gw == 0)


def test_bwd_prefill_size_sampled(dsa):
    """The 4096 x 4096 prefill with topk = 2048, in the launch
    configuration a training step uses."""
    S = S_kv = 4096
    B, H, D, topk = 1, 64, 128, 2048
    g = torch.Generator().manual_seed(11)
    q = torch.randn((S, B, H, D), generator=g).to(torch.bfloat16)
    k = torch.randn((S_kv, B, D), generator=g).to(torch.bfloat16)
    w = torch.randn((S, B, H), generator=g) * 0.125
    gs = torch.randn((B, S, topk), generator=g)
    lim = np.minimum(np.arange(S) + 1, S_kv)[None, :]
    idx = make_given_indices(B, S, topk, lim, 12)
    gq, gk, gw, st = run_gpu(dsa, q, k, w, 1, idx, gs)
    assert st == 0
    rows = [0, 1, 127, 128, 2046, 2047, 2048, 3000, 4095]

    def oracle_row(s, grad):
        # row s alone: a one-row problem at position s
        return oracle.indexer_bwd(q[s:s + 1], k, w[s:s + 1], 1,
                                  idx[:, s:s + 1], grad[:, s:s + 1],
                                  q_pos=torch.tensor([s], dtype=torch.int32))

    xq, xk, xw, _ = ambiguity(q, k, w, 1, idx, gs, rows=rows)
    for s in rows:
        r = oracle_row(s, gs)
        assert_close(f"grad_q[{s}]", gq[s:s + 1], r["grad_q"], r["abs_q"],
                     xq[s:s + 1])
        assert_close(f"grad_w[{s}]", gw[s:s + 1], r["grad_w"], r["abs_w"],
                     xw[s:s + 1])

    # homogeneity identity over the whole problem
    qf = q.float().numpy().astype(np.float64)
    kf = k.float().numpy().astype(np.float64)
    wf = w.numpy().astype(np.float64)
    a = float(np.sum(gq * qf))
    b = float(np.sum(gk * kf))
    c = float(np.sum(gw * wf))
    scale = float(np.sum(np.abs(gw) * np.abs(wf)))
    assert abs(a - c) <= 1e-3 * scale and abs(b - c) <= 1e-3 * scale, (
        a, b, c, scale)

    # grad_k exactly: upstream gradient only on the sampled rows
    gs2 = torch.zeros_like(gs)
    gs2[:, rows] = gs[:, rows]
    gq2, gk2, gw2, st = run_gpu(dsa, q, k, w, 1, idx, gs2)
    assert st == 0
    ref_k = np.zeros_like(gk2)
    abs_k = np.zeros_like(gk2)
    for s in rows:
        r = oracle_row(s, gs2)
        ref_k += r["grad_k"]
        abs_k += r["abs_k"]
    assert_close("grad_k (sampled rows)", gk2, ref_k, abs_k, xk)
    others = np.setdiff1d(np.arange(S), rows)
    assert np.all(gq2[others] == 0) and np.all(gw2[others] == 0)
