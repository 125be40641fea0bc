"""GPU parity of the packed variable-length forward (dsa_indexer_fwd_varlen)
against the oracle applied to each sequence on its own, and bit-for-bit
agreement with the batched forward when the sequences have equal lengths."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dsa_inputs import make_given_indices
from tests.helpers import compare_topk_row, score_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    return m


def packed_inputs(lens_q, lens_k, H, D, seed):
    """Seeded packed q [T, H, D], k [T_kv, D] (bf16) and w [T, H]."""
    g = torch.Generator().manual_seed(seed)
    T, T_kv = sum(lens_q), sum(lens_k)
    q = torch.randn((T, H, D), generator=g).to(torch.bfloat16)
    k = torch.randn((T_kv, D), generator=g).to(torch.bfloat16)
    w = torch.randn((T, H), generator=g) * H ** -0.5
    cq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    return q, k, w, cq, ck


def seq_view(q, k, w, cq, ck, i):
    """Sequence i as a B = 1 problem in the batched layouts."""
    qi = q[cq[i]:cq[i + 1]].unsqueeze(1).contiguous()
    ki = k[ck[i]:ck[i + 1]].unsqueeze(1).contiguous()
    wi = w[cq[i]:cq[i + 1]].unsqueeze(1).contiguous()
    return qi, ki, wi


def run_varlen(dsa, q, k, w, cq, ck, ratio, topk, q_pos=None, in_idx=None):
    d = torch.device("cuda")
    sc, idx, ws = dsa.dsa_indexer_fwd_varlen(
        q.to(d), k.to(d), w.to(d), cq, ck, ratio, topk,
        q_pos=None if q_pos is None else q_pos.to(d),
        in_idx=None if in_idx is None else in_idx.to(d))
    st = dsa.dsa_indexer_check(ws)
    return sc.cpu().numpy(), idx.cpu().numpy(), st


@pytest.mark.parametrize("lens_q,lens_k,H,D,ratio,topk,with_pos", [
    # long and short prefill sequences, an empty one, a keyless one
    ([700, 0, 130, 64, 5], [700, 3, 130, 0, 5], 64, 128, 1, 100, False),
    # C4-style ratio, ragged tails, decode-shaped sequences (1-3 rows)
    ([1, 3, 520, 2, 257], [300, 90, 130, 600, 70], 64, 128, 4, 64, True),
    # small heads, more sequences than slices
    ([40, 33, 17, 90, 8, 61], [40, 33, 17, 90, 8, 61], 16, 32, 1, 24, False),
])
def test_varlen_matches_oracle(dsa, lens_q, lens_k, H, D, ratio, topk,
                               with_pos):
    q, k, w, cq, ck = packed_inputs(lens_q, lens_k, H, D, seed=sum(lens_q))
    N = len(lens_q)
    pos = None
    if with_pos:
        rng = np.random.default_rng(N)
        pos = torch.from_numpy(rng.integers(0, 3000, size=N).astype(np.int32))
    sc, idx, st = run_varlen(dsa, q, k, w, cq, ck, ratio, topk, q_pos=pos)
    assert st == 0
    for i in range(N):
        rows = slice(cq[i], cq[i + 1])
        if cq[i + 1] == cq[i]:
            continue
        if ck[i + 1] == ck[i]:  # no keys: all padding
            assert np.all(idx[rows] == -1) and np.all(np.isneginf(sc[rows]))
            continue
        qi, ki, wi = seq_view(q, k, w, cq, ck, i)
        pi = None if pos is None else pos[i:i + 1]
        ref = oracle.indexer_fwd(qi, ki, wi, ratio, topk, q_pos=pi,
                                 want_logits=True)
        for r in range(cq[i + 1] - cq[i]):
            msg = compare_topk_row(idx[cq[i] + r], sc[cq[i] + r],
                                   ref["idx"][r], ref["scores64"][r],
                                   ref["next"][r], ref["logits"][r])
            assert not msg, (i, r, msg)


def test_varlen_equals_batched_bitwise(dsa):
    """Equal-length sequences: the packed call and the batched [S, B] call
    run the same kernels row by row, so every output bit agrees."""
    B, S, S_kv, H, D, ratio, topk = 3, 600, 150, 64, 128, 4, 100
    q, k, w, cq, ck = packed_inputs([S] * B, [S_kv] * B, H, D, seed=5)
    sc, idx, st = run_varlen(dsa, q, k, w, cq, ck, ratio, topk)
    assert st == 0
    qb = q.view(B, S, H, D).transpose(0, 1).contiguous()
    kb = k.view(B, S_kv, D).transpose(0, 1).contiguous()
    wb = w.view(B, S, H).transpose(0, 1).contiguous()
    d = torch.device("cuda")
    bsc, bidx, ws = dsa.dsa_indexer_fwd(qb.to(d), kb.to(d), wb.to(d), ratio,
                                        topk)
    assert dsa.dsa_indexer_check(ws) == 0
    np.testing.assert_array_equal(idx.reshape(B, S, topk),
                                  bidx.cpu().numpy())
    assert np.array_equal(sc.reshape(B, S, topk).view(np.uint32),
                          bsc.cpu().numpy().view(np.uint32))


def test_varlen_given_indices_and_status(dsa):
    lens_q, lens_k = [300, 5, 200], [300, 40, 50]
    H, D, ratio, topk = 32, 64, 1, 40
    q, k, w, cq, ck = packed_inputs(lens_q, lens_k, H, D, seed=9)
    T = cq[-1]
    gi = torch.full((T, topk), -1, dtype=torch.int32)
    for i in range(3):
        s = np.arange(cq[i + 1] - cq[i])
        nv = np.clip(s + 1, 0, ck[i + 1] - ck[i])[None, :]
        gi[cq[i]:cq[i + 1]] = make_given_indices(1, len(s), topk, nv,
                                                 11 + i)[0]
    sc, idx, st = run_varlen(dsa, q, k, w, cq, ck, ratio, topk, in_idx=gi)
    assert st == 0
    np.testing.assert_array_equal(idx, gi.numpy())
    for i in range(3):
        qi, ki, wi = seq_view(q, k, w, cq, ck, i)
        ref = oracle.indexer_fwd(qi, ki, wi, ratio, topk,
                                 in_idx=gi[cq[i]:cq[i + 1]].unsqueeze(0))
        o = ref["scores64"]
        g = sc[cq[i]:cq[i + 1]].astype(np.float64)
        assert np.array_equal(np.isneginf(g), np.isneginf(o))
        fin = np.isfinite(o)
        assert np.all(np.abs(g[fin] - o[fin]) <= score_tol(o[fin]))
    # an index past the third sequence's keys, on whichever slice it runs
    gi[cq[2] + 7, 3] = lens_k[2]
    sc, idx, st = run_varlen(dsa, q, k, w, cq, ck, ratio, topk, in_idx=gi)
    assert st == 6  # DSA_ERR_INDEX_RANGE
    assert np.isneginf(sc[cq[2] + 7, 3])
