"""GPU parity of the sparse MLA forward (attention in the latent space over
the selected tokens) against the fp64 oracle, through the C ABI.

Rule: out_o within 2^-7 * A + 1e-5 per element, A = sum_i p_i |c_i,d| (the
softmax-weighted magnitude of the rows the element averages; the kernel
rounds the weights to bf16, a relative 2^-9 each, and accumulates in fp32);
out_lse within 2e-4 * (1 + |lse|); rows without a valid slot give o = 0 and
lse = -inf exactly.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    return m


def mla_problem(S, B, H, Dc, T, topk, seed, invalid=0.1):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((S, B, H, Dc), generator=g).to(torch.bfloat16)
    c = torch.randn((T, B, Dc), generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, T, size=(B, S, topk)).astype(np.int32)
    idx[rng.random((B, S, topk)) < invalid] = -1
    return q, c, torch.from_numpy(idx)


def weighted_abs(q, c, idx, scale):
    """A[s,b,h,d] = sum_i softmax(x)_i |c[j_i,b,d]| over the valid slots
    (the error scale of an element; fp64 numpy, a tolerance only)."""
    qf, cf = q.double().numpy(), c.double().numpy()
    ix = idx.numpy()
    S, B, H, Dc = qf.shape
    T = cf.shape[0]
    A = np.zeros((S, B, H, Dc))
    for b in range(B):
        for s in range(S):
            js = ix[b, s][(ix[b, s] >= 0) & (ix[b, s] < T)]
            if js.size == 0:
                continue
            rows = cf[js, b]                       # [n, Dc]
            x = scale * (qf[s, b] @ rows.T)        # [H, n]
            x -= x.max(axis=1, keepdims=True)
            p = np.exp(x)
            p /= p.sum(axis=1, keepdims=True)
            A[s, b] = p @ np.abs(rows)
    return A


def check(dsa, q, c, idx, scale, want_status=0):
    d = torch.device("cuda")
    o, lse, ws = dsa.dsa_sparse_mla_fwd(q.to(d), c.to(d), idx.to(d), scale)
    assert dsa.dsa_indexer_check(ws) == want_status
    o = o.cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    ref = oracle.sparse_mla_fwd(q, c, idx, scale)
    empty = np.isneginf(ref["lse"])
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.all(o[empty] == 0)
    fin = ~empty
    assert np.all(np.abs(lse[fin] - ref["lse"][fin]) <=
                  2e-4 * (1 + np.abs(ref["lse"][fin])))
    A = weighted_abs(q, c, idx, scale)
    err = np.abs(o - ref["o"])
    bad = err > 2.0 ** -7 * A + 1e-5
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:3].tolist())


@pytest.mark.parametrize("S,B,H,Dc,T,topk", [
    (40, 2, 64, 128, 300, 200),   # two tiles with a ragged tail
    (16, 1, 128, 512, 1000, 256),  # two head groups, the full latent width
    (9, 2, 64, 256, 50, 64),      # fewer slots than a tile, repeated tokens
    (5, 1, 64, 384, 2000, 640),   # five tiles, Dc = 384
])
def test_sparse_mla_matches_oracle(dsa, S, B, H, Dc, T, topk):
    q, c, idx = mla_problem(S, B, H, Dc, T, topk, seed=S + Dc + topk)
    check(dsa, q, c, idx, 1.0 / math.sqrt(Dc))


def test_sparse_mla_empty_rows_and_range_status(dsa):
    q, c, idx = mla_problem(12, 2, 64, 128, 80, 130, seed=3, invalid=0.3)
    idx = idx.clone()
    idx[0, 3, :] = -1          # a row with no valid slot
    idx[1, 7, :] = -1
    check(dsa, q, c, idx, 0.09)
    bad = idx.clone()
    bad[1, 2, 5] = 80          # out of range: skipped, status raised
    bad[0, 0, 0] = -3
    check(dsa, q, c, bad, 0.09, want_status=6)


def test_sparse_mla_over_pooled_selection(dsa):
    """The pipeline's last step: attention over the token ids the pool
    variant selected (-1 tails included)."""
    S, B, H, D, T, kp, itopk, Dc = 64, 1, 64, 128, 64, 4, 32, 512
    g = torch.Generator().manual_seed(8)
    qi = torch.randn((S, B, H, D), generator=g).to(torch.bfloat16)
    ki = torch.randn((T, B, D), generator=g).to(torch.bfloat16)
    gate = torch.randn((T, B, D), generator=g)
    ape = torch.randn((kp, D), generator=g) * 0.5
    w = torch.randn((S, B, H), generator=g) * 0.125
    d = torch.device("cuda")
    tok, _, _, ws = dsa.dsa_indexer_fwd_pooled(
        qi.to(d), ki.to(d), gate.to(d), ape.to(d), w.to(d), kp, 0, itopk)
    assert dsa.dsa_indexer_check(ws) == 0
    q = torch.randn((S, B, 64, Dc), generator=g).to(torch.bfloat16)
    c = torch.randn((T, B, Dc), generator=g).to(torch.bfloat16)
    check(dsa, q, c, tok.cpu(), 1.0 / math.sqrt(Dc))


def test_sparse_mla_running_maximum_moves(dsa):
    """Latent rows whose norm grows along the sequence, selected in
    increasing token order: every later tile of 64 slots raises each head's
    running maximum, many times by more than the kernel's 2^8 slack, so the
    accumulated output and sums are rescaled tile after tile. The input is
    checked to do that before the kernel runs."""
    S, B, H, Dc, T, topk = 6, 1, 64, 256, 640, 640
    scale = 0.5
    g = torch.Generator().manual_seed(12)
    q = torch.randn((S, B, H, Dc), generator=g).to(torch.bfloat16)
    grow = (1.0 + torch.arange(T, dtype=torch.float32) / 40.0)[:, None, None]
    c = (torch.randn((T, B, Dc), generator=g) * grow).to(torch.bfloat16)
    idx = torch.arange(T, dtype=torch.int32).repeat(B, S, 1).contiguous()
    x = scale * math.log2(math.e) * torch.einsum(
        "shd,td->sht", q[:, 0].double(), c[:, 0].double())
    tile_max = x.reshape(S, H, T // 64, 64).amax(dim=3)
    running = torch.cummax(tile_max, dim=2).values
    jumps = (running[:, :, 1:] - running[:, :, :-1]) > 8
    assert jumps.sum(dim=2).min() >= 2
    check(dsa, q, c, idx, scale)
