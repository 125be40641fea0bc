"""GPU parity of the pool variant (page "Module glm5next_dsa": kpool_compress
-> index_scores -> topk_pools -> expand_selection) against the fp64 oracle,
through the C ABI.

Rules: pooled keys |gpu - oracle| <= 2^-8 |oracle| + 1e-6 (the kernel
computes in fp32 and rounds once to bf16, half a bf16 ulp is at most 2^-8
of the value) and the pool flags bit for bit; expansion bit for bit; the
pooled top-k row by row with the forward's rule (scores within
1e-3 + 2e-3 |o|, index sets equal away from near-ties), token ids equal to
the expansion of the GPU's own pool ids, and the -1 slots where the oracle
has them.

Both sides round the pooled keys to bf16, the oracle from fp64 and the
kernel from fp32, so a pooled-key element whose exact value lies within the
kernel's fp32 error of a bf16 rounding midpoint may land on the neighbouring
bf16 value.  The forward-level cases run on general slot logits (random per
token and channel, plus a random per-slot embedding) and allow for exactly
those elements: from the oracle's own fp64 keys alone, an element is at risk
when its distance to the nearest bf16 rounding boundary is at most
2^-19 * max_s |k_s|.  That is the kernel's fp32 error bound: the slot
weights come from expf (at most 2 ulp, 2^-22 relative) and one division,
the weighted sum and the normaliser from at most 8 roundings each
(8 * 2^-24 = 2^-21 of the sum of magnitudes), in all under 2^-19 of
sum_s p_s |k_s| <= max_s |k_s|.  Such an element has one alternative, the
bf16 neighbour across that boundary; the allowance of a (query, pool) score
is the largest change of the oracle's score over every subset of the pool's
at-risk elements taking its alternative (exact, in fp64; the 1-Lipschitz
bound of ReLU when a pool has more than six).  It is added to the forward's
tolerance of that pool's score.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import compare_topk_row

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    return m


def pool_problem(S, B, H, D, T, kpool, seed, invalid=0.0, equal=False):
    """Seeded per-token keys, gates, slot embeddings, validity, queries and
    weights with the workloads' distributions.  equal=True: the gate is
    constant within each pool (from token 0) and the slot embedding zero,
    so every pool's softmax weights are exactly 1/kpool."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((S, B, H, D), generator=g).to(torch.bfloat16)
    k = torch.randn((T, B, D), generator=g).to(torch.bfloat16)
    gate = torch.randn((T, B, D), generator=g)
    ape = torch.randn((kpool, D), generator=g) * 0.5
    if equal:
        gate = gate[(torch.arange(T) // kpool) * kpool].contiguous()
        ape = torch.zeros((kpool, D))
    w = torch.randn((S, B, H), generator=g) * H ** -0.5
    valid = None
    if invalid > 0:
        valid = torch.from_numpy(
            (np.random.default_rng(seed).random((T, B)) >= invalid).astype(
                np.uint8))
    return q, k, gate, ape, w, valid


def to_dev(*ts):
    d = torch.device("cuda")
    return [None if t is None else t.to(d) for t in ts]


@pytest.mark.parametrize("T,B,D,kpool,first_key,invalid", [
    (103, 2, 128, 4, 0, 0.05),
    (64, 3, 64, 8, 3, 0.0),
    (50, 1, 32, 1, 0, 0.2),
    (77, 2, 96, 3, 10, 0.1),
])
def test_kpool_compress_matches_oracle(dsa, T, B, D, kpool, first_key,
                                       invalid):
    _, k, gate, ape, _, valid = pool_problem(4, B, 4, D, T, kpool, T + D,
                                             invalid)
    kd, gd, ad, vd = to_dev(k, gate, ape, valid)
    keys, pv = dsa.dsa_kpool_compress(kd, gd, ad, kpool, first_key, valid=vd)
    torch.cuda.synchronize()
    ref = oracle.kpool_compress(k, gate, ape, valid, kpool, first_key)
    assert keys.shape[0] == ref["P"]
    got = keys.float().cpu().numpy().astype(np.float64)
    o = ref["keys"]
    assert np.all(np.abs(got - o) <= 2.0 ** -8 * np.abs(o) + 1e-6)
    # the same bf16 as the oracle's own rounding, except rare fp32 ties
    same = keys.cpu().view(torch.int16).numpy().view(np.uint16) == \
        oracle.round_bf16(o)
    assert same.mean() > 0.999
    np.testing.assert_array_equal(pv.cpu().numpy(), ref["valid"])


def test_expand_selection_matches_oracle(dsa):
    rng = np.random.default_rng(4)
    pools = rng.integers(-1, 500, size=(3, 70, 16)).astype(np.int32)
    for kpool, fk in ((4, 0), (3, 11), (8, 2)):
        got = dsa.dsa_expand_selection(torch.from_numpy(pools).cuda(), kpool,
                                       fk).cpu().numpy()
        np.testing.assert_array_equal(got,
                                      oracle.expand_selection(pools, kpool,
                                                              fk))


def rounding_allowance(q, k, gate, ape, valid, w, kpool, first_key,
                       max_exact=6):
    """[B*S, P] score allowance per (row, pool) for pooled-key elements the
    two sides may round to different bf16 neighbours (module docstring),
    computed from the oracle's fp64 pooled keys only.

    An element at risk has one alternative: the bf16 neighbour of the
    oracle's rounding across the rounding boundary nearest to the exact
    value.  For a pool with at most `max_exact` elements at risk the
    allowance is the exact largest change of the score over every subset of
    them taking its alternative, in fp64 from the oracle's own keys; with
    more it is the 1-Lipschitz bound sum_h |w_h| sum_d |q_hd| |delta_d|."""
    c = oracle.kpool_compress(k, gate, ape, valid, kpool, first_key)
    P = c["P"]
    S, B, H, D = q.shape
    if P == 0:
        return np.zeros((B * S, 0))
    x = c["keys"]                                         # [P, B, D] fp64
    rb = oracle.round_bf16(x)                             # bf16 bit patterns
    r = (rb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    _, e = np.frexp(np.abs(x))
    dist = np.ldexp(1.0, e - 9) - np.abs(x - r)  # to the nearest boundary
    kr = k.float().numpy().astype(np.float64)             # [T, B, D]
    tok = first_key + np.arange(P)[:, None] * kpool + np.arange(kpool)
    kmax = np.abs(kr[tok]).max(axis=1)                    # [P, B, D]
    risk = (dist <= 2.0 ** -19 * kmax) & (rb & 0x7fff != 0)
    # the neighbour across that boundary: one step of the magnitude bits
    # away from zero when |x| > |r|, towards zero otherwise
    step = np.where(np.abs(x) > np.abs(r), 1, -1).astype(np.int32)
    alt_bits = ((rb & 0x8000) | ((rb & 0x7fff).astype(np.int32) + step))
    alt = (alt_bits.astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)
    delta = np.where(risk, alt - r, 0.0)                  # [P, B, D]
    qf = q.float().numpy().astype(np.float64)             # [S, B, H, D]
    wf = w.numpy().astype(np.float64)                     # [S, B, H]
    out = np.zeros((B, S, P))
    for b in range(B):
        qb, wb = qf[:, b], wf[:, b]
        dots = (qb.reshape(S * H, D) @ r[:, b].T).reshape(S, H, P)
        for p in np.flatnonzero(risk[:, b].any(axis=1)):
            dims = np.flatnonzero(risk[p, b])
            dq = qb[:, :, dims] * delta[p, b, dims]        # [S, H, m]
            if dims.size > max_exact:
                out[b, :, p] = np.abs(wb[:, :, None] * dq).sum(axis=(1, 2))
                continue
            a = dots[:, :, p]
            base = np.maximum(a, 0.0)
            worst = np.zeros(S)
            for mask in range(1, 1 << dims.size):
                sel = [i for i in range(dims.size) if mask >> i & 1]
                moved = np.maximum(a + dq[:, :, sel].sum(axis=2), 0.0)
                worst = np.maximum(worst,
                                   np.abs((wb * (moved - base)).sum(axis=1)))
            out[b, :, p] = worst * (1 + 1e-9) + 1e-12
    return out.reshape(B * S, P)


def check_pooled(dsa, S, B, H, D, T, kpool, first_key, index_topk, seed,
                 invalid=0.0, q_pos=None, equal=False):
    q, k, gate, ape, w, valid = pool_problem(S, B, H, D, T, kpool, seed,
                                             invalid, equal=equal)
    if equal and first_key % kpool:
        # re-align the constant runs to the pools that start at first_key
        idx = torch.arange(T)
        src = torch.where(idx >= first_key,
                          first_key + ((idx - first_key) // kpool) * kpool,
                          idx)
        gate = gate[src].contiguous()
    qd, kd, gd, ad, wd, vd = to_dev(q, k, gate, ape, w, valid)
    pd = None if q_pos is None else q_pos.cuda()
    tok, pools, sc, ws = dsa.dsa_indexer_fwd_pooled(
        qd, kd, gd, ad, wd, kpool, first_key, index_topk, valid=vd, q_pos=pd)
    assert dsa.dsa_indexer_check(ws) == 0
    tok, pools, sc = tok.cpu().numpy(), pools.cpu().numpy(), sc.cpu().numpy()
    ref = oracle.indexer_pooled_fwd(q, k, gate, ape, valid, w, kpool,
                                    first_key, index_topk, q_pos=q_pos,
                                    want_logits=True)
    sk = index_topk // kpool
    gi, gs = pools.reshape(B * S, sk), sc.reshape(B * S, sk)
    extra = None if equal else rounding_allowance(q, k, gate, ape, valid, w,
                                                  kpool, first_key)
    for r in range(B * S):
        msg = compare_topk_row(gi[r], gs[r], ref["idx"][r],
                               ref["scores64"][r], ref["next"][r],
                               ref["logits"][r],
                               None if extra is None else extra[r])
        assert not msg, (r, msg)
        # a selected pool is a candidate pool
        b = r // S
        for p in gi[r][gi[r] >= 0]:
            assert ref["pool_valid"][p, b] == 1
    np.testing.assert_array_equal(
        tok, oracle.expand_selection(pools, kpool, first_key))
    return ref


@pytest.mark.parametrize("S,B,T,kpool,first_key,topk,invalid", [
    # prefill, some invalid tokens (hence invalid pools), ragged tiles
    (300, 2, 300, 4, 0, 64, 0.02),
    # pools from an odd first_key on (positions shift by first_key)
    (200, 1, 230, 2, 7, 48, 0.0),
    # one-token pools: the plain forward with a validity mask
    (129, 2, 129, 1, 0, 40, 0.1),
    # more pools wanted than exist for most rows: -1 tails
    (90, 1, 90, 8, 0, 128, 0.0),
])
def test_pooled_forward_matches_oracle(dsa, S, B, T, kpool, first_key, topk,
                                       invalid):
    check_pooled(dsa, S, B, 64, 128, T, kpool, first_key, topk,
                 seed=S + T + kpool, invalid=invalid)


def test_pooled_forward_decode_rows(dsa):
    """One query per sequence at positions from q_pos (the decode kernel),
    invalid tokens included."""
    B, T, kpool = 8, 2048, 4
    pos = torch.from_numpy(np.random.default_rng(9).integers(
        100, T, size=B).astype(np.int32))
    check_pooled(dsa, 1, B, 64, 128, T, kpool, 2, 128, seed=31,
                 invalid=0.01, q_pos=pos)


def test_pooled_forward_long_rows(dsa):
    """8192 pools per row: rows past the register-held selection (keys
    read from L2), with some pools masked invalid."""
    S, B, T, kpool = 64, 1, 32800, 4
    pos = torch.tensor([T - S], dtype=torch.int32)
    check_pooled(dsa, S, B, 64, 128, T, kpool, 0, 2048, seed=41,
                 invalid=0.001, q_pos=pos)


def test_pooled_forward_without_whole_pools(dsa):
    """Fewer tokens than one pool after first_key: every slot empty."""
    q, k, gate, ape, w, _ = pool_problem(5, 2, 64, 128, 6, 4, 3)
    qd, kd, gd, ad, wd = to_dev(q, k, gate, ape, w)
    tok, pools, sc, ws = dsa.dsa_indexer_fwd_pooled(qd, kd, gd, ad, wd, 4, 3,
                                                    8)
    assert dsa.dsa_indexer_check(ws) == 0
    assert torch.all(tok.cpu() == -1) and torch.all(pools.cpu() == -1)
    assert torch.all(torch.isneginf(sc.cpu()))
