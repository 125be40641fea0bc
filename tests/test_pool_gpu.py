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
kernel from fp32; about one value in a thousand lies so close to a rounding
midpoint that the two land on neighbouring bf16 values, and over thousands
of pools those flips can move a score past the forward's tolerance.  So the
forward-level cases use slot logits that are equal within a pool (random
per pool and channel): the pooled key is then an exact mean, both sides
round the same value, and the score comparison is the forward's own.  The
general softmax (random logits per slot) is checked by the compression
test.
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


def check_pooled(dsa, S, B, H, D, T, kpool, first_key, index_topk, seed,
                 invalid=0.0, q_pos=None):
    # exact means need kpool a power of two (the division by kpool is exact)
    assert kpool in (1, 2, 4, 8)
    q, k, gate, ape, w, valid = pool_problem(S, B, H, D, T, kpool, seed,
                                             invalid, equal=True)
    if first_key % kpool:
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
    for r in range(B * S):
        msg = compare_topk_row(gi[r], gs[r], ref["idx"][r],
                               ref["scores64"][r], ref["next"][r],
                               ref["logits"][r])
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
