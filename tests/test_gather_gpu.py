"""GPU parity of the given-indices path (scores at caller-supplied key
indices) against the CPU oracle, through the C ABI.

For H in {16, 32, 64, 128} the scores come from the kernel that gathers the
named key rows and multiplies them on the tensor cores (no logits); other H
read them from written logits.  Rule, slot by slot: the output index equals
the given one; the score is -inf exactly where the oracle's is (index -1,
outside [0, S_kv) or not visible to the row), else within
|g - o| <= 1e-3 + 2e-3 |o|; integer-valued inputs must match bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dsa_inputs import Workload, make_given_indices, make_inputs
from tests.helpers import score_tol

pytestmark = pytest.mark.gpu

RANGE_STATUS = 6  # DSA_ERR_INDEX_RANGE


@pytest.fixture(scope="module")
def dsa():
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    return m


def gpu_run(dsa, q, k, w, ratio, topk, q_pos, in_idx):
    dev = torch.device("cuda")
    pd = q_pos.to(dev) if q_pos is not None else None
    sc, idx, ws = dsa.dsa_indexer_fwd(q.to(dev), k.to(dev), w.to(dev), ratio,
                                      topk, q_pos=pd, in_idx=in_idx.to(dev))
    return sc.cpu().numpy(), idx.cpu().numpy(), dsa.dsa_indexer_check(ws)


def row_nvis(S, B, ratio, S_kv, q_pos=None):
    pos = np.arange(S)[None, :].repeat(B, 0).astype(np.int64)
    if q_pos is not None:
        pos = pos + q_pos.numpy().astype(np.int64)[:, None]
    return np.clip((pos + 1) // ratio, 0, S_kv)


def adversarial_indices(B, S, topk, nv, S_kv, seed):
    """Random visible indices (a permutation prefix per row) with planted
    cases: -1 between valid slots, repeated indices, in-range indices the
    row cannot see, the last visible key, key 0, and a row of only -1."""
    gi = make_given_indices(B, S, topk, nv, seed).numpy()
    rng = np.random.default_rng(seed)
    for b in range(B):
        for s in rng.choice(S, size=min(S, 6), replace=False):
            n = int(nv[b, s])
            e = rng.integers(0, topk, size=4)
            gi[b, s, e[0]] = -1
            if n > 0:
                gi[b, s, e[1]] = n - 1
                gi[b, s, e[2]] = 0
                gi[b, s, e[3]] = gi[b, s, e[1]]  # a repeat
            if n < S_kv:
                gi[b, s, rng.integers(0, topk)] = rng.integers(n, S_kv)
    gi[0, S // 2, :] = -1
    return torch.from_numpy(gi)


def check_against_oracle(sc, idx, gi, ref, topk):
    np.testing.assert_array_equal(idx.reshape(-1, topk),
                                  gi.numpy().reshape(-1, topk))
    o = ref["scores64"]
    g = sc.reshape(-1, topk).astype(np.float64)
    assert np.array_equal(np.isneginf(g), np.isneginf(o)), "masked slots"
    fin = np.isfinite(o)
    err = np.abs(g[fin] - o[fin])
    assert np.all(err <= score_tol(o[fin])), float(err.max())


@pytest.mark.parametrize("S,B,H,D,S_kv,ratio,topk,decode_pos", [
    (200, 2, 64, 128, 300, 1, 300, False),   # ragged last tile of slots
    (97, 1, 16, 64, 250, 2, 129, False),     # H = 16, one slot in tile 2
    (64, 3, 32, 72, 130, 1, 40, False),      # D = 72: half-empty chunk
    (33, 2, 128, 128, 1000, 4, 260, True),   # H = 128
    (5, 1, 64, 128, 9000, 4, 2048, True),    # few rows: rows split in chunks
    (1, 64, 64, 128, 8192, 4, 512, True),    # decode batch
    (70, 2, 8, 32, 90, 1, 20, False),        # H = 8: the logits route
])
def test_given_indices_match_oracle(dsa, S, B, H, D, S_kv, ratio, topk,
                                    decode_pos):
    wl = Workload("g", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=S * 7 + H + D)
    q, k, w, _ = make_inputs(wl)
    pos = None
    if decode_pos:
        rng = np.random.default_rng(S_kv + B)
        pos = torch.from_numpy(
            rng.integers(0, S_kv * ratio, size=B).astype(np.int32))
    nv = row_nvis(S, B, ratio, S_kv, pos)
    gi = adversarial_indices(B, S, topk, nv, S_kv, seed=S + topk)
    sc, idx, st = gpu_run(dsa, q, k, w, ratio, topk, pos, gi)
    assert st == 0
    ref = oracle.indexer_fwd(q, k, w, ratio, topk, q_pos=pos, in_idx=gi)
    check_against_oracle(sc, idx, gi, ref, topk)


@pytest.mark.parametrize("H,D", [(64, 128), (16, 32), (128, 64)])
def test_given_indices_integer_inputs_bit_exact(dsa, H, D):
    """Integer q, k and dyadic w: every score is exact in fp32, whatever the
    order of the sums, so the gathered scores equal the oracle's exactly."""
    rng = np.random.default_rng(H + D)
    S, B, S_kv, topk = 150, 2, 150, 140
    qi = rng.integers(-3, 4, size=(S, B, H, D)).astype(np.float32)
    ki = rng.integers(-3, 4, size=(S_kv, B, D)).astype(np.float32)
    wi = rng.choice([1, -1, 0.5, -0.5, 0.25, -0.25],
                    size=(S, B, H)).astype(np.float32)
    q = torch.from_numpy(qi).to(torch.bfloat16)
    k = torch.from_numpy(ki).to(torch.bfloat16)
    w = torch.from_numpy(wi)
    nv = row_nvis(S, B, 1, S_kv)
    gi = adversarial_indices(B, S, topk, nv, S_kv, seed=H * D)
    sc, idx, st = gpu_run(dsa, q, k, w, 1, topk, None, gi)
    assert st == 0
    ref = oracle.indexer_fwd(q, k, w, 1, topk, in_idx=gi)
    np.testing.assert_array_equal(idx.reshape(-1, topk), ref["idx"])
    np.testing.assert_array_equal(sc.reshape(-1, topk), ref["scores"])


def test_given_indices_out_of_range_flagged_tensor_path(dsa):
    wl = Workload("g", B=2, S=40, S_kv=300, H=64, D=128, compress_ratio=1,
                  topk=150, w_scale=0.125, seed=9)
    q, k, w, _ = make_inputs(wl)
    gi = torch.full((wl.B, wl.S, wl.topk), -1, dtype=torch.int32)
    gi[0, 10, 0] = 3
    gi[0, 10, 1] = wl.S_kv       # past the end
    gi[1, 39, 149] = -5          # below -1, in the ragged last tile
    gi[1, 39, 0] = 2 ** 31 - 1
    sc, idx, st = gpu_run(dsa, q, k, w, 1, wl.topk, None, gi)
    assert st == RANGE_STATUS
    assert np.isneginf(sc[0, 10, 1]) and np.isneginf(sc[1, 39, 149])
    assert np.isneginf(sc[1, 39, 0])
    assert np.isfinite(sc[0, 10, 0])
    assert idx[0, 10, 1] == wl.S_kv and idx[1, 39, 149] == -5
    assert idx[1, 39, 0] == 2 ** 31 - 1
    # the next call with clean indices reports no error
    gi[0, 10, 1] = gi[1, 39, 149] = gi[1, 39, 0] = -1
    assert gpu_run(dsa, q, k, w, 1, wl.topk, None, gi)[2] == 0
