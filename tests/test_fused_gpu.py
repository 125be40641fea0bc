"""GPU parity of the one-kernel prefill forward (scores and top-k in the
same kernel, the scores never written to device memory) and of the routes
its selection takes, against the CPU oracle; the one-kernel forward is
forced here wherever the shape fits it.

Every row is compared with tests.helpers.compare_topk_row: scores slot by
slot within |g - o| <= 1e-3 + 2e-3 |o|, each returned score the oracle score
of the index in the same slot, -1 / -inf padding identical, index sets
equal away from near-ties.  Integer-valued inputs (every score exact in
fp32 on both sides) must match bit for bit, tie order included.

Routes (the selection picks one per row):
  fast, registers  rows of at most 4096 visible keys, held in registers
  fast, L2         longer rows, read twice from the L2-resident scratch
  exact            rows whose kept buckets are crowded (ties, an outlier)
and, outside the one-kernel envelope (H not in {32, 64, 128}, topk > 2048,
decode-shaped rows), the written-logits path whose selection keeps short
rows in registers, stages long rows in shared memory when there are few
rows, and re-reads them from L2 when there are many.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dsa_inputs import Workload, make_inputs
from tests.helpers import compare_topk_row

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    """The library with the one-kernel prefill forced wherever the shape fits
    it (the default policy keeps it for rows of at least 8192 keys); the
    default is restored afterwards."""
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    m.dsa_set_prefill_policy(m.PREFILL_ONE_KERNEL)
    yield m
    m.dsa_set_prefill_policy(m.PREFILL_AUTO)


def run_and_compare(dsa, q, k, w, ratio, topk, q_pos=None, exact=False):
    dev = torch.device("cuda")
    S, B = q.shape[0], q.shape[1]
    pd = q_pos.to(dev) if q_pos is not None else None
    sc, idx, ws = dsa.dsa_indexer_fwd(q.to(dev), k.to(dev), w.to(dev), ratio,
                                      topk, q_pos=pd)
    assert dsa.dsa_indexer_check(ws) == 0
    sc = sc.cpu().numpy().reshape(B * S, topk)
    idx = idx.cpu().numpy().reshape(B * S, topk)
    ref = oracle.indexer_fwd(q, k, w, ratio, topk, q_pos=q_pos,
                             want_logits=not exact)
    if exact:
        np.testing.assert_array_equal(idx, ref["idx"])
        np.testing.assert_array_equal(sc, ref["scores"])
        return ref
    bad = []
    for r in range(B * S):
        msg = compare_topk_row(idx[r], sc[r], ref["idx"][r],
                               ref["scores64"][r], ref["next"][r],
                               ref["logits"][r])
        if msg:
            bad.append((r, msg))
    assert not bad, bad[:5]
    return ref


def deep_positions(B, S, S_kv, ratio, lo_keys, seed):
    """Per-sequence first positions giving every row between lo_keys and
    S_kv visible keys."""
    rng = np.random.default_rng(seed)
    lo = lo_keys * ratio
    hi = max(lo + 1, S_kv * ratio - S)
    pos = rng.integers(lo, hi, size=B)
    return torch.from_numpy(pos.astype(np.int32))


@pytest.mark.parametrize("S,B,H,D,S_kv,ratio,topk,lo_keys", [
    (96, 2, 64, 128, 4096, 1, 2048, 2500),   # fast route, registers
    (64, 2, 64, 128, 9000, 4, 2048, 4200),   # fast route, rows from L2
    (40, 1, 64, 128, 16384, 4, 2048, 12000),  # the long-context row lengths
    (48, 1, 64, 128, 6000, 1, 512, 4500),    # smaller topk, rows from L2
])
def test_fused_routes_real_valued(dsa, S, B, H, D, S_kv, ratio, topk,
                                  lo_keys):
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=S + S_kv)
    q, k, w, _ = make_inputs(wl)
    pos = deep_positions(B, S, S_kv, ratio, lo_keys, seed=S_kv)
    run_and_compare(dsa, q, k, w, ratio, topk, q_pos=pos)


@pytest.mark.parametrize("topk", [512, 2048])
def test_fused_bucket_count_boundaries(dsa, topk):
    """The register route sizes its buckets to the row (1024, 2048 or 4096
    for rows of at most that many keys; longer rows are read from L2).
    Three sequences starting 100 rows below each boundary give rows of every
    length across 1024, 2048 and 4096 visible keys."""
    H, D, S, S_kv = 64, 128, 200, 4200
    wl = Workload("t", B=3, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=1,
                  topk=topk, w_scale=H ** -0.5, seed=topk + 11)
    q, k, w, _ = make_inputs(wl)
    pos = torch.tensor([1024 - 101, 2048 - 101, 4096 - 101],
                       dtype=torch.int32)
    run_and_compare(dsa, q, k, w, 1, topk, q_pos=pos)


@pytest.mark.parametrize("S,B,H,D,S_kv,ratio,topk", [
    (300, 2, 32, 128, 300, 1, 50),     # H = 32: 8 rows per work item
    (260, 1, 128, 128, 500, 2, 64),    # H = 128: 2 rows per work item
    (300, 1, 64, 64, 300, 1, 40),      # D = 64: one 64-column chunk
    (200, 2, 64, 72, 180, 3, 33),      # D = 72: a zero-filled second chunk
    (150, 1, 64, 128, 40, 8, 16),      # ratio 8: leading items see no key
    (520, 1, 64, 128, 520, 1, 2048),   # topk above every row's key count
])
def test_fused_shapes(dsa, S, B, H, D, S_kv, ratio, topk):
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=3 * S + H + D)
    q, k, w, _ = make_inputs(wl)
    run_and_compare(dsa, q, k, w, ratio, topk)


@pytest.mark.parametrize("H,topk,distinct", [(64, 60, None), (32, 100, None),
                                             (128, 16, None), (64, 200, 8)])
def test_fused_exact_route_ties_bit_exact(dsa, H, topk, distinct):
    """Integer q, k and dyadic w: every score is exact and ties are common,
    so the kept buckets crowd and the exact route runs; order must match the
    oracle exactly.  With 8 distinct key vectors whole rows tie."""
    rng = np.random.default_rng(H + topk)
    S, B, S_kv, D = 260, 2, 250, 32
    qi = rng.integers(-2, 3, size=(S, B, H, D)).astype(np.float32)
    ki = rng.integers(-2, 3, size=(S_kv, B, D)).astype(np.float32)
    if distinct:
        ki = ki[np.arange(S_kv) % distinct]
    wi = rng.choice([1, -1, 0.5, -0.5], size=(S, B, H)).astype(np.float32)
    run_and_compare(dsa, torch.from_numpy(qi).to(torch.bfloat16),
                    torch.from_numpy(ki).to(torch.bfloat16),
                    torch.from_numpy(wi), 1, topk, exact=True)


@pytest.mark.parametrize("outlier", [2048.0, -2048.0])
def test_fused_far_outlier_bit_exact(dsa, outlier):
    """One key vector scaled far beyond the rest stretches each row's range
    so the other keys crowd into a few buckets: those rows take the exact
    route.  Integer inputs keep every score exact."""
    rng = np.random.default_rng(5)
    S, B, S_kv, H, D, topk = 300, 2, 290, 64, 32, 60
    qi = rng.integers(-2, 3, size=(S, B, H, D)).astype(np.float32)
    ki = rng.integers(-2, 3, size=(S_kv, B, D)).astype(np.float32)
    ki[3] *= outlier
    wi = rng.choice([1, -1, 0.5, -0.5], size=(S, B, H)).astype(np.float32)
    run_and_compare(dsa, torch.from_numpy(qi).to(torch.bfloat16),
                    torch.from_numpy(ki).to(torch.bfloat16),
                    torch.from_numpy(wi), 1, topk, exact=True)


def test_fused_long_rows_exact_route_real_valued(dsa):
    """Rows of 5000-8000 keys where one key vector is scaled 64x: its score
    stretches every row's range so the kept keys crowd a few buckets and the
    exact route runs on long rows read from L2; real-valued inputs are
    compared by the tolerance rule."""
    S, B, S_kv, H, D, ratio, topk = 32, 1, 8000, 64, 128, 1, 2048
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=99)
    q, k, w, _ = make_inputs(wl)
    k = k.clone()
    k[10] = (k[10].float() * 64).to(torch.bfloat16)
    pos = deep_positions(B, S, S_kv, ratio, 5000, seed=1)
    run_and_compare(dsa, q, k, w, ratio, topk, q_pos=pos)


@pytest.mark.parametrize("S,B,H,S_kv,ratio,topk,lo_keys", [
    (64, 1, 16, 9000, 1, 512, 5000),     # few rows: rows staged in smem
    (2048, 1, 16, 5000, 1, 256, 4200),   # many rows: rows re-read from L2
    (256, 1, 64, 6000, 1, 3000, 4500),   # topk above the one-kernel limit
])
def test_written_logits_routes_real_valued(dsa, S, B, H, S_kv, ratio, topk,
                                           lo_keys):
    """Shapes outside the one-kernel envelope write logits and select in a
    second kernel; rows over 4096 keys take its staged or L2 routes."""
    D = 128
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=S_kv + S)
    q, k, w, _ = make_inputs(wl)
    pos = deep_positions(B, S, S_kv, ratio, lo_keys, seed=S)
    run_and_compare(dsa, q, k, w, ratio, topk, q_pos=pos)


def test_fused_matches_written_logits_path(dsa):
    """The one-kernel forward and the scores-then-select path (reached here
    through the logits entry point plus a host-side selection of the same
    rule) agree on every row's index set and scores."""
    wl = Workload("t", B=2, S=200, S_kv=200, H=64, D=128, compress_ratio=1,
                  topk=32, w_scale=0.125, seed=11)
    q, k, w, _ = make_inputs(wl)
    dev = torch.device("cuda")
    sc, idx, ws = dsa.dsa_indexer_fwd(q.to(dev), k.to(dev), w.to(dev), 1, 32)
    assert dsa.dsa_indexer_check(ws) == 0
    L = dsa.indexer_logits(q.to(dev), k.to(dev), w.to(dev), 1)
    torch.cuda.synchronize()
    L = L.cpu().reshape(2 * 200, 200)
    sc = sc.cpu().reshape(400, 32)
    idx = idx.cpu().reshape(400, 32)
    for r in range(400):
        row = L[r]
        nv = int(torch.isfinite(row).sum())
        kk = min(32, nv)
        # the same rule on the written logits: score desc, index asc
        order = sorted(range(nv), key=lambda j: (-float(row[j]), j))[:kk]
        assert idx[r, :kk].tolist() == order, r
        assert torch.equal(sc[r, :kk], row[order]), r
        assert bool((idx[r, kk:] == -1).all())


@pytest.mark.parametrize("name,per_batch", [("v32_prefill", 24),
                                            ("c4_prefill", 12)])
def test_fused_full_size_sampled(dsa, name, per_batch):
    """The 4096 x 4096 and C4 prefills through the one-kernel forward (the
    default policy gives them the two-kernel forward), sampled rows against
    the oracle."""
    from dsa_inputs import WORKLOADS
    wl = WORKLOADS[name]
    q, k, w, _ = make_inputs(wl)
    dev = torch.device("cuda")
    sc, idx, ws = dsa.dsa_indexer_fwd(q.to(dev), k.to(dev), w.to(dev),
                                      wl.compress_ratio, wl.topk)
    assert dsa.dsa_indexer_check(ws) == 0
    sc = sc.cpu().numpy().reshape(wl.B * wl.S, wl.topk)
    idx = idx.cpu().numpy().reshape(wl.B * wl.S, wl.topk)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([
        [0, 1, wl.S - 1, wl.B * wl.S - 1],
        rng.integers(0, wl.B * wl.S, size=per_batch * wl.B)])).astype(np.int64)
    ref = oracle.indexer_fwd(q, k, w, wl.compress_ratio, wl.topk, rows=rows,
                             want_logits=True)
    for n, r in enumerate(rows):
        msg = compare_topk_row(idx[r], sc[r], ref["idx"][n],
                               ref["scores64"][n], ref["next"][n],
                               ref["logits"][n])
        assert msg is None, (int(r), msg)


def test_one_and_two_kernel_paths_agree(dsa):
    """The same problem through both prefill paths: identical indices, and
    scores equal (both take the same tensor-core products and the same
    epilogue arithmetic)."""
    wl = Workload("t", B=2, S=700, S_kv=2500, H=64, D=128, compress_ratio=4,
                  topk=256, w_scale=0.125, seed=21)
    q, k, w, _ = make_inputs(wl)
    dev = torch.device("cuda")
    outs = []
    for pol in (dsa.PREFILL_ONE_KERNEL, dsa.PREFILL_TWO_KERNELS):
        dsa.dsa_set_prefill_policy(pol)
        sc, idx, ws = dsa.dsa_indexer_fwd(q.to(dev), k.to(dev), w.to(dev),
                                          4, 256)
        assert dsa.dsa_indexer_check(ws) == 0
        outs.append((sc.cpu(), idx.cpu()))
    dsa.dsa_set_prefill_policy(dsa.PREFILL_ONE_KERNEL)
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][0], outs[1][0])


def test_two_kernel_path_in_several_chunks(dsa):
    """More query rows than one 64 MiB logits chunk holds: the two-kernel
    forward scores and selects chunk after chunk; rows on both sides of each
    chunk boundary are compared with the oracle, every row's invariants
    checked."""
    wl = Workload("t", B=2, S=2600, S_kv=4096, H=64, D=128, compress_ratio=1,
                  topk=64, w_scale=0.125, seed=33)
    q, k, w, _ = make_inputs(wl)
    assert dsa.dsa_indexer_fwd_launches(wl.S, wl.B, wl.H, wl.D, wl.S_kv, 1,
                                        wl.topk) == 1  # one kernel (forced)
    dsa.dsa_set_prefill_policy(dsa.PREFILL_TWO_KERNELS)
    try:
        # 2 x 4096 x 4 bytes per row: 2048 rows per chunk, two chunks
        assert dsa.dsa_indexer_fwd_launches(wl.S, wl.B, wl.H, wl.D, wl.S_kv,
                                            1, wl.topk) == 4
        dev = torch.device("cuda")
        sc, idx, ws = dsa.dsa_indexer_fwd(q.to(dev), k.to(dev), w.to(dev), 1,
                                          wl.topk)
        assert dsa.dsa_indexer_check(ws) == 0
    finally:
        dsa.dsa_set_prefill_policy(dsa.PREFILL_ONE_KERNEL)
    sc = sc.cpu().numpy().reshape(wl.B * wl.S, wl.topk)
    idx = idx.cpu().numpy().reshape(wl.B * wl.S, wl.topk)
    nv = np.minimum(np.arange(wl.S) + 1, wl.S_kv)
    for b in range(wl.B):
        rb = slice(b * wl.S, (b + 1) * wl.S)
        kept = np.minimum(nv, wl.topk)
        assert np.array_equal((idx[rb] >= 0).sum(-1), kept)
    rows = np.array([0, 1, 2047, 2048, 2049, 2599, 2600, 2600 + 2047,
                     2600 + 2048, 5199], dtype=np.int64)
    ref = oracle.indexer_fwd(q, k, w, 1, wl.topk, rows=rows, want_logits=True)
    for n, r in enumerate(rows):
        msg = compare_topk_row(idx[r], sc[r], ref["idx"][n],
                               ref["scores64"][n], ref["next"][n],
                               ref["logits"][n])
        assert msg is None, (int(r), msg)
