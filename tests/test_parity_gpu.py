"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs.

Rule: scores within |g - o| <= 1e-3 + 2e-3 |o| slot by slot; -1 / -inf
slots identical; index sets equal unless the oracle's k-th and (k+1)-th
scores are closer than that tolerance (then the near-tie rule of
tests.helpers.compare_topk_row applies).  Integer-valued inputs, where every
score is exact in fp32, must match bit for bit, tie order included.
Full-size configurations are compared on sampled rows (the oracle computes
them one by one) plus invariants checked on every row.
"""
from __future__ import annotations

import contextlib

import numpy as np
import pytest
import torch

import oracle
from dsa_inputs import WORKLOADS, Workload, make_given_indices, make_inputs
from tests.helpers import compare_topk_row, score_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    return m


def gpu_run(dsa, q, k, w, ratio, topk, q_pos=None, in_idx=None):
    dev = torch.device("cuda")
    qd, kd, wd = q.to(dev), k.to(dev), w.to(dev)
    pd = q_pos.to(dev) if q_pos is not None else None
    gd = in_idx.to(dev) if in_idx is not None else None
    sc, idx, ws = dsa.dsa_indexer_fwd(qd, kd, wd, ratio, topk, q_pos=pd,
                                      in_idx=gd)
    status = dsa.dsa_indexer_check(ws)
    return sc.cpu().numpy(), idx.cpu().numpy(), status


@contextlib.contextmanager
def prefill_policy(dsa, policy):
    """Run a block under a prefill top-k policy, then restore automatic."""
    dsa.dsa_set_prefill_policy(policy)
    try:
        yield
    finally:
        dsa.dsa_set_prefill_policy(dsa.PREFILL_AUTO)


def row_nvis(S, B, ratio, S_kv, q_pos=None):
    pos = np.arange(S)[None, :].repeat(B, 0).astype(np.int64)
    if q_pos is not None:
        pos = pos + q_pos.numpy().astype(np.int64)[:, None]
    return np.clip((pos + 1) // ratio, 0, S_kv)


def check_invariants(sc, idx, nvis, topk):
    """Properties every row must have, checked on all rows."""
    valid = idx >= 0
    want_valid = np.minimum(nvis, topk)
    assert np.array_equal(valid.sum(-1), want_valid), "valid count"
    assert np.array_equal(valid, np.arange(topk)[None, None, :]
                          < want_valid[..., None]), "valid prefix"
    assert np.all(idx[valid] < np.broadcast_to(nvis[..., None],
                                               idx.shape)[valid]), "visible"
    assert np.all(np.isneginf(sc[~valid])), "padding scores"
    assert np.all(np.isfinite(sc[valid])), "finite scores"
    with np.errstate(invalid="ignore"):
        d = np.diff(np.where(valid, sc, -np.inf), axis=-1)
    vv = valid[..., 1:]
    assert np.all(d[vv] <= 0), "non-increasing"
    srt = np.sort(np.where(valid, idx, -1 - np.arange(topk)), axis=-1)
    assert np.all(np.diff(srt, axis=-1) != 0), "distinct"


def compare_rows(sc, idx, ref, rows, S):
    bad = []
    logits = ref["logits"]  # the oracle must be run with want_logits=True
    for n, r in enumerate(rows):
        b, s = divmod(int(r), S)
        msg = compare_topk_row(idx[b, s], sc[b, s], ref["idx"][n],
                               ref["scores64"][n], ref["next"][n],
                               logits[n])
        if msg:
            bad.append((b, s, msg))
    assert not bad, bad[:5]


def sample_rows(B, S, n_per_batch, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(B):
        pick = {0, 1, S - 1, S // 2}
        pick |= set(rng.integers(0, S, size=n_per_batch).tolist())
        rows += [b * S + s for s in sorted(pick)]
    return np.array(rows, dtype=np.int64)


# ---------------------------------------------------------------------------

def test_tiny_full_parity(dsa):
    wl = WORKLOADS["tiny"]
    q, k, w, _ = make_inputs(wl)
    sc, idx, st = gpu_run(dsa, q, k, w, wl.compress_ratio, wl.topk)
    assert st == 0
    ref = oracle.indexer_fwd(q, k, w, wl.compress_ratio, wl.topk,
                             want_logits=True)
    sc = sc.reshape(wl.B, wl.S, wl.topk)
    idx = idx.reshape(wl.B, wl.S, wl.topk)
    check_invariants(sc, idx, row_nvis(wl.S, wl.B, 1, wl.S_kv), wl.topk)
    compare_rows(sc, idx, ref, np.arange(wl.B * wl.S), wl.S)


@pytest.mark.parametrize("H,D,ratio,topk", [(4, 32, 1, 16), (4, 32, 2, 40),
                                            (64, 32, 1, 24), (16, 24, 3, 7)])
def test_integer_inputs_bit_exact(dsa, H, D, ratio, topk):
    """Integer q, k and dyadic w: every score is exact in fp32 on both sides,
    so indices and scores must be identical, tie order included."""
    rng = np.random.default_rng(H * 1000 + D + ratio)
    S, B, S_kv = 300, 2, 290
    qi = rng.integers(-3, 4, size=(S, B, H, D)).astype(np.float32)
    ki = rng.integers(-3, 4, size=(S_kv, B, D)).astype(np.float32)
    wi = rng.choice([1, -1, 0.5, -0.5, 0.25, -0.25],
                    size=(S, B, H)).astype(np.float32)
    q = torch.from_numpy(qi).to(torch.bfloat16)
    k = torch.from_numpy(ki).to(torch.bfloat16)
    w = torch.from_numpy(wi)
    sc, idx, st = gpu_run(dsa, q, k, w, ratio, topk)
    assert st == 0
    ref = oracle.indexer_fwd(q, k, w, ratio, topk)
    np.testing.assert_array_equal(idx.reshape(-1, topk), ref["idx"])
    np.testing.assert_array_equal(sc.reshape(-1, topk), ref["scores"])


@pytest.mark.parametrize("S,B,H,D,S_kv,ratio", [
    (128, 1, 4, 32, 128, 1),      # the tiny shape
    (300, 2, 64, 128, 300, 1),    # several tiles, ragged query/key tails
    (257, 1, 64, 128, 70, 3),     # ratio 3, S_kv < one tile
    (130, 3, 8, 64, 200, 1),      # S_kv > S (keys past every query)
    (64, 1, 1, 16, 64, 1),        # one head: ReLU(QK^T)
    (96, 2, 2, 72, 96, 2),        # D not a multiple of 64
    (40, 1, 128, 128, 40, 1),     # H = 128
])
def test_logits_match_oracle(dsa, S, B, H, D, S_kv, ratio):
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=4, w_scale=H ** -0.5, seed=S + H + D)
    q, k, w, _ = make_inputs(wl)
    logits = dsa.indexer_logits(q.cuda(), k.cuda(), w.cuda(), ratio)
    torch.cuda.synchronize()
    L = logits.cpu().numpy().reshape(B * S, S_kv)
    ref = oracle.indexer_fwd(q, k, w, ratio, 4, want_logits=True)["logits"]
    assert np.array_equal(np.isneginf(L), np.isneginf(ref))
    fin = np.isfinite(ref)
    err = np.abs(L[fin] - ref[fin])
    assert np.all(err <= score_tol(ref[fin])), float(err.max())


@pytest.mark.parametrize("S,B,H,D,S_kv,ratio,topk", [
    (300, 2, 64, 128, 300, 1, 37),
    (257, 1, 64, 128, 70, 3, 100),   # topk > S_kv: every row padded
    (520, 1, 4, 32, 530, 1, 256),
    (1000, 1, 64, 128, 250, 4, 64),
    (64, 3, 16, 64, 64, 2, 1),       # topk = 1
])
def test_topk_match_oracle(dsa, S, B, H, D, S_kv, ratio, topk):
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=7 * S + H)
    q, k, w, _ = make_inputs(wl)
    sc, idx, st = gpu_run(dsa, q, k, w, ratio, topk)
    assert st == 0
    sc = sc.reshape(B, S, topk)
    idx = idx.reshape(B, S, topk)
    check_invariants(sc, idx, row_nvis(S, B, ratio, S_kv), topk)
    ref = oracle.indexer_fwd(q, k, w, ratio, topk, want_logits=True)
    compare_rows(sc, idx, ref, np.arange(B * S), S)


def test_decode_full_parity(dsa):
    wl = WORKLOADS["decode"]
    q, k, w, pos = make_inputs(wl)
    sc, idx, st = gpu_run(dsa, q, k, w, wl.compress_ratio, wl.topk, q_pos=pos)
    assert st == 0
    sc = sc.reshape(wl.B, wl.S, wl.topk)
    idx = idx.reshape(wl.B, wl.S, wl.topk)
    check_invariants(sc, idx, row_nvis(wl.S, wl.B, 4, wl.S_kv, pos), wl.topk)
    ref = oracle.indexer_fwd(q, k, w, wl.compress_ratio, wl.topk, q_pos=pos,
                             want_logits=True)
    compare_rows(sc, idx, ref, np.arange(wl.B * wl.S), wl.S)


@pytest.mark.parametrize("name,per_batch", [("v32_prefill", 40),
                                            ("c4_prefill", 24),
                                            ("long_c4", 16)])
def test_full_size_sampled_parity(dsa, name, per_batch):
    wl = WORKLOADS[name]
    q, k, w, _ = make_inputs(wl)
    sc, idx, st = gpu_run(dsa, q, k, w, wl.compress_ratio, wl.topk)
    assert st == 0
    sc = sc.reshape(wl.B, wl.S, wl.topk)
    idx = idx.reshape(wl.B, wl.S, wl.topk)
    check_invariants(sc, idx, row_nvis(wl.S, wl.B, wl.compress_ratio,
                                       wl.S_kv), wl.topk)
    rows = sample_rows(wl.B, wl.S, per_batch)
    ref = oracle.indexer_fwd(q, k, w, wl.compress_ratio, wl.topk, rows=rows,
                             want_logits=True)
    compare_rows(sc, idx, ref, rows, wl.S)


def test_given_indices_tiny(dsa):
    wl = WORKLOADS["tiny"]
    q, k, w, _ = make_inputs(wl)
    nv = row_nvis(wl.S, wl.B, 1, wl.S_kv)
    gi = make_given_indices(wl.B, wl.S, wl.topk, nv, wl.idx_seed)
    gi[0, 5, 3] = -1
    gi[0, 6, 0] = 100   # in range but not visible at t = 6
    sc, idx, st = gpu_run(dsa, q, k, w, 1, wl.topk, in_idx=gi)
    assert st == 0
    ref = oracle.indexer_fwd(q, k, w, 1, wl.topk, in_idx=gi)
    np.testing.assert_array_equal(idx.reshape(-1, wl.topk), ref["idx"])
    o = ref["scores64"]
    g = sc.reshape(-1, wl.topk).astype(np.float64)
    assert np.array_equal(np.isneginf(g), np.isneginf(o))
    fin = np.isfinite(o)
    assert np.all(np.abs(g[fin] - o[fin]) <= score_tol(o[fin]))


def test_given_indices_out_of_range_flagged(dsa):
    wl = WORKLOADS["tiny"]
    q, k, w, _ = make_inputs(wl)
    gi = torch.full((wl.B, wl.S, wl.topk), -1, dtype=torch.int32)
    gi[0, 10, 0] = 3
    gi[0, 10, 1] = wl.S_kv      # past the end
    gi[0, 11, 2] = -5           # below -1
    sc, idx, st = gpu_run(dsa, q, k, w, 1, wl.topk, in_idx=gi)
    assert st == 6  # DSA_ERR_INDEX_RANGE
    assert np.isneginf(sc[0, 10, 1]) and np.isneginf(sc[0, 11, 2])
    assert np.isfinite(sc[0, 10, 0])
    assert idx[0, 10, 1] == wl.S_kv and idx[0, 11, 2] == -5


def test_given_indices_long_context_sampled(dsa):
    wl = WORKLOADS["long_c4"]
    q, k, w, _ = make_inputs(wl)
    nv = row_nvis(wl.S, wl.B, wl.compress_ratio, wl.S_kv)
    gi = make_given_indices(wl.B, wl.S, wl.topk, nv, wl.idx_seed)
    sc, idx, st = gpu_run(dsa, q, k, w, wl.compress_ratio, wl.topk, in_idx=gi)
    assert st == 0
    np.testing.assert_array_equal(idx, gi.numpy())
    assert np.array_equal(np.isneginf(sc), gi.numpy() < 0)
    rows = sample_rows(wl.B, wl.S, 12, seed=3)
    ref = oracle.indexer_fwd(q, k, w, wl.compress_ratio, wl.topk, in_idx=gi,
                             rows=rows)
    g = sc.reshape(-1, wl.topk)[rows].astype(np.float64)
    o = ref["scores64"]
    fin = np.isfinite(o)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.all(np.abs(g[fin] - o[fin]) <= score_tol(o[fin]))


def test_host_buffers_round_trip(dsa):
    """The public call with host tensors copies in, runs, copies out."""
    wl = WORKLOADS["tiny"]
    q, k, w, _ = make_inputs(wl)
    sc, idx = dsa.v4_lighting_indexer(q.pin_memory(), k.pin_memory(),
                                      w.pin_memory(), 1, wl.topk)
    assert sc.device.type == "cpu" and tuple(idx.shape) == (1, 128, 16)
    sc2, idx2, _ = gpu_run(dsa, q, k, w, 1, wl.topk)
    np.testing.assert_array_equal(idx.numpy(), idx2)
    np.testing.assert_array_equal(sc.numpy(), sc2)


def test_repeat_calls_are_deterministic(dsa):
    wl = WORKLOADS["tiny"]
    q, k, w, _ = make_inputs(wl)
    a = gpu_run(dsa, q, k, w, 1, wl.topk)
    b = gpu_run(dsa, q, k, w, 1, wl.topk)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_wait_limit_reports_timeout(dsa):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert dsa.dsa_selftest_wait_limit(2000, ws) == 0
    assert dsa.dsa_indexer_check(ws) == 5  # DSA_ERR_DEVICE_TIMEOUT
    assert dsa.dsa_indexer_check(ws) == 0  # read-and-clear


@pytest.mark.parametrize("S,B,H,D,S_kv,ratio,topk", [
    (1, 5, 64, 128, 700, 4, 64),
    (3, 4, 32, 64, 300, 2, 40),
    (1, 3, 128, 128, 257, 1, 100),
    (2, 2, 64, 72, 130, 3, 16),
    (1, 8, 64, 128, 4096, 4, 512),
])
def test_decode_path_match_oracle(dsa, S, B, H, D, S_kv, ratio, topk):
    """Shapes with fewer queries per sequence than a prefill tile packs run
    the split-over-keys decode kernel; positions include rows that see no key,
    a partial key tile and more than every key."""
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=S_kv + B + H)
    q, k, w, _ = make_inputs(wl)
    rng = np.random.default_rng(S_kv)
    pos = rng.integers(0, S_kv * ratio + 40, size=B)
    pos[0] = 0
    pos = torch.from_numpy(pos.astype(np.int32))
    sc, idx, st = gpu_run(dsa, q, k, w, ratio, topk, q_pos=pos)
    assert st == 0
    sc = sc.reshape(B, S, topk)
    idx = idx.reshape(B, S, topk)
    check_invariants(sc, idx, row_nvis(S, B, ratio, S_kv, pos), topk)
    ref = oracle.indexer_fwd(q, k, w, ratio, topk, q_pos=pos,
                             want_logits=True)
    compare_rows(sc, idx, ref, np.arange(B * S), S)
    logits = dsa.indexer_logits(q.cuda(), k.cuda(), w.cuda(), ratio,
                                q_pos=pos.cuda())
    torch.cuda.synchronize()
    L = logits.cpu().numpy().reshape(B * S, S_kv)
    R = ref["logits"]
    assert np.array_equal(np.isneginf(L), np.isneginf(R))
    fin = np.isfinite(R)
    assert np.all(np.abs(L[fin] - R[fin]) <= score_tol(R[fin]))


@pytest.mark.parametrize("policy", ["auto", "two"])
@pytest.mark.parametrize("S,B,S_kv,ratio,topk", [
    (42, 2, 9000, 4, 512),    # ragged query tail and key tail
    (9, 1, 8192, 1, 2048),    # exactly 64 key tiles, large topk
])
def test_long_rows(dsa, S, B, S_kv, ratio, topk, policy):
    """Rows of more than 4096 visible keys.  Under the automatic policy
    these shapes (at least 8192 keys) run the one-kernel forward; forced to
    two kernels, fewer rows than SMs take the 512-thread selection, which
    holds rows of up to 8192 keys in registers, 16 per thread, and stages
    longer ones in shared memory.  Query positions deep into the sequence
    give every row thousands of visible keys while keeping the rows few
    enough for the oracle."""
    H, D = 64, 128
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=S_kv + S)
    q, k, w, _ = make_inputs(wl)
    rng = np.random.default_rng(S)
    pos = rng.integers(S_kv * ratio // 2, S_kv * ratio, size=B)
    pos[-1] = S_kv * ratio - S // 2   # the last rows see every key
    pos = torch.from_numpy(pos.astype(np.int32))
    pol = {"auto": dsa.PREFILL_AUTO, "two": dsa.PREFILL_TWO_KERNELS}[policy]
    with prefill_policy(dsa, pol):
        sc, idx, st = gpu_run(dsa, q, k, w, ratio, topk, q_pos=pos)
    assert st == 0
    sc = sc.reshape(B, S, topk)
    idx = idx.reshape(B, S, topk)
    check_invariants(sc, idx, row_nvis(S, B, ratio, S_kv, pos), topk)
    ref = oracle.indexer_fwd(q, k, w, ratio, topk, q_pos=pos,
                             want_logits=True)
    compare_rows(sc, idx, ref, np.arange(B * S), S)


@pytest.mark.parametrize("topk", [512, 2048])
def test_wide_selection_row_length_boundaries(dsa, topk):
    """Fewer rows than SMs take the 512-thread selection, which holds rows
    of up to 4096 keys eight per thread, rows of up to 8192 keys 16 per
    thread, and stages longer rows in shared memory.  Two sequences whose
    positions start just below 4096 and 8192 visible keys give 40 rows
    across both boundaries."""
    H, D, S, S_kv, B = 64, 128, 20, 8300, 2
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=1,
                  topk=topk, w_scale=H ** -0.5, seed=topk + 8300)
    q, k, w, _ = make_inputs(wl)
    pos = torch.tensor([4096 - 11, 8192 - 11], dtype=torch.int32)
    nvis = row_nvis(S, B, 1, S_kv, pos)
    for edge in (4096, 8192):
        assert np.any(nvis == edge) and np.any(nvis == edge + 1)
    # S_kv >= 8192 would run the one-kernel forward under the automatic
    # policy
    with prefill_policy(dsa, dsa.PREFILL_TWO_KERNELS):
        sc, idx, st = gpu_run(dsa, q, k, w, 1, topk, q_pos=pos)
    assert st == 0
    sc = sc.reshape(B, S, topk)
    idx = idx.reshape(B, S, topk)
    check_invariants(sc, idx, nvis, topk)
    ref = oracle.indexer_fwd(q, k, w, 1, topk, q_pos=pos, want_logits=True)
    compare_rows(sc, idx, ref, np.arange(B * S), S)


def test_wide_selection_long_rows_ties_bit_exact(dsa):
    """Integer q, k and dyadic w on few rows of 5000 to 8192 keys: every
    score is exact and heavy ties crowd the fine buckets, so the 512-thread
    selection leaves its register route for the radix route.  Order must
    match the oracle exactly."""
    rng = np.random.default_rng(8192)
    S, B, S_kv, H, D, topk = 6, 2, 8192, 16, 32, 512
    qi = rng.integers(-2, 3, size=(S, B, H, D)).astype(np.float32)
    ki = rng.integers(-2, 3, size=(S_kv, B, D)).astype(np.float32)
    wi = rng.choice([1, -1, 0.5, -0.5], size=(S, B, H)).astype(np.float32)
    q = torch.from_numpy(qi).to(torch.bfloat16)
    k = torch.from_numpy(ki).to(torch.bfloat16)
    w = torch.from_numpy(wi)
    pos = torch.tensor([5000, 8186], dtype=torch.int32)
    # (H = 16 has no one-kernel forward; forced all the same)
    with prefill_policy(dsa, dsa.PREFILL_TWO_KERNELS):
        sc, idx, st = gpu_run(dsa, q, k, w, 1, topk, q_pos=pos)
    assert st == 0
    ref = oracle.indexer_fwd(q, k, w, 1, topk, q_pos=pos)
    np.testing.assert_array_equal(idx.reshape(-1, topk), ref["idx"])
    np.testing.assert_array_equal(sc.reshape(-1, topk), ref["scores"])


@pytest.mark.parametrize("topk", [512, 2048])
def test_selection_bucket_count_boundaries(dsa, topk):
    """The register route sizes its buckets to the row: 1024, 2048 or 4096
    for rows of at most that many keys, and rows past 4096 keys leave the
    registers.  Three sequences whose query positions start just below
    1024, 2048 and 4096 visible keys give 600 rows (the 256-thread
    selection) of every length across each boundary."""
    H, D, S, S_kv = 64, 128, 200, 4200
    B = 3
    wl = Workload("t", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=1,
                  topk=topk, w_scale=H ** -0.5, seed=topk + 7)
    q, k, w, _ = make_inputs(wl)
    # row s of sequence b sees pos_b + s + 1 keys
    pos = torch.tensor([1024 - 101, 2048 - 101, 4096 - 101],
                       dtype=torch.int32)
    nvis = row_nvis(S, B, 1, S_kv, pos)
    for edge in (1024, 2048, 4096):
        assert np.any(nvis == edge) and np.any(nvis == edge + 1)
    sc, idx, st = gpu_run(dsa, q, k, w, 1, topk, q_pos=pos)
    assert st == 0
    sc = sc.reshape(B, S, topk)
    idx = idx.reshape(B, S, topk)
    check_invariants(sc, idx, nvis, topk)
    ref = oracle.indexer_fwd(q, k, w, 1, topk, q_pos=pos, want_logits=True)
    compare_rows(sc, idx, ref, np.arange(B * S), S)


@pytest.mark.parametrize("topk,distinct_keys", [(7, None), (100, None),
                                                (300, None), (100, 8),
                                                (300, 8)])
def test_integer_inputs_bit_exact_few_rows(dsa, topk, distinct_keys):
    """Fewer rows than SMs take the 512-thread selection.  Integer q, k and
    dyadic w make every score exact and produce runs of tied scores; with
    only 8 distinct key vectors the runs exceed the fix-up's limit and the
    full-sort fallback runs.  Order must match the oracle exactly."""
    rng = np.random.default_rng(topk)
    S, B, S_kv, H, D = 40, 2, 400, 16, 32
    qi = rng.integers(-2, 3, size=(S, B, H, D)).astype(np.float32)
    ki = rng.integers(-2, 3, size=(S_kv, B, D)).astype(np.float32)
    if distinct_keys:
        ki = ki[np.arange(S_kv) % distinct_keys]
    wi = rng.choice([1, -1, 0.5, -0.5], size=(S, B, H)).astype(np.float32)
    q = torch.from_numpy(qi).to(torch.bfloat16)
    k = torch.from_numpy(ki).to(torch.bfloat16)
    w = torch.from_numpy(wi)
    pos = torch.tensor([200, 355], dtype=torch.int32)
    sc, idx, st = gpu_run(dsa, q, k, w, 1, topk, q_pos=pos)
    assert st == 0
    ref = oracle.indexer_fwd(q, k, w, 1, topk, q_pos=pos)
    np.testing.assert_array_equal(idx.reshape(-1, topk), ref["idx"])
    np.testing.assert_array_equal(sc.reshape(-1, topk), ref["scores"])


@pytest.mark.parametrize("S,B,outlier", [(300, 2, 2048.0), (300, 2, -2048.0),
                                         (40, 2, 2048.0)])
def test_far_outlier_rows_bit_exact(dsa, S, B, outlier):
    """One key vector scaled far beyond the rest: its scores stretch each
    row's value range so that the other keys crowd into a few of the fine
    buckets, and those rows must leave the bucket route for the radix
    route.  Integer q, k and dyadic w keep every score exact, so the order
    must match the oracle exactly (many rows: 256-thread selection; 80 rows:
    512-thread selection)."""
    rng = np.random.default_rng(77 + S)
    H, D, S_kv, topk = 16, 32, 290, 60
    qi = rng.integers(-2, 3, size=(S, B, H, D)).astype(np.float32)
    ki = rng.integers(-2, 3, size=(S_kv, B, D)).astype(np.float32)
    ki[3] *= outlier
    wi = rng.choice([1, -1, 0.5, -0.5], size=(S, B, H)).astype(np.float32)
    q = torch.from_numpy(qi).to(torch.bfloat16)
    k = torch.from_numpy(ki).to(torch.bfloat16)
    w = torch.from_numpy(wi)
    pos = None if S == 300 else torch.tensor([200, 255], dtype=torch.int32)
    sc, idx, st = gpu_run(dsa, q, k, w, 1, topk, q_pos=pos)
    assert st == 0
    ref = oracle.indexer_fwd(q, k, w, 1, topk, q_pos=pos)
    np.testing.assert_array_equal(idx.reshape(-1, topk), ref["idx"])
    np.testing.assert_array_equal(sc.reshape(-1, topk), ref["scores"])
