"""The allocation-free forward, dsa_indexer_fwd_static_scratch().

It exists for callers that cannot call cudaMalloc (a caching allocator that
already holds all free memory, a plugin host that only lends out its own
tensors, a path where allocating would synchronise the device): it takes its
scratch from a fixed array inside the library.  These tests call it through
the C ABI and check that it gives what the workspace-based dsa_indexer_fwd()
gives, within the score tolerance of the other GPU tests, on consecutive
calls that reuse the shared array.  The test itself allocates the inputs and
outputs with torch; the entry point under test allocates nothing.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from dsa_inputs import WORKLOADS, make_given_indices, make_inputs
from tests.helpers import score_tol

pytestmark = pytest.mark.gpu

OK, UNSUPPORTED = 0, 2
STATIC_SCRATCH_BYTES = 64 * 1024 * 1024 + 256


@pytest.fixture(scope="module")
def dsa():
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    return m


@pytest.fixture(scope="module")
def lib(dsa):
    L = ctypes.CDLL(dsa.LIB_PATH)
    P, I = ctypes.c_void_p, ctypes.c_int
    f = L.dsa_indexer_fwd_static_scratch
    f.restype = I
    f.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P, P, P, P, P]
    return L


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def alloc_outputs(B, S, topk):
    out_idx = torch.full((B, S, topk), 7, dtype=torch.int32, device="cuda")
    out_sc = torch.full((B, S, topk), 7.0, dtype=torch.float32,
                        device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    return out_idx, out_sc, status


def call_static(lib, q, k, w, ratio, topk, outs, q_pos=None, in_idx=None):
    """One call of the allocation-free entry point into caller-owned
    outputs; returns the synchronous return code."""
    S, B, H, D = q.shape
    S_kv = k.shape[0]
    out_idx, out_sc, status = outs
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.dsa_indexer_fwd_static_scratch(
        _p(q), _p(k), _p(w), S, B, H, D, S_kv, ratio, topk, _p(q_pos),
        _p(in_idx), _p(out_idx), _p(out_sc), _p(status), stream)


def run_static(lib, q, k, w, ratio, topk, q_pos=None, in_idx=None):
    """One call of the allocation-free entry point; returns numpy outputs,
    the device status word and the synchronous return code."""
    S, B = q.shape[0], q.shape[1]
    outs = alloc_outputs(B, S, topk)
    rc = call_static(lib, q, k, w, ratio, topk, outs, q_pos=q_pos,
                     in_idx=in_idx)
    torch.cuda.synchronize()
    out_idx, out_sc, status = outs
    return out_sc.cpu().numpy(), out_idx.cpu().numpy(), int(status.item()), rc


def run_existing(dsa, q, k, w, ratio, topk, q_pos=None, in_idx=None):
    sc, idx, ws = dsa.dsa_indexer_fwd(q, k, w, ratio, topk, q_pos=q_pos,
                                      in_idx=in_idx)
    st = dsa.dsa_indexer_check(ws)
    return sc.cpu().numpy(), idx.cpu().numpy(), st


def assert_same(a_sc, a_idx, b_sc, b_idx):
    np.testing.assert_array_equal(a_idx, b_idx)
    assert np.array_equal(np.isneginf(a_sc), np.isneginf(b_sc))
    fin = np.isfinite(b_sc)
    assert np.all(np.isfinite(a_sc[fin]))
    err = np.abs(a_sc[fin].astype(np.float64) - b_sc[fin])
    assert np.all(err <= score_tol(b_sc[fin].astype(np.float64)))


def device_inputs(name):
    wl = WORKLOADS[name]
    q, k, w, pos = make_inputs(wl, device="cuda")
    return wl, q, k, w, pos


def test_matches_workspace_forward_on_consecutive_calls(dsa, lib):
    # three calls in a row share the library's one scratch array: a small
    # problem, the 4096 x 4096 prefill (one kernel, its per-CTA scratch in
    # the array), then a decode batch (logits in the array)
    for name in ("tiny", "v32_prefill", "decode"):
        wl, q, k, w, pos = device_inputs(name)
        sc, idx, st, rc = run_static(lib, q, k, w, wl.compress_ratio,
                                     wl.topk, q_pos=pos)
        assert rc == OK, name
        assert st == 0, name
        ref_sc, ref_idx, ref_st = run_existing(dsa, q, k, w,
                                               wl.compress_ratio, wl.topk,
                                               q_pos=pos)
        assert ref_st == 0
        assert_same(sc, idx, ref_sc, ref_idx)


def test_matches_oracle_on_sampled_rows(dsa, lib):
    """The 4096 x 4096 prefill through the allocation-free entry point,
    compared with the CPU oracle on sampled rows (the oracle computes them
    one by one), by the same rule as the other GPU parity tests."""
    import oracle
    from tests.helpers import compare_topk_row
    wl, q, k, w, pos = device_inputs("v32_prefill")
    sc, idx, st, rc = run_static(lib, q, k, w, wl.compress_ratio, wl.topk)
    assert rc == OK and st == 0
    rows = np.array([0, 1, 700, 2047, 2048, 2049, 3000, 4095],
                    dtype=np.int64)
    ref = oracle.indexer_fwd(q.cpu(), k.cpu(), w.cpu(), wl.compress_ratio,
                             wl.topk, rows=rows, want_logits=True)
    sc, idx = sc.reshape(-1, wl.topk), idx.reshape(-1, wl.topk)
    for n, r in enumerate(rows):
        msg = compare_topk_row(idx[r], sc[r], ref["idx"][n],
                               ref["scores64"][n], ref["next"][n],
                               ref["logits"][n])
        assert msg is None, (int(r), msg)


def test_allocates_no_device_memory(dsa, lib):
    """After a first call (which may load the library's kernels onto the
    device), a call changes the device's free memory by nothing: the entry
    point allocates and frees no device memory.  Inputs and outputs are
    allocated before the measurement."""
    wl, q, k, w, pos = device_inputs("v32_prefill")
    outs = alloc_outputs(wl.B, wl.S, wl.topk)
    assert call_static(lib, q, k, w, 1, wl.topk, outs) == OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert call_static(lib, q, k, w, 1, wl.topk, outs) == OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert int(outs[2].item()) == 0


def test_repeat_call_gives_same_result(dsa, lib):
    wl, q, k, w, pos = device_inputs("tiny")
    first = run_static(lib, q, k, w, 1, wl.topk)
    second = run_static(lib, q, k, w, 1, wl.topk)
    assert first[3] == OK and second[3] == OK
    assert_same(second[0], second[1], first[0], first[1])


def test_given_indices_and_status_word(dsa, lib):
    wl, q, k, w, _ = device_inputs("tiny")
    nv = np.clip(np.arange(wl.S) + 1, 0, wl.S_kv)[None, :]
    gi = make_given_indices(wl.B, wl.S, wl.topk, nv, wl.idx_seed).cuda()
    sc, idx, st, rc = run_static(lib, q, k, w, 1, wl.topk, in_idx=gi)
    assert rc == OK and st == 0
    ref_sc, ref_idx, _ = run_existing(dsa, q, k, w, 1, wl.topk, in_idx=gi)
    assert_same(sc, idx, ref_sc, ref_idx)
    gi[0, 3, 0] = wl.S_kv  # outside [-1, S_kv): flagged in the status word
    sc, idx, st, rc = run_static(lib, q, k, w, 1, wl.topk, in_idx=gi)
    assert rc == OK and st == 1
    assert np.isneginf(sc[0, 3, 0])
    # the next clean call starts from a cleared status word
    gi[0, 3, 0] = 0
    assert run_static(lib, q, k, w, 1, wl.topk, in_idx=gi)[2] == 0


def test_long_rows_run_scores_then_selection(dsa, lib):
    """Rows of 16384 keys need 84 MB of one-kernel score rows, more than the
    fixed array: the entry point runs scores then selection over row chunks
    instead, with the same results as the workspace forward (which takes
    the one-kernel path here) and the oracle on sampled rows."""
    import oracle
    from dsa_inputs import Workload
    from tests.helpers import compare_topk_row
    S, S_kv, ratio, topk = 256, 16384, 4, 2048
    wl = Workload("t", B=1, S=S, S_kv=S_kv, H=64, D=128, compress_ratio=ratio,
                  topk=topk, w_scale=0.125, seed=41)
    q, k, w, _ = make_inputs(wl, device="cuda")
    # row s sits at position 47999 + s and sees 12000 + s // 4 keys
    pos = torch.tensor([12000 * ratio - 1], dtype=torch.int32, device="cuda")
    need = dsa.dsa_indexer_workspace_size(S, 1, 64, 128, S_kv, ratio, topk,
                                          False)
    assert need > STATIC_SCRATCH_BYTES
    sc, idx, st, rc = run_static(lib, q, k, w, ratio, topk, q_pos=pos)
    assert rc == OK and st == 0
    ref_sc, ref_idx, ref_st = run_existing(dsa, q, k, w, ratio, topk,
                                           q_pos=pos)
    assert ref_st == 0
    assert_same(sc, idx, ref_sc, ref_idx)
    rows = np.array([0, 1, 100, 255], dtype=np.int64)
    ref = oracle.indexer_fwd(q.cpu(), k.cpu(), w.cpu(), ratio, topk,
                             q_pos=pos.cpu(), rows=rows, want_logits=True)
    sc, idx = sc.reshape(-1, topk), idx.reshape(-1, topk)
    for n, r in enumerate(rows):
        msg = compare_topk_row(idx[r], sc[r], ref["idx"][n],
                               ref["scores64"][n], ref["next"][n],
                               ref["logits"][n])
        assert msg is None, (int(r), msg)


def test_refuses_problems_beyond_the_fixed_scratch(lib):
    fake = ctypes.c_void_p(1 << 20)  # never touched: refused before any use
    # given indices with 4 heads read the scores back from the full [S, S_kv]
    # fp32 logits: 4096 query rows over 4096 keys fill the 64 MiB exactly,
    # one row more is refused
    rc = lib.dsa_indexer_fwd_static_scratch(
        fake, fake, fake, 4097, 1, 4, 32, 4096, 1, 16, None, fake, fake,
        fake, None, None)
    assert rc == UNSUPPORTED
