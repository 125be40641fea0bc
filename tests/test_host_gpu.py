"""The host-buffer forward (dsa_indexer_fwd_host): copies in, runs and
copies out with the copies pipelined against the kernels over chunks of
query rows.  Its results must equal the device-buffer forward bit for bit
(no row's arithmetic depends on the other rows), and it must report the
device status of the run."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from dsa_inputs import WORKLOADS, Workload, make_given_indices, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    return m


def device_run(dsa, q, k, w, ratio, topk, q_pos=None, in_idx=None):
    d = torch.device("cuda")
    sc, idx, ws = dsa.dsa_indexer_fwd(
        q.to(d), k.to(d), w.to(d), ratio, topk,
        q_pos=None if q_pos is None else q_pos.to(d),
        in_idx=None if in_idx is None else in_idx.to(d))
    st = dsa.dsa_indexer_check(ws)
    return sc.cpu().numpy(), idx.cpu().numpy(), st


def host_run(dsa, q, k, w, ratio, topk, q_pos=None, in_idx=None, pin=True):
    if pin:
        q, k, w = q.pin_memory(), k.pin_memory(), w.pin_memory()
        q_pos = None if q_pos is None else q_pos.pin_memory()
        in_idx = None if in_idx is None else in_idx.pin_memory()
    sc, idx, rc = dsa.dsa_indexer_fwd_host(q, k, w, ratio, topk, q_pos=q_pos,
                                           in_idx=in_idx)
    return sc.numpy(), idx.numpy(), rc


def same_bits(a, b):
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("name", ["tiny", "v32_prefill", "decode"])
def test_host_path_equals_device_path(dsa, name):
    wl = WORKLOADS[name]
    q, k, w, pos = make_inputs(wl)
    d_sc, d_idx, d_st = device_run(dsa, q, k, w, wl.compress_ratio, wl.topk,
                                   q_pos=pos)
    h_sc, h_idx, h_rc = host_run(dsa, q, k, w, wl.compress_ratio, wl.topk,
                                 q_pos=pos)
    assert d_st == 0 and h_rc == 0
    np.testing.assert_array_equal(h_idx, d_idx)
    assert same_bits(h_sc, d_sc)


@pytest.mark.parametrize("S,B,H,D,S_kv,ratio,topk,pos", [
    (2100, 2, 64, 128, 600, 4, 300, None),      # 4 chunks, strided copies
    (3000, 3, 32, 64, 3000, 1, 100, [0, 7, 900]),  # 5 chunks with positions
])
def test_host_chunks_with_batches(dsa, S, B, H, D, S_kv, ratio, topk, pos):
    wl = Workload("h", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=S + B)
    q, k, w, _ = make_inputs(wl)
    q_pos = None if pos is None else torch.tensor(pos, dtype=torch.int32)
    d_sc, d_idx, d_st = device_run(dsa, q, k, w, ratio, topk, q_pos=q_pos)
    h_sc, h_idx, h_rc = host_run(dsa, q, k, w, ratio, topk, q_pos=q_pos)
    assert d_st == 0 and h_rc == 0
    np.testing.assert_array_equal(h_idx, d_idx)
    assert same_bits(h_sc, d_sc)
    # pageable host buffers give the same result
    p_sc, p_idx, p_rc = host_run(dsa, q, k, w, ratio, topk, q_pos=q_pos,
                                 pin=False)
    assert p_rc == 0
    np.testing.assert_array_equal(p_idx, d_idx)
    assert same_bits(p_sc, d_sc)


def test_host_given_indices_and_status(dsa):
    S, B, H, D, S_kv, ratio, topk = 2048, 2, 64, 128, 512, 4, 200
    wl = Workload("h", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=0.125, seed=77)
    q, k, w, _ = make_inputs(wl)
    pos = np.arange(S)[None, :].repeat(B, 0)
    nv = np.clip((pos + 1) // ratio, 0, S_kv)
    gi = make_given_indices(B, S, topk, nv, 78)
    d_sc, d_idx, d_st = device_run(dsa, q, k, w, ratio, topk, in_idx=gi)
    h_sc, h_idx, h_rc = host_run(dsa, q, k, w, ratio, topk, in_idx=gi)
    assert d_st == 0 and h_rc == 0
    np.testing.assert_array_equal(h_idx, d_idx)
    assert same_bits(h_sc, d_sc)
    # an out-of-range index in the second chunk is reported by the call
    gi[1, 2000, 5] = S_kv
    h_sc, h_idx, h_rc = host_run(dsa, q, k, w, ratio, topk, in_idx=gi)
    assert h_rc == 6  # DSA_ERR_INDEX_RANGE
    assert np.isneginf(h_sc[1, 2000, 5]) and h_idx[1, 2000, 5] == S_kv


def test_host_compute_bound_chunk_order(dsa):
    """Rows deep into a long sequence give many visible keys per copied
    byte (above 3000 FLOP per byte), so the chunks are processed
    alternately from the costly and the cheap end (4 chunks); every row's
    result must still equal the device-buffer forward bit for bit."""
    S, B, H, D, S_kv, ratio, topk = 2048, 1, 64, 128, 8192, 1, 64
    wl = Workload("h", B=B, S=S, S_kv=S_kv, H=H, D=D, compress_ratio=ratio,
                  topk=topk, w_scale=H ** -0.5, seed=4099)
    q, k, w, _ = make_inputs(wl)
    q_pos = torch.tensor([4096], dtype=torch.int32)
    # 2 H D n_vis per row against q, w, indices and scores per row
    nv = np.minimum(S_kv, (4096 + np.arange(S) + 1) // ratio)
    assert (2 * H * D * nv.sum()) / (S * (2 * H * D + 4 * H + 8 * topk)) > 3000
    d_sc, d_idx, d_st = device_run(dsa, q, k, w, ratio, topk, q_pos=q_pos)
    h_sc, h_idx, h_rc = host_run(dsa, q, k, w, ratio, topk, q_pos=q_pos)
    assert d_st == 0 and h_rc == 0
    np.testing.assert_array_equal(h_idx, d_idx)
    assert same_bits(h_sc, d_sc)
