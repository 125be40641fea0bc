"""The Python binding's own checks (no GPU needed): every device entry point
refuses host tensors before the C library sees their pointers, and the
host-buffer call refuses device tensors."""
from __future__ import annotations

import pytest
import torch


@pytest.fixture(scope="module")
def dsa():
    import dsa_sparse_attention_fwd_gb300 as m
    m.build()
    m.load_library()
    return m


def _indexer_inputs(S=8, B=1, H=4, D=32, S_kv=16):
    q = torch.zeros((S, B, H, D), dtype=torch.bfloat16)
    k = torch.zeros((S_kv, B, D), dtype=torch.bfloat16)
    w = torch.zeros((S, B, H), dtype=torch.float32)
    return q, k, w


def test_forward_entry_points_refuse_host_tensors(dsa):
    q, k, w = _indexer_inputs()
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_indexer_fwd(q, k, w, 1, 4)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_indexer_logits(q, k, w, 1)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.indexer_logits(q, k, w, 1)
    idx = torch.zeros((1, 8, 4), dtype=torch.int32)
    gs = torch.zeros((1, 8, 4), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_indexer_bwd(q, k, w, 1, idx, gs)
    cu = [0, 8]
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_indexer_fwd_varlen(q[:, 0], k[:, 0], w[:, 0], cu, [0, 16], 1,
                                   4)


def test_other_entry_points_refuse_host_tensors(dsa):
    T, B, D, kpool = 8, 1, 32, 4
    k = torch.zeros((T, B, D), dtype=torch.bfloat16)
    gate = torch.zeros((T, B, D), dtype=torch.float32)
    ape = torch.zeros((kpool, D), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_kpool_compress(k, gate, ape, kpool)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_expand_selection(torch.zeros((2, 3), dtype=torch.int32),
                                 kpool)
    q = torch.zeros((4, B, 64, D), dtype=torch.bfloat16)
    w = torch.zeros((4, B, 64), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_indexer_fwd_pooled(q, k, gate, ape, w, kpool, 0, 8)
    c = torch.zeros((T, B, 128), dtype=torch.bfloat16)
    qm = torch.zeros((4, B, 64, 128), dtype=torch.bfloat16)
    idx = torch.zeros((B, 4, 8), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_sparse_mla_fwd(qm, c, idx, 0.1)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_indexer_check(ws)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_selftest_wait_limit(10, ws)


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a device "
                    "tensor to pass")
def test_host_call_refuses_device_tensors(dsa):
    q, k, w = _indexer_inputs()
    with pytest.raises(ValueError):
        dsa.dsa_indexer_fwd_host(q.cuda(), k, w, 1, 4)


def test_host_call_refuses_a_host_device_buffer(dsa):
    q, k, w = _indexer_inputs()
    with pytest.raises(ValueError, match="CUDA tensor"):
        dsa.dsa_indexer_fwd_host(q, k, w, 1, 4,
                                 device_buf=torch.zeros(16, dtype=torch.uint8))
