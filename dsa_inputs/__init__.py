"""Seeded synthetic inputs for the DSA lightning-indexer forward.

This module only draws random tensors of the right shapes, dtypes and value
distributions.  It contains none of the indexer's arithmetic (no scoring, no
masking, no selection), so both the CPU oracle's tests and the CUDA path's
tests and benchmark can use it without sharing any of the computation.

Layouts follow the DeepSeek-V4 SBHD indexer interface ("tilelang_indexer"
page, `v4_lighting_indexer` parameters):
  q  [S, B, H, D]   bf16
  k  [S_kv, B, D]   bf16   (keys already compressed by `compress_ratio`)
  w  [S, B, H]      fp32
  topk_indices [B, S, topk] int32  (optional, batch-major)

Values: q and k are standard normal draws rounded to bf16 (round to nearest
even, as `torch.Tensor.to(torch.bfloat16)` does); w is a standard normal draw
times `w_scale`.  Draw order on one seeded CPU generator: q, k, w, then the
query positions (decode) -- so every consumer sees identical bits.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic indexer workload (shapes, scales and seed)."""

    name: str
    B: int
    S: int
    S_kv: int
    H: int
    D: int
    compress_ratio: int
    topk: int
    w_scale: float
    seed: int
    # decode: one query per sequence at a position drawn uniformly from this
    # inclusive range; None means prefill (query s sits at position s).
    pos_range: Optional[tuple] = None
    # seed for the caller-supplied top-k indices of the given-indices path
    idx_seed: Optional[int] = None


WORKLOADS = {
    "tiny": Workload("tiny", B=1, S=128, S_kv=128, H=4, D=32, compress_ratio=1,
                     topk=16, w_scale=0.5, seed=0, idx_seed=10),
    "v32_prefill": Workload("v32_prefill", B=1, S=4096, S_kv=4096, H=64, D=128,
                            compress_ratio=1, topk=2048, w_scale=0.125, seed=1,
                            idx_seed=11),
    "decode": Workload("decode", B=64, S=1, S_kv=8192, H=64, D=128,
                       compress_ratio=4, topk=512, w_scale=0.125, seed=2,
                       pos_range=(2048, 32768), idx_seed=12),
    "c4_prefill": Workload("c4_prefill", B=2, S=16384, S_kv=4096, H=64, D=128,
                           compress_ratio=4, topk=512, w_scale=0.125, seed=3,
                           idx_seed=13),
    "long_c4": Workload("long_c4", B=1, S=65536, S_kv=16384, H=64, D=128,
                        compress_ratio=4, topk=2048, w_scale=0.125, seed=4,
                        idx_seed=5),
    # the last 12288 query rows of the long-context prefill (positions
    # 53248..65535, 13312..16384 visible keys each): a profiling slice of
    # the same kernels at a fifth of the size (q is 192 MiB, past L2)
    "long_c4_tail": Workload("long_c4_tail", B=1, S=12288, S_kv=16384, H=64,
                             D=128, compress_ratio=4, topk=2048,
                             w_scale=0.125, seed=7,
                             pos_range=(53248, 53248), idx_seed=8),
}


@dataclasses.dataclass(frozen=True)
class VarlenWorkload:
    """Packed variable-length sequences: query rows per sequence (lens_q)
    and compressed keys per sequence (lens_q // compress_ratio)."""

    name: str
    lens_q: tuple
    H: int
    D: int
    compress_ratio: int
    topk: int
    w_scale: float
    seed: int


VARLEN_WORKLOADS = {
    # a packed C4 batch: one long document and a tail of shorter ones
    "varlen_c4": VarlenWorkload("varlen_c4",
                                lens_q=(16384, 8192, 4096, 2048, 1024, 512,
                                        256, 128),
                                H=64, D=128, compress_ratio=4, topk=512,
                                w_scale=0.125, seed=6),
}


def make_varlen_inputs(vw: VarlenWorkload, device: str = "cpu"):
    """Draw packed (q [T,H,D] bf16, k [T_kv,D] bf16, w [T,H] fp32) and the
    host offsets (cu_seqlens_q, cu_seqlens_k) for a varlen workload, from
    one seeded CPU generator in the order q, k, w."""
    lens_k = [n // vw.compress_ratio for n in vw.lens_q]
    T, T_kv = sum(vw.lens_q), sum(lens_k)
    g = torch.Generator(device="cpu")
    g.manual_seed(vw.seed)
    q = torch.randn((T, vw.H, vw.D), generator=g,
                    dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((T_kv, vw.D), generator=g,
                    dtype=torch.float32).to(torch.bfloat16)
    w = torch.randn((T, vw.H), generator=g, dtype=torch.float32) * vw.w_scale
    cq = np.concatenate([[0], np.cumsum(vw.lens_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    if device != "cpu":
        q, k, w = q.to(device), k.to(device), w.to(device)
    return q, k, w, cq, ck


def describe(wl: Workload) -> str:
    pos = (f", q_pos~U{{{wl.pos_range[0]}..{wl.pos_range[1]}}}"
           if wl.pos_range else "")
    return (f"{wl.name}: B={wl.B} S={wl.S} S_kv={wl.S_kv} H={wl.H} D={wl.D} "
            f"ratio={wl.compress_ratio} topk={wl.topk} "
            f"w~N(0,1)*{wl.w_scale:g}{pos} seed={wl.seed}")


def make_inputs(wl: Workload, device: str = "cpu"):
    """Draw (q, k, w, q_pos) for a workload.

    Returns torch tensors on `device`: q bf16 [S,B,H,D], k bf16 [S_kv,B,D],
    w fp32 [S,B,H], q_pos int32 [B] or None (prefill).  Generation always
    happens on the CPU generator so the bits do not depend on the device.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(wl.seed)
    q = torch.randn((wl.S, wl.B, wl.H, wl.D), generator=g,
                    dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((wl.S_kv, wl.B, wl.D), generator=g,
                    dtype=torch.float32).to(torch.bfloat16)
    w = torch.randn((wl.S, wl.B, wl.H), generator=g,
                    dtype=torch.float32) * wl.w_scale
    q_pos = None
    if wl.pos_range is not None:
        lo, hi = wl.pos_range
        q_pos = torch.randint(lo, hi + 1, (wl.B,), generator=g,
                              dtype=torch.int64).to(torch.int32)
    if device != "cpu":
        q, k, w = q.to(device), k.to(device), w.to(device)
        q_pos = q_pos.to(device) if q_pos is not None else None
    return q, k, w, q_pos


def make_given_indices(B: int, S: int, topk: int, row_limits: np.ndarray,
                       seed: int) -> torch.Tensor:
    """Draw caller-supplied indices [B, S, topk] int32.

    Row (b, s) gets min(topk, row_limits[b, s]) distinct values drawn
    uniformly from [0, row_limits[b, s]) (a random-permutation prefix), the
    rest of the row is -1.  `row_limits` is supplied by the caller (for
    valid indices: the number of keys the row may address); this module
    does not decide which keys are visible.
    """
    rng = np.random.Generator(np.random.Philox(seed))
    lim = np.asarray(row_limits, dtype=np.int64).reshape(B, S)
    out = np.full((B, S, topk), -1, dtype=np.int32)
    for b in range(B):
        for s in range(S):
            n = int(lim[b, s])
            m = min(topk, n)
            if m <= 0:
                continue
            perm = rng.choice(n, size=m, replace=False, shuffle=True)
            out[b, s, :m] = perm
    return torch.from_numpy(out)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU bf16 tensor as a uint16 numpy array."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
