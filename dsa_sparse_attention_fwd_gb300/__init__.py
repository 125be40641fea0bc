"""GB300 (sm_103a) DSA lightning-indexer forward.

A thin ctypes binding over the C ABI in `include/dsa_indexer.h`.  This module
only marshals arguments: it allocates outputs and workspace with PyTorch,
passes raw device pointers and the current CUDA stream, and raises on error
codes.  Every step of the computation runs in the library's CUDA kernels; if
the library is missing, every call raises instead of falling back.

Interface after the DeepSeek-V4 SBHD indexer of NeMo AutoModel
("tilelang_indexer" page: `v4_lighting_indexer(index_q, index_k, weights,
compress_ratio, topk, topk_indices=None)`):
    index_q  [S, B, H, D] bf16, index_k [S_kv, B, D] bf16,
    weights  [S, B, H] fp32, topk_indices [B, S, topk] int32 (optional)
returns (scores [B, S, topk] fp32, indices [B, S, topk] int32).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB_PATH, build

__all__ = [
    "DsaError", "load_library", "build", "dsa_indexer_workspace_size",
    "dsa_set_prefill_policy", "dsa_indexer_fwd_launches", "PREFILL_AUTO",
    "PREFILL_ONE_KERNEL", "PREFILL_TWO_KERNELS",
    "dsa_indexer_fwd", "dsa_indexer_logits", "dsa_indexer_check",
    "dsa_status_string", "dsa_selftest_wait_limit", "v4_lighting_indexer",
    "indexer_logits", "dsa_indexer_host_buffer_size", "dsa_indexer_fwd_host",
    "dsa_indexer_varlen_workspace_size", "dsa_indexer_fwd_varlen",
    "dsa_indexer_bwd", "dsa_indexer_bwd_workspace_size",
    "dsa_kpool_compress", "dsa_expand_selection",
    "dsa_indexer_pooled_workspace_size", "dsa_indexer_fwd_pooled",
    "dsa_sparse_mla_fwd", "dsa_sparse_mla_workspace_size", "STATUS",
]

STATUS = {
    0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED",
    3: "DSA_ERR_WORKSPACE", 4: "DSA_ERR_CUDA", 5: "DSA_ERR_DEVICE_TIMEOUT",
    6: "DSA_ERR_INDEX_RANGE",
}

_lib = None
_lock = threading.Lock()


class DsaError(RuntimeError):
    """A non-zero dsa_status from the library."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} "
                         f"({dsa_status_string(code)})")


def load_library(path: str | None = None):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library not built ({p}); run "
                "dsa_sparse_attention_fwd_gb300.build() first")
        lib = ctypes.CDLL(p)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.dsa_indexer_workspace_size.restype = Z
        lib.dsa_indexer_workspace_size.argtypes = [I] * 8
        lib.dsa_set_prefill_policy.restype = I
        lib.dsa_set_prefill_policy.argtypes = [I]
        lib.dsa_indexer_fwd_launches.restype = I
        lib.dsa_indexer_fwd_launches.argtypes = [I] * 8
        lib.dsa_indexer_fwd.restype = I
        lib.dsa_indexer_fwd.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P, P,
                                        P, P, Z, P]
        lib.dsa_indexer_fwd_profiled.restype = I
        lib.dsa_indexer_fwd_profiled.argtypes = [P, P, P, I, I, I, I, I, I, I,
                                                 P, P, P, P, P, Z, P, P, I]
        lib.dsa_indexer_logits_workspace_size.restype = Z
        lib.dsa_indexer_logits_workspace_size.argtypes = []
        lib.dsa_indexer_logits.restype = I
        lib.dsa_indexer_logits.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P,
                                           Z, P]
        lib.dsa_indexer_check.restype = I
        lib.dsa_indexer_check.argtypes = [P, P]
        lib.dsa_status_string.restype = ctypes.c_char_p
        lib.dsa_status_string.argtypes = [I]
        lib.dsa_selftest_wait_limit.restype = I
        lib.dsa_selftest_wait_limit.argtypes = [I, P, Z, P]
        lib.dsa_indexer_host_buffer_size.restype = Z
        lib.dsa_indexer_host_buffer_size.argtypes = [I] * 8
        lib.dsa_indexer_host_plan.restype = I
        lib.dsa_indexer_host_plan.argtypes = [I, I, I, I, I, I, I, P, I, I,
                                              P, P]
        lib.dsa_indexer_varlen_workspace_size.restype = Z
        lib.dsa_indexer_varlen_workspace_size.argtypes = [I, P, P, I, I, I, I,
                                                          I]
        lib.dsa_indexer_fwd_varlen.restype = I
        lib.dsa_indexer_fwd_varlen.argtypes = [P, P, P, I, P, P, I, I, I, I,
                                               P, P, P, P, P, Z, P]
        lib.dsa_indexer_fwd_host.restype = I
        lib.dsa_indexer_fwd_host.argtypes = [P, P, P, I, I, I, I, I, I, I, P,
                                             P, P, P, P, Z, P]
        lib.dsa_indexer_bwd_workspace_size.restype = Z
        lib.dsa_indexer_bwd_workspace_size.argtypes = []
        lib.dsa_indexer_bwd.restype = I
        lib.dsa_indexer_bwd.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P, P,
                                        P, P, P, P, Z, P]
        L = ctypes.c_longlong
        lib.dsa_kpool_compress.restype = I
        lib.dsa_kpool_compress.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P]
        lib.dsa_expand_selection.restype = I
        lib.dsa_expand_selection.argtypes = [P, L, I, I, I, P, P]
        lib.dsa_indexer_pooled_workspace_size.restype = Z
        lib.dsa_indexer_pooled_workspace_size.argtypes = [I] * 8
        lib.dsa_indexer_fwd_pooled.restype = I
        lib.dsa_indexer_fwd_pooled.argtypes = [P, P, P, P, P, P, I, I, I, I,
                                               I, I, I, I, P, P, P, P, P, Z,
                                               P]
        lib.dsa_sparse_mla_workspace_size.restype = Z
        lib.dsa_sparse_mla_workspace_size.argtypes = []
        lib.dsa_sparse_mla_fwd.restype = I
        lib.dsa_sparse_mla_fwd.argtypes = [P, P, P, I, I, I, I, I, I,
                                           ctypes.c_float, P, P, P, Z, P]
        _lib = lib
        return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def dsa_status_string(code: int) -> str:
    return load_library().dsa_status_string(int(code)).decode()


# prefill top-k path policies (dsa_set_prefill_policy)
PREFILL_AUTO, PREFILL_ONE_KERNEL, PREFILL_TWO_KERNELS = 0, 1, 2


def dsa_set_prefill_policy(policy: int) -> None:
    """Process-wide choice between the one-kernel and the two-kernel prefill
    forward (PREFILL_AUTO picks by row length)."""
    rc = load_library().dsa_set_prefill_policy(int(policy))
    if rc != 0:
        raise DsaError(rc, "dsa_set_prefill_policy")


def dsa_indexer_fwd_launches(S, B, H, D, S_kv, compress_ratio, topk,
                             has_in_idx=False) -> int:
    """Kernels one forward of this shape launches under the current policy."""
    return int(load_library().dsa_indexer_fwd_launches(
        S, B, H, D, S_kv, compress_ratio, topk, 1 if has_in_idx else 0))


def dsa_indexer_workspace_size(S, B, H, D, S_kv, compress_ratio, topk,
                               has_in_idx=False) -> int:
    return int(load_library().dsa_indexer_workspace_size(
        S, B, H, D, S_kv, compress_ratio, topk, int(bool(has_in_idx))))


def _require_cuda(where: str, **tensors):
    """Device entry points read every tensor's pointer as device memory:
    each given tensor must be a CUDA tensor, all on one device (host
    tensors go through dsa_indexer_fwd_host / v4_lighting_indexer)."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError(f"{where}: {name} must be a CUDA tensor, got "
                             f"{t.device}")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{where}: {name} is on {t.device}, the other "
                             f"tensors on {dev}")


def _check_inputs(q, k, w, q_pos, in_idx):
    for name, t, dt in (("index_q", q, torch.bfloat16),
                        ("index_k", k, torch.bfloat16),
                        ("weights", w, torch.float32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    S, B, H, D = q.shape
    S_kv = k.shape[0]
    if tuple(k.shape) != (S_kv, B, D):
        raise ValueError(f"index_k shape {tuple(k.shape)} != "
                         f"({S_kv}, {B}, {D})")
    if tuple(w.shape) != (S, B, H):
        raise ValueError(f"weights shape {tuple(w.shape)} != ({S}, {B}, {H})")
    if q_pos is not None and (q_pos.dtype != torch.int32
                              or q_pos.numel() != B):
        raise ValueError("q_pos must be int32 [B]")
    if in_idx is not None and (in_idx.dtype != torch.int32
                               or not in_idx.is_contiguous()):
        raise ValueError("topk_indices must be contiguous int32")
    return S, B, H, D, S_kv


def dsa_indexer_fwd(q, k, w, compress_ratio, topk, q_pos=None, in_idx=None,
                    out_idx=None, out_scores=None, workspace=None,
                    stream=None, stage_events=None):
    """Enqueue the forward on device tensors; returns (out_scores, out_idx,
    workspace).  Raises DsaError on a synchronous error.  `stage_events`
    (torch.cuda.Event created with enable_timing, at most 1024) are recorded
    before the first kernel and after each kernel launch, in launch order
    (dsa_indexer_fwd_launches gives the count); events left over after the
    last launch are recorded at the end."""
    lib = load_library()
    _require_cuda("dsa_indexer_fwd", q=q, k=k, w=w, q_pos=q_pos,
                  in_idx=in_idx, out_idx=out_idx, out_scores=out_scores,
                  workspace=workspace)
    S, B, H, D, S_kv = _check_inputs(q, k, w, q_pos, in_idx)
    dev = q.device
    if in_idx is not None and tuple(in_idx.shape) != (B, S, topk):
        raise ValueError("topk_indices must be [B, S, topk]")
    if out_idx is None:
        out_idx = torch.empty((B, S, topk), dtype=torch.int32, device=dev)
    if out_scores is None:
        out_scores = torch.empty((B, S, topk), dtype=torch.float32,
                                 device=dev)
    ws = dsa_indexer_workspace_size(S, B, H, D, S_kv, compress_ratio, topk,
                                    in_idx is not None)
    if workspace is None:
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
    if stage_events:
        evs = (ctypes.c_void_p * len(stage_events))(
            *[ctypes.c_void_p(e.cuda_event) for e in stage_events])
        rc = lib.dsa_indexer_fwd_profiled(
            _ptr(q), _ptr(k), _ptr(w), S, B, H, D, S_kv, int(compress_ratio),
            int(topk), _ptr(q_pos), _ptr(in_idx), _ptr(out_idx),
            _ptr(out_scores), _ptr(workspace), workspace.numel(),
            _stream(stream), evs, len(stage_events))
    else:
        rc = lib.dsa_indexer_fwd(
            _ptr(q), _ptr(k), _ptr(w), S, B, H, D, S_kv, int(compress_ratio),
            int(topk), _ptr(q_pos), _ptr(in_idx), _ptr(out_idx),
            _ptr(out_scores), _ptr(workspace), workspace.numel(),
            _stream(stream))
    if rc != 0:
        raise DsaError(rc, "dsa_indexer_fwd")
    return out_scores, out_idx, workspace


def dsa_indexer_bwd_workspace_size() -> int:
    return int(load_library().dsa_indexer_bwd_workspace_size())


def dsa_indexer_bwd(q, k, w, compress_ratio, idx, grad_scores, q_pos=None,
                    grad_q=None, grad_k=None, grad_w=None, workspace=None,
                    stream=None):
    """Enqueue the backward of the given-slots scores on device tensors:
    idx [B, S, topk] int32 and grad_scores [B, S, topk] fp32 give grad_q
    [S, B, H, D], grad_k [S_kv, B, D] and grad_w [S, B, H] (fp32).  Returns
    (grad_q, grad_k, grad_w, workspace)."""
    lib = load_library()
    _require_cuda("dsa_indexer_bwd", q=q, k=k, w=w, idx=idx,
                  grad_scores=grad_scores, q_pos=q_pos, grad_q=grad_q,
                  grad_k=grad_k, grad_w=grad_w, workspace=workspace)
    S, B, H, D, S_kv = _check_inputs(q, k, w, q_pos, idx)
    topk = idx.shape[-1]
    if tuple(idx.shape) != (B, S, topk):
        raise ValueError("idx must be [B, S, topk]")
    if (grad_scores.dtype != torch.float32 or not grad_scores.is_contiguous()
            or tuple(grad_scores.shape) != (B, S, topk)):
        raise ValueError("grad_scores must be contiguous fp32 [B, S, topk]")
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    if grad_q is None:
        grad_q = torch.empty((S, B, H, D), **f32)
    if grad_k is None:
        grad_k = torch.empty((S_kv, B, D), **f32)
    if grad_w is None:
        grad_w = torch.empty((S, B, H), **f32)
    if workspace is None:
        workspace = torch.empty(dsa_indexer_bwd_workspace_size(),
                                dtype=torch.uint8, device=dev)
    rc = lib.dsa_indexer_bwd(
        _ptr(q), _ptr(k), _ptr(w), S, B, H, D, S_kv, int(compress_ratio),
        int(topk), _ptr(q_pos), _ptr(idx), _ptr(grad_scores), _ptr(grad_q),
        _ptr(grad_k), _ptr(grad_w), _ptr(workspace), workspace.numel(),
        _stream(stream))
    if rc != 0:
        raise DsaError(rc, "dsa_indexer_bwd")
    return grad_q, grad_k, grad_w, workspace


def _pool_inputs(k, gate, ape, valid, kpool):
    if k.dtype != torch.bfloat16 or k.dim() != 3 or not k.is_contiguous():
        raise ValueError("k must be contiguous bf16 [T, B, D]")
    T, B, D = k.shape
    if (gate.dtype != torch.float32 or tuple(gate.shape) != (T, B, D)
            or not gate.is_contiguous()):
        raise ValueError("gate must be contiguous fp32 [T, B, D]")
    if (ape.dtype != torch.float32 or tuple(ape.shape) != (kpool, D)
            or not ape.is_contiguous()):
        raise ValueError("ape must be contiguous fp32 [kpool, D]")
    if valid is not None and (valid.dtype != torch.uint8
                              or tuple(valid.shape) != (T, B)
                              or not valid.is_contiguous()):
        raise ValueError("valid must be contiguous uint8 [T, B]")
    return T, B, D


def dsa_kpool_compress(k, gate, ape, kpool, first_key=0, valid=None,
                       stream=None):
    """Pool compression on device tensors: returns (keys [P, B, D] bf16,
    pool_valid [P, B] uint8)."""
    lib = load_library()
    _require_cuda("dsa_kpool_compress", k=k, gate=gate, ape=ape,
                  valid=valid)
    T, B, D = _pool_inputs(k, gate, ape, valid, kpool)
    P = max(0, (T - first_key) // kpool)
    keys = torch.empty((max(P, 1), B, D), dtype=torch.bfloat16,
                       device=k.device)
    pv = torch.empty((max(P, 1), B), dtype=torch.uint8, device=k.device)
    rc = lib.dsa_kpool_compress(_ptr(k), _ptr(gate), _ptr(ape), _ptr(valid),
                                T, B, D, int(kpool), int(first_key),
                                _ptr(keys), _ptr(pv), _stream(stream))
    if rc != 0:
        raise DsaError(rc, "dsa_kpool_compress")
    return keys[:P], pv[:P]


def dsa_expand_selection(pools, kpool, first_key=0, out=None, stream=None):
    """Pool ids [..., select_k] int32 -> token ids [..., select_k*kpool]."""
    lib = load_library()
    _require_cuda("dsa_expand_selection", pools=pools, out=out)
    if pools.dtype != torch.int32 or not pools.is_contiguous():
        raise ValueError("pools must be contiguous int32")
    select_k = pools.shape[-1]
    if out is None:
        out = torch.empty(tuple(pools.shape[:-1]) + (select_k * kpool,),
                          dtype=torch.int32, device=pools.device)
    rows = pools.numel() // select_k
    rc = lib.dsa_expand_selection(_ptr(pools), rows, select_k, int(kpool),
                                  int(first_key), _ptr(out), _stream(stream))
    if rc != 0:
        raise DsaError(rc, "dsa_expand_selection")
    return out


def dsa_indexer_pooled_workspace_size(S, B, H, D, T, kpool, first_key,
                                      index_topk) -> int:
    return int(load_library().dsa_indexer_pooled_workspace_size(
        S, B, H, D, T, kpool, first_key, index_topk))


def dsa_indexer_fwd_pooled(q, k, gate, ape, w, kpool, first_key, index_topk,
                           valid=None, q_pos=None, out_tokens=None,
                           out_pools=None, out_scores=None, workspace=None,
                           stream=None):
    """The pool variant on device tensors: q [S,B,H,D] bf16, per-token k
    [T,B,D] bf16, gate [T,B,D] fp32, ape [kpool,D] fp32, w [S,B,H] fp32,
    valid [T,B] uint8 or None.  Returns (tokens [B,S,index_topk] int32,
    pools [B,S,index_topk/kpool] int32, scores [B,S,index_topk/kpool] fp32,
    workspace)."""
    lib = load_library()
    _require_cuda("dsa_indexer_fwd_pooled", q=q, k=k, gate=gate, ape=ape,
                  w=w, valid=valid, q_pos=q_pos, out_tokens=out_tokens,
                  out_pools=out_pools, out_scores=out_scores,
                  workspace=workspace)
    T, B, D = _pool_inputs(k, gate, ape, valid, kpool)
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise ValueError("q must be contiguous bf16")
    S, Bq, H, Dq = q.shape
    if (Bq, Dq) != (B, D) or tuple(w.shape) != (S, B, H):
        raise ValueError("q / w shapes do not match k")
    if index_topk % kpool:
        raise ValueError("index_topk must be a multiple of kpool")
    sk = index_topk // kpool
    dev = q.device
    if out_tokens is None:
        out_tokens = torch.empty((B, S, index_topk), dtype=torch.int32,
                                 device=dev)
    if out_pools is None:
        out_pools = torch.empty((B, S, sk), dtype=torch.int32, device=dev)
    if out_scores is None:
        out_scores = torch.empty((B, S, sk), dtype=torch.float32, device=dev)
    if workspace is None:
        n = dsa_indexer_pooled_workspace_size(S, B, H, D, T, kpool,
                                              first_key, index_topk)
        if n == 0:
            raise DsaError(2, "dsa_indexer_pooled_workspace_size")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    rc = lib.dsa_indexer_fwd_pooled(
        _ptr(q), _ptr(k), _ptr(gate), _ptr(ape), _ptr(valid), _ptr(w), S, B,
        H, D, T, int(kpool), int(first_key), int(index_topk), _ptr(q_pos),
        _ptr(out_tokens), _ptr(out_pools), _ptr(out_scores), _ptr(workspace),
        workspace.numel(), _stream(stream))
    if rc != 0:
        raise DsaError(rc, "dsa_indexer_fwd_pooled")
    return out_tokens, out_pools, out_scores, workspace


def dsa_sparse_mla_workspace_size() -> int:
    return int(load_library().dsa_sparse_mla_workspace_size())


def dsa_sparse_mla_fwd(q, c, idx, scale, out_o=None, out_lse=None,
                       workspace=None, stream=None):
    """Sparse MLA forward on device tensors: q [S,B,H,Dc] bf16, latent
    cache c [T,B,Dc] bf16, idx [B,S,topk] int32 token ids.  Returns (o
    [S,B,H,Dc] fp32, lse [S,B,H] fp32, workspace)."""
    lib = load_library()
    _require_cuda("dsa_sparse_mla_fwd", q=q, c=c, idx=idx, out_o=out_o,
                  out_lse=out_lse, workspace=workspace)
    for name, t, dt in (("q", q, torch.bfloat16), ("c", c, torch.bfloat16),
                        ("idx", idx, torch.int32)):
        if t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous {dt}")
    S, B, H, Dc = q.shape
    T = c.shape[0]
    if tuple(c.shape) != (T, B, Dc) or idx.shape[:2] != (B, S):
        raise ValueError("c must be [T, B, Dc] and idx [B, S, topk]")
    topk = idx.shape[-1]
    dev = q.device
    if out_o is None:
        out_o = torch.empty((S, B, H, Dc), dtype=torch.float32, device=dev)
    if out_lse is None:
        out_lse = torch.empty((S, B, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(dsa_sparse_mla_workspace_size(),
                                dtype=torch.uint8, device=dev)
    rc = lib.dsa_sparse_mla_fwd(_ptr(q), _ptr(c), _ptr(idx), S, B, H, Dc, T,
                                topk, float(scale), _ptr(out_o),
                                _ptr(out_lse), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    if rc != 0:
        raise DsaError(rc, "dsa_sparse_mla_fwd")
    return out_o, out_lse, workspace


def dsa_indexer_logits(q, k, w, compress_ratio, q_pos=None, logits=None,
                       workspace=None, stream=None):
    """Enqueue the scoring step alone: logits [B, S, S_kv] fp32 (-inf where
    a key is not visible).  Returns (logits, workspace)."""
    lib = load_library()
    _require_cuda("dsa_indexer_logits", q=q, k=k, w=w, q_pos=q_pos,
                  logits=logits, workspace=workspace)
    S, B, H, D, S_kv = _check_inputs(q, k, w, q_pos, None)
    dev = q.device
    if logits is None:
        logits = torch.empty((B, S, S_kv), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(int(lib.dsa_indexer_logits_workspace_size()),
                                dtype=torch.uint8, device=dev)
    rc = lib.dsa_indexer_logits(
        _ptr(q), _ptr(k), _ptr(w), S, B, H, D, S_kv, int(compress_ratio),
        _ptr(q_pos), _ptr(logits), _ptr(workspace), workspace.numel(),
        _stream(stream))
    if rc != 0:
        raise DsaError(rc, "dsa_indexer_logits")
    return logits, workspace


def dsa_indexer_check(workspace, stream=None) -> int:
    """Synchronise the stream and return the device status code (0 = ok)."""
    _require_cuda("dsa_indexer_check", workspace=workspace)
    return int(load_library().dsa_indexer_check(_ptr(workspace),
                                                 _stream(stream)))


def dsa_selftest_wait_limit(limit_us: int, workspace, stream=None) -> int:
    _require_cuda("dsa_selftest_wait_limit", workspace=workspace)
    return int(load_library().dsa_selftest_wait_limit(
        int(limit_us), _ptr(workspace), workspace.numel(), _stream(stream)))


def _host_i32(a):
    """A contiguous host int32 tensor (kept alive by the caller)."""
    t = torch.as_tensor(a, dtype=torch.int32, device="cpu").contiguous()
    return t


def dsa_indexer_varlen_workspace_size(cu_seqlens_q, cu_seqlens_k, H, D,
                                      compress_ratio, topk,
                                      has_in_idx=False) -> int:
    cq, ck = _host_i32(cu_seqlens_q), _host_i32(cu_seqlens_k)
    if cq.numel() != ck.numel() or cq.numel() < 2:
        raise ValueError("cu_seqlens_q / cu_seqlens_k must both be [N + 1]")
    return int(load_library().dsa_indexer_varlen_workspace_size(
        cq.numel() - 1, _ptr(cq), _ptr(ck), H, D, compress_ratio, topk,
        int(bool(has_in_idx))))


def dsa_indexer_fwd_varlen(q, k, w, cu_seqlens_q, cu_seqlens_k,
                           compress_ratio, topk, q_pos=None, in_idx=None,
                           out_idx=None, out_scores=None, workspace=None,
                           stream=None):
    """The forward over packed variable-length sequences: q [T, H, D] bf16,
    k [T_kv, D] bf16, w [T, H] fp32 and the optional q_pos [N] / in_idx
    [T, topk] on the device; cu_seqlens_q / cu_seqlens_k are host int32
    offsets [N + 1].  Returns (out_scores [T, topk], out_idx [T, topk],
    workspace); indices are local to each row's sequence."""
    lib = load_library()
    _require_cuda("dsa_indexer_fwd_varlen", q=q, k=k, w=w, q_pos=q_pos,
                  in_idx=in_idx, out_idx=out_idx, out_scores=out_scores,
                  workspace=workspace)
    cq, ck = _host_i32(cu_seqlens_q), _host_i32(cu_seqlens_k)
    N = cq.numel() - 1
    if ck.numel() != N + 1 or N < 1:
        raise ValueError("cu_seqlens_q / cu_seqlens_k must both be [N + 1]")
    if q.dim() != 3 or k.dim() != 2 or w.dim() != 2:
        raise ValueError("q [T, H, D], k [T_kv, D], w [T, H] expected")
    T, H, D = q.shape
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("w", w, torch.float32)):
        if t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous {dt}")
    if int(cq[-1]) != T or int(ck[-1]) != k.shape[0] or k.shape[1] != D or \
            tuple(w.shape) != (T, H):
        raise ValueError("shapes do not match the offsets")
    if q_pos is not None and (q_pos.dtype != torch.int32 or
                              q_pos.numel() != N):
        raise ValueError("q_pos must be int32 [N]")
    if in_idx is not None and (in_idx.dtype != torch.int32 or
                               tuple(in_idx.shape) != (T, topk) or
                               not in_idx.is_contiguous()):
        raise ValueError("in_idx must be contiguous int32 [T, topk]")
    dev = q.device
    if out_idx is None:
        out_idx = torch.empty((T, topk), dtype=torch.int32, device=dev)
    if out_scores is None:
        out_scores = torch.empty((T, topk), dtype=torch.float32, device=dev)
    if workspace is None:
        need = dsa_indexer_varlen_workspace_size(cq, ck, H, D,
                                                 compress_ratio, topk,
                                                 in_idx is not None)
        if need == 0:
            raise DsaError(2, "dsa_indexer_varlen_workspace_size")
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    rc = lib.dsa_indexer_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(w), N, _ptr(cq), _ptr(ck), H, D,
        int(compress_ratio), int(topk), _ptr(q_pos), _ptr(in_idx),
        _ptr(out_idx), _ptr(out_scores), _ptr(workspace), workspace.numel(),
        _stream(stream))
    if rc != 0:
        raise DsaError(rc, "dsa_indexer_fwd_varlen")
    return out_scores, out_idx, workspace


def dsa_indexer_host_buffer_size(S, B, H, D, S_kv, compress_ratio, topk,
                                 has_in_idx=False) -> int:
    return int(load_library().dsa_indexer_host_buffer_size(
        S, B, H, D, S_kv, compress_ratio, topk, int(bool(has_in_idx))))


def dsa_indexer_host_plan(S, B, H, D, S_kv, compress_ratio, topk,
                          q_pos=None, has_in_idx=False, sms=0):
    """How dsa_indexer_fwd_host splits and orders the query rows: returns
    (chunk starts, the last one S; processing order).  q_pos: host int32
    [B] or None.  sms: the SM count the chunk starts assume (0: the current
    device's).  Raises DsaError for an invalid shape."""
    lib = load_library()
    starts = (ctypes.c_int * 17)()
    order = (ctypes.c_int * 16)()
    pos = None
    if q_pos is not None:
        pos = _host_i32(q_pos)
    n = lib.dsa_indexer_host_plan(
        S, B, H, D, S_kv, int(compress_ratio), int(topk),
        None if pos is None else pos.data_ptr(), int(bool(has_in_idx)),
        int(sms), starts, order)
    if n <= 0:
        raise DsaError(1, "dsa_indexer_host_plan")
    return list(starts[:n + 1]), list(order[:n])


def dsa_indexer_fwd_host(q, k, w, compress_ratio, topk, q_pos=None,
                         in_idx=None, out_idx=None, out_scores=None,
                         device_buf=None, stream=None):
    """The forward on host (CPU) tensors through the C entry point that
    pipelines the copies against the kernels; returns (out_scores, out_idx,
    status).  Outputs are page-locked when q is.  `device_buf` (uint8 on the
    current CUDA device) is allocated when not given.  The call returns with
    the results in the host outputs; `status` is the library's return code
    (0, or the device status of the run)."""
    lib = load_library()
    S, B, H, D, S_kv = _check_inputs(q, k, w, q_pos, in_idx)
    for name, t in (("index_q", q), ("index_k", k), ("weights", w),
                    ("q_pos", q_pos), ("topk_indices", in_idx),
                    ("out_idx", out_idx), ("out_scores", out_scores)):
        if t is not None and t.device.type != "cpu":
            raise ValueError(f"{name} must be a host tensor")
    _require_cuda("dsa_indexer_fwd_host", device_buf=device_buf)
    if in_idx is not None and tuple(in_idx.shape) != (B, S, topk):
        raise ValueError("topk_indices must be [B, S, topk]")
    pinned = q.is_pinned()
    if out_idx is None:
        out_idx = torch.empty((B, S, topk), dtype=torch.int32,
                              pin_memory=pinned)
    if out_scores is None:
        out_scores = torch.empty((B, S, topk), dtype=torch.float32,
                                 pin_memory=pinned)
    need = dsa_indexer_host_buffer_size(S, B, H, D, S_kv, compress_ratio,
                                        topk, in_idx is not None)
    if need == 0:
        raise DsaError(2, "dsa_indexer_host_buffer_size")
    if device_buf is None:
        device_buf = torch.empty(need, dtype=torch.uint8,
                                 device=torch.device(
                                     "cuda", torch.cuda.current_device()))
    rc = lib.dsa_indexer_fwd_host(
        _ptr(q), _ptr(k), _ptr(w), S, B, H, D, S_kv, int(compress_ratio),
        int(topk), _ptr(q_pos), _ptr(in_idx), _ptr(out_idx),
        _ptr(out_scores), _ptr(device_buf), device_buf.numel(),
        _stream(stream))
    if rc not in (0, 5, 6):  # device status codes are returned, not raised
        raise DsaError(rc, "dsa_indexer_fwd_host")
    return out_scores, out_idx, rc


def v4_lighting_indexer(index_q, index_k, weights, compress_ratio, topk,
                        topk_indices=None, q_pos=None, check=True):
    """The indexer forward with the V4 argument order.

    Device tensors run on the current stream.  Host (CPU) tensors are copied
    to the current CUDA device, run there, and the results copied back into
    host tensors (pinned when the inputs are pinned); the whole host round
    trip happens inside this call.  Returns (scores [B,S,topk] fp32,
    indices [B,S,topk] int32).  With check=True the call synchronises and
    raises on a device-side status (bad given index, expired wait).
    """
    if index_q.device.type == "cpu":
        # host buffers: the C entry point copies in, runs and copies out,
        # overlapping the copies with the kernels
        scores, idx, rc = dsa_indexer_fwd_host(
            index_q, index_k, weights, compress_ratio, topk, q_pos=q_pos,
            in_idx=topk_indices)
        if check and rc != 0:
            raise DsaError(rc, "device status")
        return scores, idx
    scores, idx, ws = dsa_indexer_fwd(index_q, index_k, weights,
                                      compress_ratio, topk, q_pos=q_pos,
                                      in_idx=topk_indices)
    if check:
        rc = dsa_indexer_check(ws)
        if rc != 0:
            raise DsaError(rc, "device status")
    return scores, idx


def indexer_logits(index_q, index_k, weights, compress_ratio, q_pos=None):
    """Logits [B, S, S_kv] fp32 on the device (-inf where masked)."""
    logits, _ = dsa_indexer_logits(index_q, index_k, weights, compress_ratio,
                                   q_pos=q_pos)
    return logits
