"""CPU oracle for the DSA lightning-indexer forward (fp64, plain C).

TEST INFRASTRUCTURE ONLY: import this package only from `tests/`, from the
smoke check and from the benchmark's CPU-baseline leg.  The product path
(`dsa_sparse_attention_fwd_gb300`) never imports it, and it imports nothing
from the product path.

The arithmetic lives in `indexer_oracle.c`; this module only builds that file
with gcc, marshals numpy arrays into it and returns numpy arrays.  See the C
file's header for what is computed and which page passage each rule follows.

Parity pins for every function are in `tests/test_oracle.py`.  The one part
with no pin is the fp32 accumulation order of the GPU side, which only the
tolerance covers ("parity unpinned" for that aspect alone).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "indexer_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE double, no FMA contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            lib.oracle_indexer_fwd.restype = ctypes.c_int
            lib.oracle_indexer_fwd.argtypes = [
                P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                P, P, P, P, ctypes.c_longlong, P, P, P, P, P, P,
                ctypes.c_int]
            lib.oracle_kpool_compress.restype = ctypes.c_longlong
            lib.oracle_kpool_compress.argtypes = [
                P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, P, P]
            lib.oracle_sparse_mla_fwd.restype = ctypes.c_int
            lib.oracle_sparse_mla_fwd.argtypes = [
                P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                P, P, ctypes.c_int]
            lib.oracle_expand_selection.restype = None
            lib.oracle_expand_selection.argtypes = [
                P, ctypes.c_longlong, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, P]
            lib.oracle_indexer_bwd.restype = None
            lib.oracle_indexer_bwd.argtypes = [
                P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                P, P, P, P, P, P, P, P, P]
            lib.oracle_key_visible.restype = ctypes.c_int
            lib.oracle_key_visible.argtypes = [ctypes.c_longlong,
                                               ctypes.c_longlong, ctypes.c_int]
            _lib = lib
    return _lib


def _bits(x) -> np.ndarray:
    """bf16 input as a contiguous uint16 array of bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            assert x.dtype == torch.bfloat16, x.dtype
            return x.view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, x.dtype
    return x


def _arr(x, dtype) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def key_visible(j: int, t: int, ratio: int) -> bool:
    """Causal rule: compressed key j is visible at position t."""
    return bool(_load().oracle_key_visible(j, t, ratio))


def indexer_fwd(q, k, w, compress_ratio: int, topk: int, q_pos=None,
                in_idx=None, rows=None, n_threads: int | None = None,
                want_logits: bool = False, key_valid=None):
    """Run the oracle on a list of rows.

    q [S,B,H,D] bf16, k [S_kv,B,D] bf16, w [S,B,H] fp32, q_pos [B] int32 or
    None, in_idx [B,S,topk] int32 or None, key_valid [S_kv,B] (0 = the key
    is not a candidate) or None.  `rows` lists row ids b*S+s
    (default: every row, in (b, s) order).  Returns a dict of numpy arrays,
    one line per requested row: idx, scores (fp32), scores64, next (the
    (topk+1)-th visible score, -inf if none), nvis, logits (if asked),
    plus `threads` (threads used) and `rows`.
    """
    lib = _load()
    qb, kb = _bits(q), _bits(k)
    wf = _arr(w, np.float32)
    S, B, H, D = qb.shape
    S_kv = kb.shape[0]
    assert kb.shape == (S_kv, B, D), kb.shape
    assert wf.shape == (S, B, H), wf.shape
    qp = None if q_pos is None else _arr(q_pos, np.int32).reshape(B)
    gi = None if in_idx is None else _arr(in_idx, np.int32).reshape(B, S, topk)
    kv = None if key_valid is None else _arr(key_valid, np.uint8).reshape(
        S_kv, B)
    if rows is None:
        rows = np.arange(B * S, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    out = {
        "idx": np.empty((n, topk), np.int32),
        "scores": np.empty((n, topk), np.float32),
        "scores64": np.empty((n, topk), np.float64),
        "next": np.empty((n,), np.float64),
        "nvis": np.empty((n,), np.int32),
    }
    logits = np.empty((n, S_kv), np.float64) if want_logits else None
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    used = lib.oracle_indexer_fwd(
        _ptr(qb), _ptr(kb), _ptr(wf), S, B, H, D, S_kv, int(compress_ratio),
        int(topk), _ptr(qp), _ptr(kv), _ptr(gi), _ptr(rows), n,
        _ptr(out["idx"]), _ptr(out["scores"]), _ptr(out["scores64"]),
        _ptr(out["next"]), _ptr(out["nvis"]), _ptr(logits), int(n_threads))
    if want_logits:
        out["logits"] = logits
    out["threads"] = used
    out["rows"] = rows
    return out


def indexer_bwd(q, k, w, compress_ratio: int, idx, grad_scores, q_pos=None):
    """Backward of the given-slots forward: gradients of sum(grad_scores *
    scores) with respect to q, k and w, in double.

    q [S,B,H,D] bf16, k [S_kv,B,D] bf16, w [S,B,H] fp32, idx [B,S,topk]
    int32 (the slots the forward scored), grad_scores [B,S,topk] fp32,
    q_pos [B] int32 or None.  Returns a dict: grad_q [S,B,H,D],
    grad_k [S_kv,B,D], grad_w [S,B,H] and abs_q / abs_k / abs_w, the sums of
    the absolute values of each output's terms.
    """
    lib = _load()
    qb, kb = _bits(q), _bits(k)
    wf = _arr(w, np.float32)
    S, B, H, D = qb.shape
    S_kv = kb.shape[0]
    gi = _arr(idx, np.int32)
    topk = gi.shape[-1]
    gi = gi.reshape(B, S, topk)
    gs = _arr(grad_scores, np.float32).reshape(B, S, topk)
    qp = None if q_pos is None else _arr(q_pos, np.int32).reshape(B)
    out = {n: np.empty(shape, np.float64) for n, shape in (
        ("grad_q", (S, B, H, D)), ("grad_k", (S_kv, B, D)),
        ("grad_w", (S, B, H)), ("abs_q", (S, B, H, D)),
        ("abs_k", (S_kv, B, D)), ("abs_w", (S, B, H)))}
    lib.oracle_indexer_bwd(
        _ptr(qb), _ptr(kb), _ptr(wf), S, B, H, D, S_kv, int(compress_ratio),
        int(topk), _ptr(qp), _ptr(gi), _ptr(gs), _ptr(out["grad_q"]),
        _ptr(out["grad_k"]), _ptr(out["grad_w"]), _ptr(out["abs_q"]),
        _ptr(out["abs_k"]), _ptr(out["abs_w"]))
    return out


def kpool_compress(k, gate, ape, valid, kpool: int, first_key: int = 0):
    """Pool compression (see oracle_kpool_compress in the C file).

    k [T,B,D] bf16, gate [T,B,D] fp32, ape [kpool,D] fp32, valid [T,B]
    (nonzero = valid) or None.  Returns {"keys": [P,B,D] float64,
    "valid": [P,B] uint8, "P": P}.
    """
    lib = _load()
    kb = _bits(k)
    T, B, D = kb.shape
    gf = _arr(gate, np.float32).reshape(T, B, D)
    af = _arr(ape, np.float32).reshape(kpool, D)
    vv = None if valid is None else _arr(valid, np.uint8).reshape(T, B)
    P = max(0, (T - first_key) // kpool)
    keys = np.zeros((max(P, 1), B, D), np.float64)
    pv = np.zeros((max(P, 1), B), np.uint8)
    got = lib.oracle_kpool_compress(_ptr(kb), _ptr(gf), _ptr(af), _ptr(vv),
                                    T, B, D, int(kpool), int(first_key),
                                    _ptr(keys), _ptr(pv))
    assert got == P
    return {"keys": keys[:P], "valid": pv[:P], "P": P}


def expand_selection(pools, kpool: int, first_key: int = 0):
    """Pool ids [..., select_k] -> token ids [..., select_k * kpool] (see
    oracle_expand_selection in the C file)."""
    lib = _load()
    pl = _arr(pools, np.int32)
    select_k = pl.shape[-1]
    rows = pl.size // select_k if select_k else 0
    out = np.empty(pl.shape[:-1] + (select_k * kpool,), np.int32)
    lib.oracle_expand_selection(_ptr(pl), rows, select_k, int(kpool),
                                int(first_key), _ptr(out))
    return out


def round_bf16(x) -> np.ndarray:
    """float64 -> bf16 bit patterns, rounded once to nearest, ties to even
    (the pooled keys are handed to the scoring step as bf16, like every
    indexer key).  Finite normal-range values only."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(np.abs(x))       # |x| = m * 2^e, m in [0.5, 1)
    q = np.ldexp(m, 8)               # the 8 significant bits, in [128, 256)
    fl = np.floor(q)
    r = q - fl
    fl = fl + ((r > 0.5) | ((r == 0.5) & (np.fmod(fl, 2.0) == 1.0)))
    mag = np.ldexp(fl, e - 8)                # exact in float32
    val = np.where(np.signbit(x), -mag, mag)
    return (val.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def indexer_pooled_fwd(q, k_raw, gate, ape, valid, w, kpool: int,
                       first_key: int, index_topk: int, q_pos=None,
                       want_logits: bool = False, rows=None):
    """The pool variant end to end (page "Module glm5next_dsa", "Shape of the
    pipeline"): kpool_compress -> index_scores over pools (a pool is a
    candidate when valid and whole-block visible) -> top index_topk / kpool
    pools -> expand_selection to index_topk token ids.

    Pool p covers tokens first_key + p*kpool .. + kpool - 1 and is visible at
    position t when its last token is at or before t: the plain rule with
    ratio kpool at the shifted position t - first_key.  Returns the oracle's
    forward dict over pools plus "tokens", "keys_bf16" and "pool_valid".
    """
    assert index_topk > 0 and index_topk % kpool == 0
    c = kpool_compress(k_raw, gate, ape, valid, kpool, first_key)
    B = c["keys"].shape[1] if c["P"] else _bits(k_raw).shape[1]
    keys = round_bf16(c["keys"])
    import torch
    kt = torch.from_numpy(keys.view(np.int16)).view(torch.bfloat16)
    base = np.zeros(B, np.int64) if q_pos is None else \
        _arr(q_pos, np.int32).astype(np.int64).reshape(B)
    shifted = (base - first_key).astype(np.int32)
    out = indexer_fwd(q, kt, w, kpool, index_topk // kpool, q_pos=shifted,
                      want_logits=want_logits, key_valid=c["valid"],
                      rows=rows)
    out["tokens"] = expand_selection(out["idx"], kpool, first_key)
    out["keys_bf16"] = keys
    out["pool_valid"] = c["valid"]
    return out


def sparse_mla_fwd(q, c, idx, scale: float, n_threads: int | None = None):
    """Sparse MLA forward over selected tokens (see oracle_sparse_mla_fwd in
    the C file): q [S,B,H,Dc] bf16, latent cache c [T,B,Dc] bf16, idx
    [B,S,topk] int32 token ids.  Returns {"o": [S,B,H,Dc] float64,
    "lse": [S,B,H] float64}."""
    lib = _load()
    qb, cb = _bits(q), _bits(c)
    S, B, H, Dc = qb.shape
    T = cb.shape[0]
    assert cb.shape == (T, B, Dc), cb.shape
    gi = _arr(idx, np.int32)
    topk = gi.shape[-1]
    gi = gi.reshape(B, S, topk)
    o = np.empty((S, B, H, Dc), np.float64)
    lse = np.empty((S, B, H), np.float64)
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    lib.oracle_sparse_mla_fwd(_ptr(qb), _ptr(cb), _ptr(gi), S, B, H, Dc, T,
                              topk, float(scale), _ptr(o), _ptr(lse),
                              int(n_threads))
    return {"o": o, "lse": lse}
