"""The C ABI library: it builds, loads, exports every declared entry point
and rejects bad arguments synchronously (no GPU needed: every case here
returns before the library touches a device)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

from dsa_sparse_attention_fwd_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA, TIMEOUT, RANGE = range(7)


@pytest.fixture(scope="module")
def lib():
    path = _build.build()
    L = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.dsa_indexer_fwd.restype = I
    L.dsa_indexer_fwd.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P, P, P,
                                  P, Z, P]
    L.dsa_indexer_fwd_profiled.restype = I
    L.dsa_indexer_fwd_profiled.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P,
                                           P, P, P, Z, P, P, I]
    L.dsa_indexer_logits.restype = I
    L.dsa_indexer_logits.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P, Z, P]
    L.dsa_indexer_workspace_size.restype = Z
    L.dsa_indexer_workspace_size.argtypes = [I] * 8
    L.dsa_set_prefill_policy.restype = I
    L.dsa_set_prefill_policy.argtypes = [I]
    L.dsa_indexer_fwd_launches.restype = I
    L.dsa_indexer_fwd_launches.argtypes = [I] * 8
    L.dsa_indexer_logits_workspace_size.restype = Z
    L.dsa_status_string.restype = ctypes.c_char_p
    L.dsa_status_string.argtypes = [I]
    L.dsa_indexer_check.restype = I
    L.dsa_indexer_check.argtypes = [P, P]
    L.dsa_selftest_wait_limit.restype = I
    L.dsa_selftest_wait_limit.argtypes = [I, P, Z, P]
    L.dsa_indexer_varlen_workspace_size.restype = Z
    L.dsa_indexer_varlen_workspace_size.argtypes = [I, P, P, I, I, I, I, I]
    L.dsa_indexer_fwd_varlen.restype = I
    L.dsa_indexer_fwd_varlen.argtypes = [P, P, P, I, P, P, I, I, I, I, P, P,
                                         P, P, P, Z, P]
    L.dsa_indexer_host_buffer_size.restype = Z
    L.dsa_indexer_host_buffer_size.argtypes = [I] * 8
    L.dsa_indexer_fwd_host.restype = I
    L.dsa_indexer_fwd_host.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P, P,
                                       P, P, Z, P]
    L.dsa_kpool_compress.restype = I
    L.dsa_kpool_compress.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P]
    L.dsa_expand_selection.restype = I
    L.dsa_expand_selection.argtypes = [P, ctypes.c_longlong, I, I, I, P, P]
    L.dsa_indexer_pooled_workspace_size.restype = Z
    L.dsa_indexer_pooled_workspace_size.argtypes = [I] * 8
    L.dsa_indexer_fwd_pooled.restype = I
    L.dsa_indexer_fwd_pooled.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I,
                                         I, I, P, P, P, P, P, Z, P]
    L.dsa_sparse_mla_workspace_size.restype = Z
    L.dsa_sparse_mla_workspace_size.argtypes = []
    L.dsa_sparse_mla_fwd.restype = I
    L.dsa_sparse_mla_fwd.argtypes = [P, P, P, I, I, I, I, I, I,
                                     ctypes.c_float, P, P, P, Z, P]
    L.dsa_indexer_bwd_workspace_size.restype = Z
    L.dsa_indexer_bwd_workspace_size.argtypes = []
    L.dsa_indexer_bwd.restype = I
    L.dsa_indexer_bwd.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P, P, P, P,
                                  P, P, Z, P]
    return L


def declared_functions():
    names = set()
    for h in os.listdir(INCLUDE):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(INCLUDE, h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(dsa_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("dsa_indexer_fwd", "dsa_indexer_workspace_size",
              "dsa_status_string", "dsa_indexer_check", "dsa_indexer_logits",
              "dsa_indexer_fwd_profiled", "dsa_set_prefill_policy",
              "dsa_indexer_fwd_launches"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib):
    """Only the declared C entry points are visible (hidden visibility)."""
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH],
                         capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines()
                if " T " in l and l.split()[-1].startswith("dsa_")}
    assert exported == set(declared_functions())


def test_status_strings(lib):
    for code in range(7):
        s = lib.dsa_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.dsa_status_string(99).decode() == "unknown status"


def test_workspace_size(lib):
    ws = lib.dsa_indexer_workspace_size
    # one-kernel prefill (scores and selection in the same kernel): the
    # status header, then the kernel's per-CTA scratch (160 CTAs x 2 item
    # slots x 256/H rows of S_kv rounded up to 32, plus 32, fp32), whatever S
    fused = lambda H, S_kv: 256 + 160 * 2 * (256 // H) * (
        (S_kv + 31) // 32 * 32 + 32) * 4
    # two-kernel top-k path: the status header, then the logits of one chunk
    # of query rows (all rows when B*S*S_kv*4 <= 64 MiB, else the most whole
    # scoring tiles of 256/H rows that fit), whatever S
    def chunked(S, B, H, S_kv):
        per_row = B * S_kv * 4
        if S * per_row <= 64 << 20:
            return 256 + S * per_row
        tq = 256 // H
        rows = max(tq, (64 << 20) // per_row // tq * tq)
        return 256 + min(rows, S) * per_row
    # default policy: one kernel for rows of at least 8192 keys
    assert ws(65536, 1, 64, 128, 16384, 4, 2048, 0) == fused(64, 16384)
    assert ws(8192, 1, 32, 128, 8192, 1, 2048, 0) == fused(32, 8192)
    assert ws(4096, 1, 64, 128, 4096, 1, 2048, 0) == chunked(4096, 1, 64, 4096)
    assert ws(4096, 1, 64, 128, 4096, 1, 2048, 0) == 256 + (64 << 20)
    assert ws(16384, 2, 64, 128, 4096, 4, 512, 0) == 256 + 2 * 2048 * 4096 * 4
    assert ws(40, 1, 128, 128, 40, 1, 7, 0) == chunked(40, 1, 128, 40)
    # shapes the one-kernel forward does not take: chunked logits
    assert ws(8192, 1, 64, 128, 8192, 1, 4096, 0) == chunked(8192, 1, 64, 8192)
    assert ws(64, 1, 16, 64, 64, 1, 8, 0) == 256 + 64 * 64 * 4
    assert ws(1, 64, 32, 64, 8192, 4, 512, 0) == 256 + 64 * 8192 * 4  # decode
    assert ws(3, 2, 64, 128, 500, 1, 16, 0) == 256 + 2 * 3 * 500 * 4
    # forced policies
    try:
        assert lib.dsa_set_prefill_policy(1) == 0
        assert ws(4096, 1, 64, 128, 4096, 1, 2048, 0) == fused(64, 4096)
        assert ws(16384, 2, 64, 128, 4096, 4, 512, 0) == fused(64, 4096)
        assert ws(8, 1, 64, 64, 1000, 1, 100, 0) == fused(64, 1000)
        assert ws(64, 1, 16, 64, 64, 1, 8, 0) == 256 + 64 * 64 * 4  # H = 16
        assert lib.dsa_set_prefill_policy(2) == 0
        assert ws(65536, 1, 64, 128, 16384, 4, 2048, 0) == chunked(
            65536, 1, 64, 16384)
        assert lib.dsa_set_prefill_policy(3) == 1  # DSA_ERR_INVALID_ARG
    finally:
        assert lib.dsa_set_prefill_policy(0) == 0
    # given indices: H in {16, 32, 64, 128} gathers keys (status header
    # only); other H read the scores back from logits
    assert ws(65536, 1, 64, 128, 16384, 4, 2048, 1) == 256
    assert ws(1, 64, 16, 64, 8192, 4, 512, 1) == 256
    assert ws(64, 1, 4, 32, 64, 1, 8, 1) == 256 + 64 * 64 * 4
    assert ws(0, 1, 64, 128, 4096, 1, 2048, 1) == 0
    assert ws(0, 1, 64, 128, 4096, 1, 2048, 0) == 0
    assert ws(16, 1, 3, 128, 16, 1, 4, 0) == 0
    assert ws(16, 1, 4, 128, 16, 1, 0, 0) == 0
    assert lib.dsa_indexer_logits_workspace_size() == 256


FAKE = 1 << 20  # aligned, never dereferenced: every case fails before use


def _fwd(lib, q=FAKE, k=FAKE, w=FAKE, S=16, B=1, H=4, D=32, S_kv=16, r=1,
         topk=4, q_pos=None, in_idx=None, oi=FAKE, os_=FAKE, ws=FAKE,
         wsb=1 << 30):
    return lib.dsa_indexer_fwd(q, k, w, S, B, H, D, S_kv, r, topk, q_pos,
                               in_idx, oi, os_, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), INVALID), (dict(k=None), INVALID), (dict(w=None), INVALID),
    (dict(oi=None), INVALID), (dict(os_=None), INVALID),
    (dict(S=0), INVALID), (dict(B=-1), INVALID), (dict(S_kv=0), INVALID),
    (dict(r=0), INVALID), (dict(topk=0), INVALID), (dict(D=0), INVALID),
    (dict(H=3), UNSUPPORTED), (dict(H=256), UNSUPPORTED),
    (dict(D=12), UNSUPPORTED), (dict(D=136), UNSUPPORTED),
    (dict(topk=8193), UNSUPPORTED),
    (dict(q=FAKE + 8), INVALID), (dict(k=FAKE + 2), INVALID),
    (dict(ws=None), WORKSPACE), (dict(wsb=100), WORKSPACE),
    (dict(ws=FAKE + 4), INVALID),
])
def test_fwd_rejects_bad_arguments(lib, kw, code):
    assert _fwd(lib, **kw) == code


def test_profiled_rejects_bad_events(lib):
    f = lib.dsa_indexer_fwd_profiled
    args = [FAKE, FAKE, FAKE, 16, 1, 4, 32, 16, 1, 4, None, None, FAKE, FAKE,
            FAKE, 1 << 30, None]
    assert f(*args, None, 2) == INVALID
    assert f(*args, None, -1) == INVALID
    evs = (ctypes.c_void_p * 2)(None, None)
    assert f(*args, evs, 2) == INVALID


def test_logits_rejects_bad_arguments(lib):
    f = lib.dsa_indexer_logits
    assert f(None, FAKE, FAKE, 8, 1, 4, 32, 8, 1, None, FAKE, FAKE, 256,
             None) == INVALID
    assert f(FAKE, FAKE, FAKE, 8, 1, 5, 32, 8, 1, None, FAKE, FAKE, 256,
             None) == UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, 8, 1, 4, 32, 8, 1, None, FAKE, FAKE, 16,
             None) == WORKSPACE


def test_check_rejects_null_workspace(lib):
    assert lib.dsa_indexer_check(None, None) == INVALID
    assert lib.dsa_selftest_wait_limit(10, None, 0, None) == WORKSPACE


def test_python_binding_fails_loudly_without_library(tmp_path):
    import dsa_sparse_attention_fwd_gb300 as m
    saved = m._lib
    try:
        m._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            m.load_library(str(tmp_path / "missing.so"))
    finally:
        m._lib = saved


def test_launch_counts(lib):
    n = lib.dsa_indexer_fwd_launches
    assert n(65536, 1, 64, 128, 16384, 4, 2048, 0) == 1   # one kernel
    assert n(4096, 1, 64, 128, 4096, 1, 2048, 0) == 2     # one chunk
    assert n(16384, 2, 64, 128, 4096, 4, 512, 0) == 16    # 8 chunks x 2
    assert n(65536, 1, 64, 128, 16384, 4, 2048, 1) == 1   # gathered keys
    assert n(64, 1, 4, 32, 64, 1, 8, 1) == 2              # logits + gather
    assert n(1, 64, 64, 128, 8192, 4, 512, 0) == 2        # decode
    assert n(0, 1, 64, 128, 4096, 1, 2048, 0) == 0


def test_host_buffer_size(lib):
    hb = lib.dsa_indexer_host_buffer_size
    ws = lib.dsa_indexer_workspace_size
    assert hb(0, 1, 64, 128, 4096, 1, 2048, 0) == 0
    assert hb(16, 1, 3, 128, 16, 1, 4, 0) == 0
    # one chunk: inputs + outputs + status + the workspace of the whole call
    S, B, H, D, S_kv, k = 128, 1, 4, 32, 128, 16
    need = hb(S, B, H, D, S_kv, 1, k, 0)
    inputs = S_kv * B * D * 2 + S * B * H * D * 2 + S * B * H * 4
    assert need >= inputs + 2 * B * S * k * 4 + ws(S, B, H, D, S_kv, 1, k, 0)
    # eight chunks of 512 rows: the workspace is one chunk's, not the call's
    big = hb(4096, 1, 16, 128, 4096, 1, 2048, 0)
    assert big < (4096 * 16 * 128 * 2 + 2 * 4096 * 2048 * 4
                  + ws(4096, 1, 16, 128, 4096, 1, 2048, 0))
    assert big >= 4096 * 16 * 128 * 2 + 2 * 4096 * 2048 * 4 + ws(
        512, 1, 16, 128, 4096, 1, 2048, 0)


def test_host_fwd_rejects_bad_arguments(lib):
    f = lib.dsa_indexer_fwd_host
    H = FAKE
    need = lib.dsa_indexer_host_buffer_size(16, 1, 4, 32, 16, 1, 4, 0)
    args = dict(q=H, k=H, w=H, oi=H, os_=H, buf=FAKE, nb=need)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["q"], a["k"], a["w"], 16, 1, 4, 32, 16, 1, 4, None, None,
                 a["oi"], a["os_"], a["buf"], a["nb"], None)
    assert call(q=None) == INVALID
    assert call(oi=None) == INVALID
    assert call(buf=None) == WORKSPACE
    assert call(nb=need - 1) == WORKSPACE
    assert call(buf=FAKE + 16) == INVALID  # not 256-byte aligned
    assert f(H, H, H, 16, 1, 3, 32, 16, 1, 4, None, None, H, H, FAKE, 1 << 30,
             None) == UNSUPPORTED
    assert f(H, H, H, 0, 1, 4, 32, 16, 1, 4, None, None, H, H, FAKE, 1 << 30,
             None) == INVALID


def _i32(*v):
    return (ctypes.c_int32 * len(v))(*v)


def test_varlen_workspace_size(lib):
    vw = lib.dsa_indexer_varlen_workspace_size
    ws = lib.dsa_indexer_workspace_size
    up = lambda x: (x + 255) // 256 * 256
    # two sequences with rows: two slices of the larger one's workspace
    cq, ck = _i32(0, 100, 300), _i32(0, 25, 75)
    assert vw(2, cq, ck, 64, 128, 4, 32, 0) == 2 * up(
        ws(200, 1, 64, 128, 50, 4, 32, 0))
    # an empty sequence and a keyless one add no slices
    cq, ck = _i32(0, 0, 10, 40), _i32(0, 5, 5, 20)
    assert vw(3, cq, ck, 16, 64, 1, 8, 0) == 2 * up(
        ws(30, 1, 16, 64, 15, 1, 8, 0))
    # at most four slices
    cq = _i32(*[i * 10 for i in range(9)])
    ck = _i32(*[i * 10 for i in range(9)])
    assert vw(8, cq, ck, 4, 32, 1, 4, 0) == 4 * up(ws(10, 1, 4, 32, 10, 1, 4, 0))
    # malformed offsets
    assert vw(2, _i32(1, 5, 9), _i32(0, 5, 9), 4, 32, 1, 4, 0) == 0
    assert vw(2, _i32(0, 5, 4), _i32(0, 5, 9), 4, 32, 1, 4, 0) == 0
    assert vw(0, _i32(0), _i32(0), 4, 32, 1, 4, 0) == 0
    assert vw(1, _i32(0, 5), _i32(0, 5), 3, 32, 1, 4, 0) == 0  # H = 3


def test_varlen_rejects_bad_arguments(lib):
    f = lib.dsa_indexer_fwd_varlen
    cq, ck = _i32(0, 16, 40), _i32(0, 16, 40)
    need = lib.dsa_indexer_varlen_workspace_size(2, cq, ck, 4, 32, 1, 4, 0)

    def call(q=FAKE, cq=cq, ck=ck, n=2, ws=FAKE, nb=need, topk=4):
        return f(q, FAKE, FAKE, n, cq, ck, 4, 32, 1, topk, None, None, FAKE,
                 FAKE, ws, nb, None)
    assert call(q=None) == INVALID
    assert call(cq=None) == INVALID
    assert call(n=0) == INVALID
    assert call(topk=0) == INVALID
    assert call(ws=None) == WORKSPACE
    assert call(nb=need // 2 - 1) == WORKSPACE  # less than one slice
    assert call(ws=FAKE + 16) == INVALID
    assert call(cq=_i32(0, 16, 8)) == INVALID


def test_bwd_rejects_bad_arguments(lib):
    f = lib.dsa_indexer_bwd
    assert lib.dsa_indexer_bwd_workspace_size() == 256

    def call(q=FAKE, k=FAKE, gk=FAKE, H=64, D=128, S=8, topk=4, ws=FAKE,
             nb=256, idx=FAKE):
        return f(q, k, FAKE, S, 1, H, D, 8, 1, topk, None, idx, FAKE, FAKE,
                 gk, FAKE, ws, nb, None)
    assert call(q=None) == INVALID
    assert call(idx=None) == INVALID
    assert call(gk=None) == INVALID
    assert call(S=0) == INVALID
    assert call(topk=0) == INVALID
    assert call(H=32) == UNSUPPORTED
    assert call(D=136) == UNSUPPORTED
    assert call(D=60) == UNSUPPORTED
    assert call(k=FAKE + 8) == INVALID   # k not 16-byte aligned
    assert call(gk=FAKE + 4) == INVALID  # grad_k not 16-byte aligned
    assert call(ws=None) == WORKSPACE
    assert call(nb=255) == WORKSPACE
    assert call(ws=FAKE + 16) == INVALID


def test_pool_entry_points_reject_bad_arguments(lib):
    pw = lib.dsa_indexer_pooled_workspace_size
    assert pw(16, 1, 64, 128, 64, 4, 0, 32) > 256
    assert pw(16, 1, 64, 128, 64, 4, 0, 30) == 0   # topk not a multiple
    assert pw(16, 1, 64, 128, 64, 0, 0, 32) == 0   # kpool 0
    assert pw(16, 1, 64, 128, 3, 4, 0, 32) == 256  # no whole pool
    need = pw(16, 1, 64, 128, 64, 4, 0, 32)
    f = lib.dsa_indexer_fwd_pooled

    def call(q=FAKE, k=FAKE, kpool=4, topk=32, D=128, ws=FAKE, nb=need,
             fk=0):
        return f(q, k, FAKE, FAKE, None, FAKE, 16, 1, 64, D, 64, kpool, fk,
                 topk, None, FAKE, FAKE, FAKE, ws, nb, None)
    assert call(q=None) == INVALID
    assert call(k=None) == INVALID
    assert call(kpool=9) == UNSUPPORTED   # more slots than the kernel holds
    assert call(topk=30) == INVALID
    assert call(D=60) == UNSUPPORTED
    assert call(fk=-1) == INVALID
    assert call(ws=None) == WORKSPACE
    assert call(nb=need - 1) == WORKSPACE
    assert call(ws=FAKE + 16) == INVALID
    c = lib.dsa_kpool_compress
    assert c(None, FAKE, FAKE, None, 64, 1, 128, 4, 0, FAKE, None,
             None) == INVALID
    assert c(FAKE, FAKE, FAKE, None, 64, 1, 128, 9, 0, FAKE, None,
             None) == UNSUPPORTED
    assert c(FAKE + 8, FAKE, FAKE, None, 64, 1, 128, 4, 0, FAKE, None,
             None) == INVALID
    e = lib.dsa_expand_selection
    assert e(None, 1, 4, 4, 0, FAKE, None) == INVALID
    assert e(FAKE, 1, 0, 4, 0, FAKE, None) == INVALID


def test_sparse_mla_rejects_bad_arguments(lib):
    f = lib.dsa_sparse_mla_fwd
    assert lib.dsa_sparse_mla_workspace_size() == 256

    def call(q=FAKE, H=64, Dc=512, scale=0.05, ws=FAKE, nb=256, topk=32):
        return f(q, FAKE, FAKE, 4, 1, H, Dc, 100, topk, scale, FAKE, FAKE, ws,
                 nb, None)
    assert call(q=None) == INVALID
    assert call(topk=0) == INVALID
    assert call(scale=0.0) == INVALID
    assert call(scale=-1.0) == INVALID
    assert call(H=32) == UNSUPPORTED
    assert call(Dc=576) == UNSUPPORTED
    assert call(Dc=64) == UNSUPPORTED
    assert call(q=FAKE + 8) == INVALID
    assert call(ws=None) == WORKSPACE
    assert call(nb=100) == WORKSPACE


# ---- how the host-buffer entry point splits and orders the rows ----------

def _plan(S, B, H, D, S_kv, ratio, topk, q_pos=None, given=False, sms=152):
    import dsa_sparse_attention_fwd_gb300 as m
    return m.dsa_indexer_host_plan(S, B, H, D, S_kv, ratio, topk, q_pos=q_pos,
                                   has_in_idx=given, sms=sms)


def _check_starts(starts, S, unit):
    assert starts[0] == 0 and starts[-1] == S
    assert all(b > a for a, b in zip(starts, starts[1:]))
    assert all(s % 4 == 0 for s in starts[:-1])
    assert all(s % unit == 0 for s in starts[:-1])


def test_host_plan_compute_bound_alternates():
    """Long-context C4 (about 4070 tensor FLOPs per copied byte) alternates
    the costliest and the cheapest chunk left; with 152 SMs and H = 64 the
    chunk starts fall on whole waves of 152 items of 4 rows."""
    starts, order = _plan(65536, 1, 64, 128, 16384, 4, 2048)
    assert len(order) == 16
    _check_starts(starts, 65536, 608)
    assert order == [15, 0, 14, 1, 13, 2, 12, 3, 11, 4, 10, 5, 9, 6, 8, 7]
    # rows deep into a long sequence: compute-bound at 2048 rows as well
    starts, order = _plan(2048, 1, 64, 128, 8192, 1, 64, q_pos=[4096])
    assert order == [3, 0, 2, 1] and starts == [0, 512, 1024, 1536, 2048]


def test_host_plan_link_bound_takes_last_rows_first():
    # C4 prefill: 2 sequences, so a wave of 152 items is 304 rows
    starts, order = _plan(16384, 2, 64, 128, 4096, 4, 512)
    _check_starts(starts, 16384, 304)
    assert order == list(range(15, -1, -1))
    # V3.2: 512-row chunks hold less than a wave, plain 4-row starts
    starts, order = _plan(4096, 1, 64, 128, 4096, 1, 2048)
    assert starts == [512 * i for i in range(9)]
    assert order == list(range(7, -1, -1))
    # given indices at long C4: q, the indices and the outputs per row
    # against at most topk products per row
    starts, order = _plan(65536, 1, 64, 128, 16384, 4, 2048, given=True)
    assert order == list(range(15, -1, -1))


def test_host_plan_edges():
    # fewer than 1024 rows: one chunk
    assert _plan(1000, 1, 64, 128, 4096, 4, 512) == ([0, 1000], [0])
    # decode rows: one chunk
    assert _plan(1, 64, 64, 128, 8192, 4, 512,
                 q_pos=list(range(2048, 2048 + 64))) == ([0, 1], [0])
    # no SM count given and no device: 4-row starts of an even split
    import torch
    if not torch.cuda.is_available():
        starts, _ = _plan(65536, 1, 64, 128, 16384, 4, 2048, sms=0)
        assert starts == [4096 * i for i in range(17)]
    # an invalid shape is refused
    import dsa_sparse_attention_fwd_gb300 as m
    with pytest.raises(m.DsaError):
        _plan(0, 1, 64, 128, 16384, 4, 2048)
