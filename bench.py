#!/usr/bin/env python3
"""Benchmark of the DSA lightning-indexer forward on GB300.

One step = the whole forward (scoring + top-k selection) over one batch of
synthetic input of the long-context C4 prefill workload (B=1, S=65536,
compress_ratio=4 so S_kv=16384, H=64, D=128, topk=2048, causal), the
largest configuration that fits one GPU, inputs resident in HBM.  Metric:
TFLOP/s over visible (query, key) pairs, 2*H*D FLOPs per pair, plus
queries/s.  L2 is flushed (a 256 MiB write, outside the timed events)
before every timed step.  `--workload v32_prefill | c4_prefill | decode |
tiny` times the other configurations.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--given-indices]

`--given-indices` times the given-indices forward instead (scores gathered
at caller-supplied indices: per row min(topk, n_vis) distinct visible keys,
the rest -1); its TFLOP/s counts 2*H*D per valid given index.

Under torchrun (N > 1) every rank runs an independent replica of the same
workload (the forward has no exchange step); the reported value is the sum
of all ranks' work over the slowest rank's time.  `--impl reference` times
the CPU oracle (plain C, fp64) on the host cores on a bounded row sample of
the same workload; only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("indexer fwd TFLOP/s (visible pairs) + queries/s; "
          "% of bf16 TC peak / HBM BW")
WORKLOAD = "long_c4"
L2_FLUSH_BYTES = 256 << 20


def prefill_policy(dsa, name: str) -> None:
    """Apply --prefill (auto: one kernel for rows of at least 8192 keys,
    else scores then selection; one / two: force a path)."""
    dsa.dsa_set_prefill_policy({"auto": dsa.PREFILL_AUTO,
                                "one": dsa.PREFILL_ONE_KERNEL,
                                "two": dsa.PREFILL_TWO_KERNELS}[name])


def visible_pairs(wl, q_pos=None) -> int:
    """Sum over rows of the number of visible compressed keys."""
    total = 0
    for b in range(wl.B):
        base = 0 if q_pos is None else int(q_pos[b])
        for s in range(wl.S):
            t = base + s
            total += max(0, min(wl.S_kv, (t + 1) // wl.compress_ratio))
    return total


def row_visible(wl, q_pos=None):
    """[B, S] number of visible compressed keys of every row."""
    import numpy as np
    pos = np.arange(wl.S, dtype=np.int64)[None, :].repeat(wl.B, 0)
    if q_pos is not None:
        pos = pos + np.asarray(q_pos, dtype=np.int64)[:, None]
    return np.clip((pos + 1) // wl.compress_ratio, 0, wl.S_kv)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return json.load(fh), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_sha(kernel: str = "index_scores") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dsa_sparse_attention_fwd_gb300", "csrc")
    for name in (kernel.replace("gather_logits", "topk_select") + ".cu",
                 "ptx.cuh", "common.cuh"):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of a kernel on a bench workload, from the
    committed ncu summary, only if it was taken on the current kernel source
    and for this workload (a call that launches the kernel once per row
    chunk records the sum over the call's launches)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    sha = kernel_source_sha(kernel)
    for e in d.get("entries", []):
        if e.get("bench_workload") == workload and e.get("source_sha") == sha:
            return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}",
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        pw = [v for v in (num(r[3]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier_ranks(world: int) -> None:
    """Barrier across the replicas (no-op for one process)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (the slowest replica's time); the
    tensor lives on `device` (the GPU under NCCL, the CPU under gloo)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# the oracle's pace on the host (fp64 multiply-adds per second over all
# cores), used only to size the timed row sample to about 15 s of work
ORACLE_MAC_PER_S = 1.5e10
CPU_SAMPLE_S = 15.0


def cpu_sample_stride(wl, pairs: int) -> int:
    """Row stride that gives the oracle about CPU_SAMPLE_S seconds of work
    (1 = every row)."""
    macs = float(pairs) * wl.H * wl.D
    return max(1, int(math.ceil(macs / (ORACLE_MAC_PER_S * CPU_SAMPLE_S))))


def cpu_oracle_sample(wl, rows_every: int, in_idx=None):
    """Time the oracle on every `rows_every`-th row (from the last row down,
    so the longest rows are in the sample)."""
    import numpy as np

    import oracle
    from dsa_inputs import make_inputs
    q, k, w, q_pos = make_inputs(wl)
    rows = np.arange(wl.B * wl.S - 1, -1, -rows_every, dtype=np.int64)
    oracle.build()
    t0 = time.perf_counter()
    out = oracle.indexer_fwd(q, k, w, wl.compress_ratio, wl.topk, q_pos=q_pos,
                             rows=rows, in_idx=in_idx)
    dt = time.perf_counter() - t0
    if in_idx is None:
        pairs = int(np.asarray(out["nvis"], dtype=np.int64).sum())
    else:
        pairs = int((in_idx.reshape(-1, wl.topk)[rows] >= 0).sum())
    flops = 2.0 * wl.H * wl.D * pairs
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s",
            "cores": int(out["threads"]), "kind": "oracle",
            "sample": f"{rows.size} of {wl.B * wl.S} rows (every "
                      f"{rows_every}th from the last), {pairs} visible pairs, "
                      f"{dt:.2f} s",
            "queries_per_s": rows.size / dt}


def run_reference(args):
    """The reference arm: the CPU oracle, timed on the host cores."""
    rank, _, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from dsa_inputs import WORKLOADS, make_inputs
    wl = WORKLOADS[args.workload]
    q, k, w, q_pos = make_inputs(wl)
    oracle.build()
    n = wl.B * wl.S
    per_step = 16  # stride-spaced rows per step, rotating through the rows
    stride = max(1, n // per_step)
    times, pairs_total, threads = [], 0, 1
    for i in range(args.warmup + args.steps):
        off = (i * 7919) % stride
        rows = np.arange(off, n, stride, dtype=np.int64)[:per_step]
        t0 = time.perf_counter()
        out = oracle.indexer_fwd(q, k, w, wl.compress_ratio, wl.topk,
                                 q_pos=q_pos, rows=rows)
        dt = time.perf_counter() - t0
        threads = int(out["threads"])
        if i >= args.warmup:
            times.append(dt)
            pairs_total += int(np.asarray(out["nvis"], np.int64).sum())
    tot = sum(times)
    value = 2.0 * wl.H * wl.D * pairs_total / tot / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "S": wl.S,
                   "S_kv": wl.S_kv, "H": wl.H, "D": wl.D,
                   "compress_ratio": wl.compress_ratio, "topk": wl.topk,
                   "step": f"{per_step} stride-spaced rows per step"},
        "queries_per_s": per_step * len(times) / tot,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{per_step} rows per step x {len(times)} "
                                   f"steps, {pairs_total} visible pairs"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    import dsa_sparse_attention_fwd_gb300 as dsa
    from dsa_inputs import WORKLOADS, describe, make_inputs

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.build()
    dsa.load_library()
    prefill_policy(dsa, args.prefill)

    wl = WORKLOADS[args.workload]
    q, k, w, q_pos = make_inputs(wl)
    gi = gid = None
    if args.given_indices:
        from dsa_inputs import make_given_indices
        nv = row_visible(wl, None if q_pos is None else q_pos.tolist())
        gi = make_given_indices(wl.B, wl.S, wl.topk, nv, wl.idx_seed)
        pairs = int((gi >= 0).sum())
        gid = gi.to(dev)
    else:
        pairs = visible_pairs(wl, None if q_pos is None else q_pos.tolist())
    flops = 2.0 * wl.H * wl.D * pairs
    qd, kd, wd = q.to(dev), k.to(dev), w.to(dev)
    pd = q_pos.to(dev) if q_pos is not None else None
    out_idx = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device=dev)
    out_sc = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.float32,
                         device=dev)
    ws = torch.empty(dsa.dsa_indexer_workspace_size(
        wl.S, wl.B, wl.H, wl.D, wl.S_kv, wl.compress_ratio, wl.topk,
        gi is not None),
        dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(evs=None):
        dsa.dsa_indexer_fwd(qd, kd, wd, wl.compress_ratio, wl.topk, q_pos=pd,
                            in_idx=gid, out_idx=out_idx, out_scores=out_sc,
                            workspace=ws, stream=stream, stage_events=evs)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    rc = dsa.dsa_indexer_check(ws)
    if rc != 0:
        raise RuntimeError(f"device status {dsa.STATUS.get(rc, rc)}")

    K = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)
    # timed region: exactly K steps, one event pair around each (nothing
    # recorded between the kernels, so they chain as they do for a caller)
    ev = [(mk(), mk()) for _ in range(K)]
    for pair in ev:  # torch creates the CUDA event at its first record
        for e in pair:
            e.record(stream)
    sampler = ClockSampler(local)
    barrier_ranks(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(1.0)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier_ranks(world)
    clocks = sampler.stop()
    rc = dsa.dsa_indexer_check(ws)
    if rc != 0:
        raise RuntimeError(f"device status {dsa.STATUS.get(rc, rc)}")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    t_step = max_over_ranks(sum(step_ms) / K, world, dev)

    # per-kernel split: another K steps with an event after every kernel
    # (these can keep the next kernel from starting early, so they time the
    # kernels, not the step).  The two-kernel forward alternates scores and
    # selection, chunk by chunk.
    n_launch = dsa.dsa_indexer_fwd_launches(
        wl.S, wl.B, wl.H, wl.D, wl.S_kv, wl.compress_ratio, wl.topk,
        gi is not None)
    sev = [[mk() for _ in range(1 + max(2, n_launch))] for _ in range(K)]
    for evs in sev:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(1.0)
        step(sev[i])
    torch.cuda.synchronize()
    score_ms = [sum(e[j].elapsed_time(e[j + 1])
                    for j in range(0, max(1, n_launch - 1), 2))
                for e in sev]
    select_ms = [sum(e[j].elapsed_time(e[j + 1])
                     for j in range(1, max(2, n_launch), 2))
                 for e in sev]

    # ---- end to end through the C entry point on host buffers ----
    # (page-locked inputs and outputs and the device buffer are allocated
    # once, as a serving loop would; every step copies its inputs in and its
    # results out inside the timed region)
    qh, kh, wh = q.pin_memory(), k.pin_memory(), w.pin_memory()
    ph = q_pos.pin_memory() if q_pos is not None else None
    gh = gi.pin_memory() if gi is not None else None
    idx_h = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32,
                        pin_memory=True)
    sc_h = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.float32,
                       pin_memory=True)
    dbuf = torch.empty(dsa.dsa_indexer_host_buffer_size(
        wl.S, wl.B, wl.H, wl.D, wl.S_kv, wl.compress_ratio, wl.topk,
        gi is not None), dtype=torch.uint8, device=dev)

    def host_step():
        _, _, rc = dsa.dsa_indexer_fwd_host(
            qh, kh, wh, wl.compress_ratio, wl.topk, q_pos=ph, in_idx=gh,
            out_idx=idx_h, out_scores=sc_h, device_buf=dbuf, stream=stream)
        if rc != 0:
            raise RuntimeError(f"device status {dsa.STATUS.get(rc, rc)}")
    for _ in range(2):
        host_step()
    torch.cuda.synchronize()
    Ke = max(3, min(K, 50))
    e2e_ms = []
    for _ in range(Ke):
        a, b = mk(), mk()
        a.record(stream)
        host_step()
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    t_e2e = max_over_ranks(sum(e2e_ms) / Ke, world, dev)
    h2d = q.numel() * 2 + k.numel() * 2 + w.numel() * 4 + (
        q_pos.numel() * 4 if q_pos is not None else 0) + (
        gi.numel() * 4 if gi is not None else 0)
    d2h = sc_h.numel() * 4 + idx_h.numel() * 4

    if rank != 0:
        dist.destroy_process_group()
        return 0

    peaks, peak_src = read_peaks()
    t_score = statistics.mean(score_ms)
    t_second = statistics.mean(select_ms)
    tc_peak = float(peaks["bf16_tflops"])
    hbm_peak = float(peaks["hbm_gbs"])
    value = world * flops / (t_step * 1e-3) / 1e12
    rows = wl.B * wl.S
    # the given-indices path is one kernel when H has a gather instantiation
    direct = gi is not None and wl.H in (16, 32, 64, 128)
    decode_shape = wl.S < 256 // wl.H
    # the one-kernel forward (scores and selection together) ran
    fused = gi is None and n_launch == 1
    wkey = wl.name + (" given-indices" if gi is not None else "")

    def tensor_line(kernel, ms):
        a = flops / (ms * 1e-3) / 1e12
        return {"kernel": kernel, "bound": "tensor", "achieved": a,
                "peak": tc_peak, "unit": "TFLOP/s", "frac": a / tc_peak,
                "peak_source": f"{peak_src} bf16 burst",
                "algorithmic": f"{flops:.4g} FLOP per launch (2*H*D per pair)",
                "traffic": read_traffic(kernel, wkey)}

    def hbm_line(kernel, ms, nbytes, what):
        a = nbytes / (ms * 1e-3) / 1e9
        return {"kernel": kernel, "bound": "hbm", "achieved": a,
                "peak": hbm_peak, "unit": "GB/s", "frac": a / hbm_peak,
                "peak_source": f"{peak_src} copy bandwidth",
                "algorithmic": f"{nbytes:.4g} B per launch ({what})",
                "traffic": read_traffic(kernel, wkey)}

    if direct:
        kernels = {"gather_scores": t_score, "step": t_step}
        rooflines = {"gather_scores": tensor_line("gather_scores", t_score)}
        launches = 1
    elif fused:
        kernels = {"index_topk": t_score, "step": t_step}
        rooflines = {"index_topk": tensor_line("index_topk", t_score)}
        launches = 1
    else:
        if decode_shape and gi is None:
            sname = "decode_scores"
            kbytes = pairs * wl.D * 2 + rows * (wl.H * wl.D * 2 + wl.H * 4)
            first = hbm_line(sname, t_score, kbytes, "visible k rows + q + w")
        else:
            sname = "index_scores"
            first = tensor_line(sname, t_score)
        second = "gather_logits" if gi is not None else "topk_select"
        # the selection reads each visible logit once and writes the outputs
        sbytes = (pairs * 4 if gi is None else gi.numel() * 4 * 2) + \
            rows * wl.topk * 8
        kernels = {sname: t_score, second: t_second, "step": t_step}
        rooflines = {sname: first,
                     second: hbm_line(second, t_second, sbytes,
                                      "visible logits read + idx/scores "
                                      "written")}
        launches = n_launch
    top = max((k for k in kernels if k != "step"), key=lambda k: kernels[k])
    name = wl.name + (" given-indices" if gi is not None else "")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": t_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": name, "desc": describe(wl),
                   "pairs": ("valid given indices" if gi is not None
                             else "visible (query, key) pairs"),
                   "visible_pairs": pairs, "flops_per_step": flops,
                   "l2": "flushed before each step (256 MiB write, outside "
                         "the timed events)",
                   "prefill_path": ("one kernel" if fused else
                                    f"{n_launch} kernels"),
                   "parallelism": f"replicas x{world}"},
        "queries_per_s": world * wl.B * wl.S / (t_step * 1e-3),
        "pct_of_bf16_peak": 100.0 * value / world / tc_peak,
        "kernels_ms": kernels,
        "roofline": rooflines[top],
        "rooflines": rooflines,
        "e2e": {"value": world * flops / (t_e2e * 1e-3) / 1e12,
                "unit": "TFLOP/s", "ms_per_step": t_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "dsa_indexer_fwd_host (C entry point, pinned host "
                       "buffers, copies pipelined over row chunks)"},
        "gpu_launches": launches * K,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        if gi is None:
            line["cpu_baseline"] = cpu_oracle_sample(
                wl, cpu_sample_stride(wl, pairs))
        else:
            every = max(1, wl.B * wl.S // 1024)
            line["cpu_baseline"] = cpu_oracle_sample(wl, every, in_idx=gi)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_varlen(args):
    """Packed variable-length sequences through dsa_indexer_fwd_varlen."""
    import numpy as np
    import torch

    import dsa_sparse_attention_fwd_gb300 as dsa
    from dsa_inputs import VARLEN_WORKLOADS, make_varlen_inputs

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.build()
    dsa.load_library()
    prefill_policy(dsa, args.prefill)
    vw = VARLEN_WORKLOADS[args.workload]
    q, k, w, cq, ck = make_varlen_inputs(vw)
    pairs = 0
    for i in range(len(vw.lens_q)):
        s = np.arange(cq[i + 1] - cq[i], dtype=np.int64)
        pairs += int(np.clip((s + 1) // vw.compress_ratio, 0,
                             ck[i + 1] - ck[i]).sum())
    flops = 2.0 * vw.H * vw.D * pairs
    qd, kd, wd = q.to(dev), k.to(dev), w.to(dev)
    T = int(cq[-1])
    oi = torch.empty((T, vw.topk), dtype=torch.int32, device=dev)
    osc = torch.empty((T, vw.topk), dtype=torch.float32, device=dev)
    ws = torch.empty(dsa.dsa_indexer_varlen_workspace_size(
        cq, ck, vw.H, vw.D, vw.compress_ratio, vw.topk), dtype=torch.uint8,
        device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        dsa.dsa_indexer_fwd_varlen(qd, kd, wd, cq, ck, vw.compress_ratio,
                                   vw.topk, out_idx=oi, out_scores=osc,
                                   workspace=ws, stream=stream)
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if dsa.dsa_indexer_check(ws) != 0:
        raise RuntimeError("device status")
    K = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(mk(), mk()) for _ in range(K)]
    for a_, b_ in ev:
        a_.record(stream)
        b_.record(stream)
    sampler = ClockSampler(local)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)
    for i in range(K):
        flush.fill_(1.0)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier_ranks(world)
    clocks = sampler.stop()
    t_step = max_over_ranks(sum(a_.elapsed_time(b_) for a_, b_ in ev) / K,
                            world, dev)
    # end to end: inputs copied in from pinned host memory and the outputs
    # copied back, around the same call
    qh, kh, wh = q.pin_memory(), k.pin_memory(), w.pin_memory()
    oih = torch.empty((T, vw.topk), dtype=torch.int32, pin_memory=True)
    osh = torch.empty((T, vw.topk), dtype=torch.float32, pin_memory=True)
    e2e = []
    for i in range(max(3, min(K, 20)) + 2):
        a_, b_ = mk(), mk()
        a_.record(stream)
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        wd.copy_(wh, non_blocking=True)
        step()
        oih.copy_(oi, non_blocking=True)
        osh.copy_(osc, non_blocking=True)
        b_.record(stream)
        b_.synchronize()
        if i >= 2:
            e2e.append(a_.elapsed_time(b_))
    t_e2e = max_over_ranks(sum(e2e) / len(e2e), world, dev)
    if rank != 0:
        return 0
    peaks, peak_src = read_peaks()
    tc_peak = float(peaks["bf16_tflops"])
    value = world * flops / (t_step * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": t_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": vw.name, "lens_q": list(vw.lens_q),
                   "H": vw.H, "D": vw.D, "compress_ratio": vw.compress_ratio,
                   "topk": vw.topk, "visible_pairs": pairs,
                   "flops_per_step": flops,
                   "l2": "flushed before each step (256 MiB write, outside "
                         "the timed events)",
                   "parallelism": f"replicas x{world}"},
        "queries_per_s": world * T / (t_step * 1e-3),
        "roofline": {"kernel": "varlen dispatch (every kernel of the call)",
                     "bound": "tensor", "achieved": value / world,
                     "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": value / world / tc_peak,
                     "peak_source": f"{peak_src} bf16 burst",
                     "traffic": None},
        "e2e": {"value": world * flops / (t_e2e * 1e-3) / 1e12,
                "unit": "TFLOP/s", "ms_per_step": t_e2e,
                "h2d_bytes_per_step": q.numel() * 2 + k.numel() * 2 +
                w.numel() * 4,
                "d2h_bytes_per_step": oi.numel() * 8,
                "api": "torch copies + dsa_indexer_fwd_varlen"},
        # per sequence with keys the kernels of one B = 1 forward, plus the
        # status merge when more than one stream slice ran
        "gpu_launches": K * (sum(
            dsa.dsa_indexer_fwd_launches(cq[i + 1] - cq[i], 1, vw.H, vw.D,
                                         ck[i + 1] - ck[i], vw.compress_ratio,
                                         vw.topk)
            for i in range(len(vw.lens_q))
            if ck[i + 1] > ck[i] and cq[i + 1] > cq[i])
            + (1 if ws.numel() > ws.numel() // 2 and
               len(vw.lens_q) > 1 else 0)),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_oracle_bwd_sample(wl, gi, gs, q, k, w, n_rows: int):
    """Time the oracle's backward on `n_rows` rows spread over the problem,
    each as a one-row problem at its own position."""
    import numpy as np
    import torch

    import oracle
    oracle.build()
    rows = np.linspace(0, wl.S - 1, n_rows).astype(np.int64)
    pairs, dt = 0, 0.0
    for s in rows:
        for b in range(wl.B):
            pos = torch.tensor([int(s)], dtype=torch.int32)
            ix = gi[b:b + 1, s:s + 1]
            t0 = time.perf_counter()
            oracle.indexer_bwd(q[s:s + 1, b:b + 1], k[:, b:b + 1],
                               w[s:s + 1, b:b + 1], wl.compress_ratio, ix,
                               gs[b:b + 1, s:s + 1], q_pos=pos)
            dt += time.perf_counter() - t0
            pairs += int((ix >= 0).sum())
    return {"value": 6.0 * wl.H * wl.D * pairs / dt / 1e12,
            "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows.size * wl.B} rows (evenly spaced), {pairs} "
                      f"valid slots, {dt:.2f} s"}


def run_backward(args):
    """The indexer backward (gradients of the given-slots scores) at the
    workload's shape, with random valid visible indices and N(0, 1)
    upstream gradients."""
    import torch

    import dsa_sparse_attention_fwd_gb300 as dsa
    from dsa_inputs import WORKLOADS, describe, make_given_indices, make_inputs

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.build()
    dsa.load_library()
    wl = WORKLOADS[args.workload]
    q, k, w, q_pos = make_inputs(wl)
    nv = row_visible(wl, None if q_pos is None else q_pos.tolist())
    gi = make_given_indices(wl.B, wl.S, wl.topk, nv, wl.idx_seed)
    gs = torch.randn((wl.B, wl.S, wl.topk),
                     generator=torch.Generator().manual_seed(wl.seed + 100))
    pairs = int((gi >= 0).sum())
    flops = 6.0 * wl.H * wl.D * pairs  # three products of 2*H*D per slot
    qd, kd, wd = q.to(dev), k.to(dev), w.to(dev)
    pd = q_pos.to(dev) if q_pos is not None else None
    gid, gsd = gi.to(dev), gs.to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    gq = torch.empty((wl.S, wl.B, wl.H, wl.D), **f32)
    gk = torch.empty((wl.S_kv, wl.B, wl.D), **f32)
    gw = torch.empty((wl.S, wl.B, wl.H), **f32)
    ws = torch.empty(dsa.dsa_indexer_bwd_workspace_size(), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        dsa.dsa_indexer_bwd(qd, kd, wd, wl.compress_ratio, gid, gsd,
                            q_pos=pd, grad_q=gq, grad_k=gk, grad_w=gw,
                            workspace=ws, stream=stream)
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if dsa.dsa_indexer_check(ws) != 0:
        raise RuntimeError("device status")
    K = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(mk(), mk()) for _ in range(K)]
    sampler = ClockSampler(local)
    torch.cuda.synchronize()
    barrier_ranks(world)
    sampler.start()
    time.sleep(0.2)
    t0 = time.perf_counter()
    for i in range(K):
        flush.fill_(1.0)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier_ranks(world)
    clocks = sampler.stop()
    t_step = max_over_ranks(sum(a_.elapsed_time(b_) for a_, b_ in ev) / K,
                            world, dev)
    if dsa.dsa_indexer_check(ws) != 0:
        raise RuntimeError("device status")
    # end to end: inputs copied in from pinned host memory, the three
    # gradients copied back
    hin = [t.pin_memory() for t in (q, k, w, gi, gs)]
    din = [qd, kd, wd, gid, gsd]
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            for t in (gq, gk, gw)]
    e2e = []
    for i in range(max(3, min(K, 20)) + 2):
        a_, b_ = mk(), mk()
        a_.record(stream)
        for d_, h_ in zip(din, hin):
            d_.copy_(h_, non_blocking=True)
        step()
        for h_, d_ in zip(hout, (gq, gk, gw)):
            h_.copy_(d_, non_blocking=True)
        b_.record(stream)
        b_.synchronize()
        if i >= 2:
            e2e.append(a_.elapsed_time(b_))
    t_e2e = max_over_ranks(sum(e2e) / len(e2e), world, dev)
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    if rank != 0:
        return 0
    peaks, peak_src = read_peaks()
    tc_peak = float(peaks["bf16_tflops"])
    value = world * flops / (t_step * 1e-3) / 1e12
    achieved = flops / (t_step * 1e-3) / 1e12
    line = {
        "metric": "indexer bwd TFLOP/s (valid slots)", "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name + " backward", "desc": describe(wl),
                   "slots": "random distinct visible keys per row",
                   "valid_slots": pairs, "flops_per_step": flops,
                   "l2": "flushed before each step (256 MiB write, outside "
                         "the timed events)",
                   "parallelism": f"replicas x{world}"},
        "queries_per_s": world * wl.B * wl.S / (t_step * 1e-3),
        "kernels_ms": {"indexer_bwd (with the grad_k clear)": t_step},
        "roofline": {"kernel": "indexer_bwd", "bound": "tensor",
                     "achieved": achieved, "peak": tc_peak,
                     "unit": "TFLOP/s", "frac": achieved / tc_peak,
                     "peak_source": f"{peak_src} bf16 burst",
                     "algorithmic": f"{flops:.4g} FLOP per launch (6*H*D "
                                    "per valid slot)",
                     "timed": "the C call: grad_k clear + status clear + "
                              "the kernel",
                     "traffic": read_traffic("indexer_bwd",
                                             wl.name + " backward")},
        "e2e": {"value": world * flops / (t_e2e * 1e-3) / 1e12,
                "unit": "TFLOP/s", "ms_per_step": t_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "torch copies + dsa_indexer_bwd"},
        "gpu_launches": K,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_bwd_sample(wl, gi, gs, q, k, w, 24)
    print(json.dumps(line), flush=True)
    return 0


def run_pooled(args):
    """The pool variant at the C4 prefill shape: 2 x 16384 tokens pooled 4
    at a time (4096 pools per sequence), 16384 queries per sequence, the
    best 512 pools = 2048 tokens per row."""
    import numpy as np
    import torch

    import dsa_sparse_attention_fwd_gb300 as dsa

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.build()
    dsa.load_library()
    prefill_policy(dsa, args.prefill)
    B, S, T, H, D, kpool, fk, itopk = 2, 16384, 16384, 64, 128, 4, 0, 2048
    g = torch.Generator().manual_seed(21)
    q = torch.randn((S, B, H, D), generator=g).to(torch.bfloat16)
    k = torch.randn((T, B, D), generator=g).to(torch.bfloat16)
    gate = torch.randn((T, B, D), generator=g)
    ape = torch.randn((kpool, D), generator=g) * 0.5
    w = torch.randn((S, B, H), generator=g) * 0.125
    P = (T - fk) // kpool
    pos = np.arange(S, dtype=np.int64)
    pairs = B * int(np.clip((pos + 1 - fk) // kpool, 0, P).sum())
    flops = 2.0 * H * D * pairs
    qd, kd, gd, ad, wd = (t.to(dev) for t in (q, k, gate, ape, w))
    sk = itopk // kpool
    tok = torch.empty((B, S, itopk), dtype=torch.int32, device=dev)
    pl = torch.empty((B, S, sk), dtype=torch.int32, device=dev)
    sc = torch.empty((B, S, sk), dtype=torch.float32, device=dev)
    ws = torch.empty(dsa.dsa_indexer_pooled_workspace_size(
        S, B, H, D, T, kpool, fk, itopk), dtype=torch.uint8, device=dev)
    keys = torch.empty((P, B, D), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    lib = dsa.load_library()

    def step():
        dsa.dsa_indexer_fwd_pooled(qd, kd, gd, ad, wd, kpool, fk, itopk,
                                   out_tokens=tok, out_pools=pl,
                                   out_scores=sc, workspace=ws, stream=stream)

    def compress():
        rc = lib.dsa_kpool_compress(
            ctypes.c_void_p(kd.data_ptr()), ctypes.c_void_p(gd.data_ptr()),
            ctypes.c_void_p(ad.data_ptr()), None, T, B, D, kpool, fk,
            ctypes.c_void_p(keys.data_ptr()), None,
            ctypes.c_void_p(stream.cuda_stream))
        if rc != 0:
            raise RuntimeError(f"dsa_kpool_compress {rc}")
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step()
        compress()
    torch.cuda.synchronize()
    if dsa.dsa_indexer_check(ws) != 0:
        raise RuntimeError("device status")
    K = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(mk(), mk(), mk(), mk()) for _ in range(K)]
    sampler = ClockSampler(local)
    torch.cuda.synchronize()
    barrier_ranks(world)
    sampler.start()
    time.sleep(0.2)
    t0 = time.perf_counter()
    for i in range(K):
        flush.fill_(1.0)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
        flush.fill_(1.0)
        ev[i][2].record(stream)
        compress()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier_ranks(world)
    clocks = sampler.stop()
    t_step = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in ev) / K,
                            world, dev)
    t_comp = sum(e[2].elapsed_time(e[3]) for e in ev) / K
    # end to end: inputs in from pinned host memory, token ids back
    hin = [t.pin_memory() for t in (q, k, gate, ape, w)]
    din = [qd, kd, gd, ad, wd]
    hout = torch.empty(tok.shape, dtype=torch.int32, pin_memory=True)
    e2e = []
    for i in range(max(3, min(K, 10)) + 2):
        a_, b_ = mk(), mk()
        a_.record(stream)
        for d_, h_ in zip(din, hin):
            d_.copy_(h_, non_blocking=True)
        step()
        hout.copy_(tok, non_blocking=True)
        b_.record(stream)
        b_.synchronize()
        if i >= 2:
            e2e.append(a_.elapsed_time(b_))
    t_e2e = max_over_ranks(sum(e2e) / len(e2e), world, dev)
    if rank != 0:
        return 0
    peaks, peak_src = read_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    cbytes = T * B * D * (2 + 4) + kpool * D * 4 + P * B * D * 2
    comp_gbs = cbytes / (t_comp * 1e-3) / 1e9
    value = world * flops / (t_step * 1e-3) / 1e12
    line = {
        "metric": "indexer pooled fwd TFLOP/s (visible pool pairs)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "c4_pool (pool variant)", "B": B, "S": S,
                   "T_tokens": T, "kpool": kpool, "first_key": fk,
                   "pools": P, "index_topk": itopk, "H": H, "D": D,
                   "visible_pool_pairs": pairs, "flops_per_step": flops,
                   "l2": "flushed before each step (256 MiB write, outside "
                         "the timed events)",
                   "parallelism": f"replicas x{world}"},
        "queries_per_s": world * B * S / (t_step * 1e-3),
        "kernels_ms": {"whole call (compress + score + select + expand)":
                       t_step, "kpool_compress alone": t_comp},
        "roofline": {"kernel": "kpool_compress", "bound": "hbm",
                     "achieved": comp_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": comp_gbs / hbm_peak,
                     "peak_source": f"{peak_src} copy bandwidth",
                     "algorithmic": f"{cbytes:.4g} B per launch (k bf16 + "
                                    "gate fp32 read, pooled keys written)",
                     "traffic": read_traffic("pool", "c4_pool")},
        "e2e": {"value": world * flops / (t_e2e * 1e-3) / 1e12,
                "unit": "TFLOP/s", "ms_per_step": t_e2e,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size()
                                          for t in hin),
                "d2h_bytes_per_step": hout.numel() * 4,
                "api": "torch copies + dsa_indexer_fwd_pooled"},
        # per step: compression, the forward over the pools and the
        # expansion, plus the compression timed alone
        "gpu_launches": K * (3 + dsa.dsa_indexer_fwd_launches(
            S, B, H, D, P, kpool, itopk // kpool)),
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        rows = np.arange(B * S - 1, -1, -(B * S // 16), dtype=np.int64)
        t0 = time.perf_counter()
        ref = oracle.indexer_pooled_fwd(q, k, gate, ape, None, w, kpool, fk,
                                        itopk, rows=rows)
        dt = time.perf_counter() - t0
        sp = int(np.asarray(ref["nvis"], np.int64).sum())
        line["cpu_baseline"] = {
            "value": 2.0 * H * D * sp / dt / 1e12, "unit": "TFLOP/s",
            "cores": int(ref["threads"]), "kind": "oracle",
            "sample": f"compression of all {P * B} pools + {rows.size} rows "
                      f"({sp} visible pool pairs), {dt:.2f} s"}
    print(json.dumps(line), flush=True)
    return 0


def run_mla(args):
    """Sparse MLA forward over selected tokens at the 4096 x 4096 prefill:
    64 heads, latent width 512, 2048 random distinct visible tokens per row
    (fewer for the first rows)."""
    import numpy as np
    import torch

    import dsa_sparse_attention_fwd_gb300 as dsa
    from dsa_inputs import make_given_indices

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.build()
    dsa.load_library()
    S, B, H, Dc, T, topk = 4096, 1, 64, 512, 4096, 2048
    scale = 1.0 / math.sqrt(Dc)
    g = torch.Generator().manual_seed(31)
    q = torch.randn((S, B, H, Dc), generator=g).to(torch.bfloat16)
    c = torch.randn((T, B, Dc), generator=g).to(torch.bfloat16)
    lim = np.minimum(np.arange(S) + 1, T)[None, :]
    idx = make_given_indices(B, S, topk, lim, 32)
    slots = int((idx >= 0).sum())
    flops = 4.0 * H * Dc * slots  # q.c and p.c, 2*H*Dc each per valid slot
    qd, cd, xd = q.to(dev), c.to(dev), idx.to(dev)
    o = torch.empty((S, B, H, Dc), dtype=torch.float32, device=dev)
    lse = torch.empty((S, B, H), dtype=torch.float32, device=dev)
    ws = torch.empty(dsa.dsa_sparse_mla_workspace_size(), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        dsa.dsa_sparse_mla_fwd(qd, cd, xd, scale, out_o=o, out_lse=lse,
                               workspace=ws, stream=stream)
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if dsa.dsa_indexer_check(ws) != 0:
        raise RuntimeError("device status")
    K = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(mk(), mk()) for _ in range(K)]
    sampler = ClockSampler(local)
    torch.cuda.synchronize()
    barrier_ranks(world)
    sampler.start()
    time.sleep(0.2)
    t0 = time.perf_counter()
    for i in range(K):
        flush.fill_(1.0)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier_ranks(world)
    clocks = sampler.stop()
    t_step = max_over_ranks(sum(a_.elapsed_time(b_) for a_, b_ in ev) / K,
                            world, dev)
    hin = [t.pin_memory() for t in (q, c, idx)]
    din = [qd, cd, xd]
    ho = torch.empty(o.shape, dtype=torch.float32, pin_memory=True)
    e2e = []
    for i in range(max(3, min(K, 10)) + 2):
        a_, b_ = mk(), mk()
        a_.record(stream)
        for d_, h_ in zip(din, hin):
            d_.copy_(h_, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)
        b_.record(stream)
        b_.synchronize()
        if i >= 2:
            e2e.append(a_.elapsed_time(b_))
    t_e2e = max_over_ranks(sum(e2e) / len(e2e), world, dev)
    if rank != 0:
        return 0
    peaks, peak_src = read_peaks()
    tc_peak = float(peaks["bf16_tflops"])
    achieved = flops / (t_step * 1e-3) / 1e12
    line = {
        "metric": "sparse MLA fwd TFLOP/s (valid slots)",
        "value": world * achieved, "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": t_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "sparse MLA over selected tokens", "B": B,
                   "S": S, "T": T, "H": H, "Dc": Dc, "topk": topk,
                   "valid_slots": slots, "flops_per_step": flops,
                   "l2": "flushed before each step (256 MiB write, outside "
                         "the timed events)",
                   "parallelism": f"replicas x{world}"},
        "queries_per_s": world * B * S / (t_step * 1e-3),
        "roofline": {"kernel": "sparse_mla", "bound": "tensor",
                     "achieved": achieved, "peak": tc_peak,
                     "unit": "TFLOP/s", "frac": achieved / tc_peak,
                     "peak_source": f"{peak_src} bf16 burst",
                     "algorithmic": f"{flops:.4g} FLOP per launch (4*H*Dc "
                                    "per valid slot: the score and the "
                                    "output products)",
                     "traffic": read_traffic("sparse_mla", "sparse_mla")},
        "e2e": {"value": world * flops / (t_e2e * 1e-3) / 1e12,
                "unit": "TFLOP/s", "ms_per_step": t_e2e,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size()
                                          for t in hin),
                "d2h_bytes_per_step": ho.numel() * 4,
                "api": "torch copies + dsa_sparse_mla_fwd"},
        "gpu_launches": K,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        rows = [0, 1000, 2047, 4095]
        sel = idx[:, rows].contiguous()
        t0 = time.perf_counter()
        oracle.sparse_mla_fwd(q[rows].contiguous(), c, sel, scale)
        dt = time.perf_counter() - t0
        n = int((sel >= 0).sum())
        line["cpu_baseline"] = {
            "value": 4.0 * H * Dc * n / dt / 1e12, "unit": "TFLOP/s",
            "cores": os.cpu_count() or 1, "kind": "oracle",
            "sample": f"{len(rows)} rows, {n} valid slots, {dt:.2f} s"}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--given-indices", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="time the indexer backward instead of the forward")
    ap.add_argument("--prefill", choices=["auto", "one", "two"],
                    default="auto",
                    help="prefill top-k path: auto (one kernel for rows of "
                         "at least 8192 keys), or force one / two kernels")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    from dsa_inputs import VARLEN_WORKLOADS
    if args.workload in VARLEN_WORKLOADS:
        return run_varlen(args)
    if args.backward:
        return run_backward(args)
    if args.workload == "c4_pool":
        return run_pooled(args)
    if args.workload == "sparse_mla":
        return run_mla(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
