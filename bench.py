#!/usr/bin/env python3
"""Benchmark of the KPool DSA indexer hot path on GB300.

One step = the whole path over one batch of synthetic input:
  kpool_compress -> [kpool_quantize_fp8 (FP8 mode)] -> kpool_score_topk ->
  kpool_expand_indices
on the default workload ``long_128k`` (one sequence of T = 131072 tokens,
H = 64, D = 128, kpool = 4, index_topk = 2048), the size the scoring
kernel's tensor-core target is stated at.

Prints ONE JSON line (rank 0).  ``value`` is whole-job queries/s with inputs
resident in HBM; ``e2e`` is the same metric through the public API with the
inputs copied from pinned host memory and the token indices read back every
step; ``roofline`` is the dominant kernel (kpool_score_topk) against the
measured dense BF16 tensor peak; ``cpu_baseline`` is the CPU oracle timed on
a bounded sample of query rows of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle arm
Under torchrun (N > 1) every rank runs an independent replica (the path has
no exchange step); time is the max over ranks.
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
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_kpool_compress_gb300 import workloads as W  # noqa: E402

METRIC = "KPool indexer queries/s and scoring TFLOP/s (% of GB300 BF16/FP8 peak)"
UNIT = "queries/s"
SCORE_SRC = os.path.join(ROOT, "sparse_attention_kpool_compress_gb300", "csrc", "kpool_score.cu")


def sum_floor(L, kp):
    """sum_{x=1}^{L} floor(x / kp)."""
    m = L // kp
    return kp * m * (m - 1) // 2 + m * (L - m * kp + 1)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def measure_fp8_peak(dev, sustained_s=4.0):
    """Dense E4M3 tensor peak of this GPU, measured the way the BF16 peaks in
    MEASURED_PEAKS.json are: a library GEMM (torch._scaled_mm, cuBLASLt) on
    8192^3 E4M3 operands with FP32 accumulation and BF16 output, 2*N^3 flops;
    best of 10 CUDA-event-timed calls (burst) and calls back to back for
    `sustained_s` seconds (sustained).  Returns TFLOP/s figures and the clocks
    seen during the sustained loop."""
    n = 8192
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn).t()
    one = torch.ones((), device=dev, dtype=torch.float32)

    def gemm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    for _ in range(5):
        gemm()
    torch.cuda.synchronize()
    flop = 2.0 * n ** 3
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        gemm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    calls = 0
    t_end = time.perf_counter() + sustained_s
    e0.record()
    while time.perf_counter() < t_end:
        for _ in range(20):
            gemm()
        calls += 20
        torch.cuda.synchronize()
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    sus_ms = e0.elapsed_time(e1) / calls
    del a, b
    return {"fp8_tflops": flop / (best / 1000.0) / 1e12,
            "fp8_tflops_sustained": flop / (sus_ms / 1000.0) / 1e12,
            "how": "torch._scaled_mm E4M3 8192^3 (BF16 out), best of 10 and %.0f s back to back"
                   % sustained_s, "clocks_sustained": clocks}


def file_hash(path):
    """Fingerprint of a C/CUDA source: sha256 (16 hex digits) of its code with
    comments removed and whitespace collapsed, so that comment edits keep a
    recorded profile valid while any code change invalidates it."""
    import re
    with open(path, encoding="utf-8") as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    src = " ".join(src.split())
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """Per-launch DRAM bytes from a committed ncu summary, or None if absent or
    taken on a different version of the kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get("%s/%s" % (kernel, workload))
    if not e or e.get("source_sha256_16") != file_hash(SCORE_SRC):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def job_time_ms(local_ms, world, device=None):
    """Whole-job step time: the max of the per-rank times over all ranks."""
    if world <= 1:
        return float(local_ms)
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms):
    """Units processed by all ranks per second (weak scaling: each rank runs
    its own replica of the workload)."""
    return world * units_per_rank / (ms / 1000.0)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# the CPU oracle (baseline leg and the reference arm only)
# ---------------------------------------------------------------------------

def oracle_sample(inp, rows, n_threads=None):
    """Time the oracle as it stands on the given query rows: compression of
    every pool, selection for the rows, expansion of the rows."""
    import oracle as ora
    ora.build()
    wl = inp.wl
    cu = inp.cu_seqlens.numpy() if inp.cu_seqlens.numel() > 2 else None
    kb, gb, qb = W.bits(inp.k), W.bits(inp.gate), W.bits(inp.q)
    t0 = time.perf_counter()
    pk = ora.compress(kb, gb, inp.ape.numpy(), cu, wl.kpool)
    if wl.fp8:
        qc, qs = ora.fp8_rows(qb[rows].reshape(-1, 128))
        pc, ps = ora.fp8_rows(pk)
        # score only the sampled rows: place their codes at their token rows
        qfull = np.zeros((wl.T, wl.H, 128), np.uint8)
        qsf = np.ones((wl.T, wl.H), np.float32)
        qfull[rows] = qc.reshape(len(rows), wl.H, 128)
        qsf[rows] = qs.reshape(len(rows), wl.H)
        ops = ora.Operands(qfull, inp.w.numpy(), pc, qsf, ps)
    else:
        ops = ora.Operands(qb, inp.w.numpy(), pk)
    o = ora.select_rows(ops, cu, wl.kpool, wl.Kp, rows)
    ora.expand_rows(o["sel"], cu, wl.T, wl.kpool, wl.Kp, wl.tail, rows)
    dt = time.perf_counter() - t0
    return dt, ora.num_threads()


def positioned_rows(inp, n, seed=1):
    """Query rows of a positioned workload timed on the oracle: all of them
    when there are at most n, else n drawn without replacement."""
    if inp.Tq <= n:
        return np.arange(inp.Tq, dtype=np.int64)
    g = torch.Generator().manual_seed(seed)
    return torch.sort(torch.randperm(inp.Tq, generator=g)[:n]).values.numpy().astype(np.int64)


def oracle_sample_at(inp, rows, pk=None):
    """Time the oracle as it stands on positioned query rows: for a chunk of
    one sequence, compression of the chunk's pools; then selection and
    expansion of the rows against the pooled keys of their documents."""
    import oracle as ora
    ora.build()
    wl = inp.wl
    cu_k = inp.cu_seqlens.numpy()
    cq, qp = inp.cu_q.numpy(), inp.q_pos.numpy()
    kb, gb = W.bits(inp.k), W.bits(inp.gate)
    if pk is None:
        pk = ora.compress(kb, gb, inp.ape.numpy(), cu_k if len(cu_k) > 2 else None, wl.kpool)
    plan = chunk_compress_plan(inp)
    t0 = time.perf_counter()
    if plan is not None:
        pk = pk.copy()
        pk[plan[1]:] = ora.compress(kb[plan[0]:], gb[plan[0]:], inp.ape.numpy(), None, wl.kpool)
    ops = ora.Operands(W.bits(inp.q), inp.w.numpy(), pk)
    o = ora.select_rows_at(ops, cq, qp, cu_k, wl.kpool, wl.Kp, rows)
    ora.expand_rows_at(o["sel"], cq, qp, cu_k, wl.kpool, wl.Kp, wl.tail, rows)
    dt = time.perf_counter() - t0
    return dt, ora.num_threads()


def l2_policy(in_bytes):
    """How L2 is kept from carrying data between timed steps (timed_loop)."""
    if in_bytes < 512 * 2 ** 20:
        return ("L2 flushed between timed steps (512 MiB write); step time = mean of "
                "per-step CUDA events")
    return "inputs larger than L2 (%.2f GiB read per step)" % (in_bytes / 2 ** 30)


def step_in_bytes(wl, inp):
    """Bytes a timed step of the GPU arm reads from its resident inputs."""
    if wl.queries == "all":
        return sum(x.numel() * x.element_size() for x in (inp.q, inp.k, inp.gate, inp.w))
    nc = positioned_counts(inp)
    cq = inp.cu_q.numpy()
    vis = sum(int(nc[cq[d + 1] - 1]) for d in range(len(cq) - 1) if cq[d + 1] > cq[d])
    b = vis * wl.D * 2 + inp.Tq * wl.H * wl.D * 2 + inp.Tq * wl.H * 4 + inp.Tq * wl.Kp * 8
    plan = chunk_compress_plan(inp)
    return b + ((wl.T - plan[0]) * wl.D * 4 if plan is not None else 0)


def bench_config(wl, inp, world):
    """The "config" object of the JSON line: the same keys and values in the
    GPU arm and in the oracle (reference) arm."""
    par = "replicas" if world > 1 else "single"
    l2 = l2_policy(step_in_bytes(wl, inp))
    if wl.queries == "all":
        return {"workload": wl.name, "desc": wl.desc, "T": wl.T, "H": wl.H, "D": wl.D,
                "kpool": wl.kpool, "index_topk": wl.index_topk, "tail": wl.tail, "fp8": wl.fp8,
                "parallelism": par, "l2": l2}
    plan = chunk_compress_plan(inp)
    return {"workload": wl.name, "desc": wl.desc, "T_keys": wl.T, "T_queries": inp.Tq,
            "H": wl.H, "D": wl.D, "kpool": wl.kpool, "index_topk": wl.index_topk,
            "tail": wl.tail, "fp8": False, "queries": wl.queries,
            "step": ("kpool_compress (the chunk's keys) + " if plan is not None else
                     "pooled-key cache resident; ") +
                    "kpool_score_topk_at + kpool_expand_indices_at",
            "parallelism": par, "l2": l2}


def baseline_rows(wl, n, seed=1):
    g = torch.Generator().manual_seed(seed)
    return torch.sort(torch.randperm(wl.T, generator=g)[:n]).values.numpy().astype(np.int64)


# ---------------------------------------------------------------------------

def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = W.make_inputs(wl)
    if wl.queries != "all":
        import oracle as ora
        ora.build()
        cu_k = inp.cu_seqlens.numpy()
        pk = ora.compress(W.bits(inp.k), W.bits(inp.gate), inp.ape.numpy(),
                          cu_k if len(cu_k) > 2 else None, wl.kpool)
        rows = positioned_rows(inp, args.ref_rows)
        sample_fn = lambda r: oracle_sample_at(inp, r, pk)   # noqa: E731
        sample = ("%d query rows of %s per step (selection and expansion of the rows over the "
                  "pooled-key cache%s)" % (len(rows), wl.name,
                                           "; compression of the chunk's pools"
                                           if chunk_compress_plan(inp) else ""))
    else:
        rows = baseline_rows(wl, args.ref_rows)
        sample_fn = lambda r: oracle_sample(inp, r)   # noqa: E731
        sample = ("%d uniformly drawn query rows of %s per step (compression of all %d pools, "
                  "selection and expansion of the rows)" % (len(rows), wl.name,
                                                            wl.T // wl.kpool))
    for _ in range(args.warmup):
        sample_fn(rows[: max(1, len(rows) // 8)])
    times = []
    cores = 1
    for _ in range(args.steps):
        dt, cores = sample_fn(rows)
        times.append(dt)
    ms = 1000.0 * sum(times) / len(times)
    value = len(rows) / (ms / 1000.0)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(wl, inp, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def timed_loop(step, n_seg, steps, stream, in_bytes, local, barrier):
    """Time ``steps`` calls of ``step(events)`` with CUDA events on ``stream``.

    ``step`` records ``n_seg + 1`` events (segment boundaries).  When the
    bytes a step reads are below 512 MiB, L2 (129 MB) is flushed before
    every step by writing a 512 MiB buffer and the step time is the mean of
    the per-step events; otherwise it is the whole region / steps.  Returns
    (ms per step, [mean ms per segment], clocks, note on L2)."""
    dev = torch.device("cuda", local)
    flush = None
    if in_bytes < 512 * 2 ** 20:
        flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(local)
    sampler.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_seg + 1)]
           for _ in range(steps)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    e0.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        step(evs[i])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    if flush is None:
        ms_step = e0.elapsed_time(e1) / steps
    else:
        ms_step = statistics.mean(e[0].elapsed_time(e[n_seg]) for e in evs)
    note = l2_policy(in_bytes)
    segs = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j in range(n_seg)]
    return ms_step, segs, clocks, note


def run_mla(args):
    """The sparse attention that consumes the selection, fused with the
    expansion (kpool_sparse_mla_fwd_pools): one call per step over the whole
    workload, on the indexer's own selection (computed once, untimed).
    Tensor-bound: 4 * H * Dc FLOPs per (query, listed token) pair (scores and
    output), counted over the valid listed tokens."""
    wl = W.MLA_WORKLOADS[args.workload]
    if args.T is not None:
        from dataclasses import replace
        if wl.n_docs > 1:
            raise ValueError("--T applies to single-sequence workloads only")
        wl = replace(wl, T=args.T, name="%s_T%d" % (wl.name, args.T))
    world, rank, local = dist_env()
    if args.impl == "reference":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm covers the indexer "
                          "workloads; the sparse attention reports its oracle sample as "
                          "cpu_baseline"}), flush=True)
        return 0
    torch.cuda.set_device(local)
    import sparse_attention_kpool_compress_gb300 as K
    from sparse_attention_kpool_compress_gb300 import binding as B
    dev = torch.device("cuda", local)
    inp = W.make_inputs(wl, seed=wl.seed)
    cu_d = cp_d = P = None
    if wl.n_docs > 1:
        cp_h, P = K.kpool_num_pools(inp.cu_seqlens, wl.T, wl.kpool)
        cu_d, cp_d = inp.cu_seqlens.to(dev), cp_h.to(dev)
    _, pool_idx, _ = K.kpool_indexer_forward(inp.q.to(dev), inp.k.to(dev), inp.gate.to(dev),
                                             inp.ape.to(dev), inp.w.to(dev), wl.kpool,
                                             wl.index_topk, wl.tail, cu_d, cp_d, P)
    mi = W.make_mla_inputs(wl.T, seed=wl.seed)
    q, kv = mi.q.to(dev), mi.kv.to(dev)
    T, H, Dc = q.shape
    o = torch.empty(T, H, Dc, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    ws = torch.zeros(K.kpool_sparse_mla_workspace_size(), dtype=torch.uint8, device=dev)
    # listed tokens per row: the selected pools' tokens plus the tail
    if cu_d is None:
        tau = torch.arange(T, device=dev)
    else:
        starts = inp.cu_seqlens.to(dev).long()
        doc = torch.searchsorted(starts[1:], torch.arange(T, device=dev), right=True)
        tau = torch.arange(T, device=dev) - starts[doc]
    n_tok = (pool_idx >= 0).sum(dim=1).long() * wl.kpool
    if wl.tail:
        n_tok += (tau + 1) % wl.kpool
    pairs = int(n_tok.sum().item())
    flops = 4.0 * H * Dc * pairs
    L = B._lib
    sp = B._stream(dev)
    stream = torch.cuda.current_stream(dev)
    n_docs = wl.n_docs if cu_d is not None else 1

    def call():
        rc = L.kpool_sparse_mla_fwd_pools(B._ptr(q), B._ptr(kv), B._ptr(pool_idx), B._ptr(cu_d),
                                          B._ptr(cp_d), n_docs, T, H, Dc, wl.kpool,
                                          wl.index_topk, int(wl.tail), ctypes.c_float(mi.scale),
                                          B._ptr(o), B._ptr(lse), B._ptr(ws), ws.numel(), sp)
        if rc != 0:
            raise B.KPoolError(rc, "kpool_sparse_mla_fwd_pools")

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        call()
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if K.kpool_read_status(ws) != 0:
        raise RuntimeError("device status after warm-up")
    in_bytes = q.numel() * 2 + kv.numel() * 2 + pool_idx.numel() * 4
    ms, _, clocks, l2_note = timed_loop(step, 1, args.steps, stream, in_bytes, local,
                                        lambda: None)
    peaks, peak_src = load_peaks()
    tflops = flops / ms / 1e9
    e2e = None
    if not args.no_e2e:
        hq, hkv = mi.q.pin_memory(), mi.kv.pin_memory()
        hsel = pool_idx.cpu().pin_memory()
        ho = torch.empty(T, H, Dc, dtype=torch.bfloat16).pin_memory()
        hl = torch.empty(T, H, dtype=torch.float32).pin_memory()

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            kv.copy_(hkv, non_blocking=True)
            pool_idx.copy_(hsel, non_blocking=True)
            call()
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(5):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        me = a0.elapsed_time(a1) / 5
        e2e = {"value": T / (me / 1000.0), "unit": "queries/s", "ms_per_step": me, "steps": 5,
               "h2d_bytes_per_step": (hq.numel() + hkv.numel()) * 2 + hsel.numel() * 4,
               "d2h_bytes_per_step": ho.numel() * 2 + hl.numel() * 4}
    cpu = None
    if not args.no_cpu_baseline:
        import oracle as ora
        ora.build()
        rows = W.sample_rows(T, n_sample=4, edge=0, seed=1).numpy()
        rows = rows[rows >= T // 2][:4]
        sel = pool_idx.cpu().numpy()[rows]
        tok = ora.expand_rows(sel, inp.cu_seqlens.numpy() if cu_d is not None else None, T,
                              wl.kpool, wl.Kp, wl.tail, rows)
        t0 = time.time()
        ora.sparse_attn(W.bits(mi.q), W.bits(mi.kv), tok, mi.scale, rows)
        dt = time.time() - t0
        cpu = {"value": len(rows) / dt, "unit": "queries/s", "cores": ora.num_threads(),
               "kind": "oracle", "sample": "%d query rows of the second half (%d listed tokens "
               "each at most), fp64 C" % (len(rows), wl.Kp * wl.kpool + wl.kpool - 1)}
    line = {
        "metric": "Sparse attention over the KPool selection (absorbed NoPE MLA, fused "
                  "expansion), queries/s", "value": T / (ms / 1000.0),
        "unit": "queries/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "desc": wl.desc, "T": T, "heads": H, "latent": Dc,
                   "kpool": wl.kpool, "index_topk": wl.index_topk, "tail": wl.tail,
                   "n_docs": wl.n_docs, "parallelism": "single", "l2": l2_note},
        "e2e": e2e, "gpu_launches": args.steps,
        "roofline": {"bound": "tensor", "kernel": "sparse_mla_kernel", "achieved": tflops,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tflops / peaks["bf16_tflops"],
                     "frac_of_sustained": tflops / peaks["bf16_tflops_sustained"],
                     "traffic": None, "peak_source": "bf16 burst (%s)" % peak_src,
                     "algorithmic_flops_per_launch": flops, "listed_tokens": pairs},
        "cpu_baseline": cpu, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_128k",
                    choices=sorted(W.WORKLOADS) + sorted(W.PROJECTION_WORKLOADS) +
                    sorted(W.MLA_WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--baseline-rows", type=int, default=3584)
    ap.add_argument("--e2e-chunk-rows", type=int, default=0,
                    help="query rows per chunk of the end-to-end pass (0 = the library's default)")
    ap.add_argument("--ref-rows", type=int, default=48)
    ap.add_argument("--replicas", action="store_true",
                    help="N > 1: every rank runs the whole workload (weak scaling) instead of "
                         "scoring its share of the query rows (strong scaling)")
    ap.add_argument("--no-fp8-peak", action="store_true",
                    help="FP8 workloads: skip measuring the E4M3 peak (profiling runs); the "
                         "roofline then uses 2 x the BF16 burst peak, and says so")
    ap.add_argument("--T", type=int, default=None,
                    help="same recipe at another token count (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warmup raised to 3 (minimum)", file=sys.stderr)
        args.warmup = 3
    if args.workload in W.PROJECTION_WORKLOADS:
        return run_projection(args)
    if args.workload in W.MLA_WORKLOADS:
        return run_mla(args)
    wl = W.WORKLOADS[args.workload]
    if args.T is not None:
        from dataclasses import replace
        wl = replace(wl, T=args.T, name="%s_T%d" % (wl.name, args.T))
    if args.impl == "reference":
        return run_reference(args, wl)

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import sparse_attention_kpool_compress_gb300 as K

    dev = torch.device("cuda", local)
    inp = W.make_inputs(wl)
    if wl.queries != "all":
        return run_positioned(args, wl, inp, K, dev, world, rank, local)
    if world > 1 and not args.replicas:
        return run_sharded(args, wl, inp, dev, world, rank, local)
    T, H, D, kp, topk, Kp = wl.T, wl.H, wl.D, wl.kpool, wl.index_topk, wl.Kp
    multi = inp.cu_seqlens.numel() > 2
    if multi:
        cu_pools_h, P = K.kpool_num_pools(inp.cu_seqlens, T, kp)
        cu = inp.cu_seqlens.to(dev)
        cp = cu_pools_h.to(dev)
        n_docs = inp.cu_seqlens.numel() - 1
    else:
        P, cu, cp, n_docs = T // kp, None, None, 1

    q = inp.q.to(dev)
    k = inp.k.to(dev)
    gate = inp.gate.to(dev)
    ape = inp.ape.to(dev)
    w = inp.w.to(dev)
    pk = torch.empty(P, D, dtype=torch.bfloat16, device=dev)
    pool_idx = torch.empty(T, Kp, dtype=torch.int32, device=dev)
    pool_score = torch.empty(T, Kp, dtype=torch.float32, device=dev)
    Wd = Kp * kp + kp - 1
    tok = torch.empty(T, Wd, dtype=torch.int32, device=dev)
    ws = K.new_workspace(T, H, n_docs, dev)
    if wl.fp8:
        pk8 = torch.empty(P, D, dtype=torch.uint8, device=dev)
        pks = torch.empty(P, dtype=torch.float32, device=dev)
        q8 = torch.empty(T, H, D, dtype=torch.uint8, device=dev)
        qs = torch.empty(T, H, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    from sparse_attention_kpool_compress_gb300 import binding as B
    L = B._lib
    sp = B._stream(dev)

    def chk(rc, name):
        if rc != 0:
            raise B.KPoolError(rc, name)

    def step(ev=None):
        # segments: compress | quantize q (FP8 mode; empty otherwise) | score | expand
        if ev is not None:
            ev[0].record(stream)
        if wl.fp8:
            chk(L.kpool_compress(B._ptr(k), B._ptr(gate), B._ptr(ape), B._ptr(cu), B._ptr(cp),
                                 n_docs, T, D, kp, P, B._ptr(pk), B._ptr(pk8), B._ptr(pks), sp),
                "kpool_compress")
            if ev is not None:
                ev[1].record(stream)
            chk(L.kpool_quantize_fp8(B._ptr(q), T * H, D, B._ptr(q8), B._ptr(qs), sp),
                "kpool_quantize_fp8")
        else:
            chk(L.kpool_compress(B._ptr(k), B._ptr(gate), B._ptr(ape), B._ptr(cu), B._ptr(cp),
                                 n_docs, T, D, kp, P, B._ptr(pk), None, None, sp),
                "kpool_compress")
            if ev is not None:
                ev[1].record(stream)
        if ev is not None:
            ev[2].record(stream)
        if wl.fp8:
            chk(L.kpool_score_topk(B._ptr(q8), B._ptr(qs), B._ptr(w), B._ptr(pk8), B._ptr(pks),
                                   B._ptr(cu), B._ptr(cp), n_docs, T, P, H, D, kp, topk, 1,
                                   B._ptr(pool_idx), B._ptr(pool_score), B._ptr(ws), ws.numel(),
                                   sp), "kpool_score_topk")
        else:
            chk(L.kpool_score_topk(B._ptr(q), None, B._ptr(w), B._ptr(pk), None, B._ptr(cu),
                                   B._ptr(cp), n_docs, T, P, H, D, kp, topk, 0, B._ptr(pool_idx),
                                   B._ptr(pool_score), B._ptr(ws), ws.numel(), sp),
                "kpool_score_topk")
        if ev is not None:
            ev[3].record(stream)
        chk(L.kpool_expand_indices(B._ptr(pool_idx), B._ptr(cu), B._ptr(cp), n_docs, T, kp, topk,
                                   int(wl.tail), B._ptr(tok), sp), "kpool_expand_indices")
        if ev is not None:
            ev[4].record(stream)

    launches_per_step = 1 + (1 if wl.fp8 else 0) + 2 + 1

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = K.kpool_read_status(ws)
    if status != 0:
        raise RuntimeError("device status %d after warm-up" % status)

    in_bytes = sum(x.numel() * x.element_size() for x in (q, k, gate, w))
    ms_step, (t_compress, t_quant, t_score, t_expand), clocks, l2_note = timed_loop(
        step, 4, args.steps, stream, in_bytes, local, barrier)
    ms_step = job_time_ms(ms_step, world, dev)
    status = K.kpool_read_status(ws)
    if status != 0:
        raise RuntimeError("device status %d after the timed steps" % status)

    # ---- end to end through the C ABI from pinned host memory ---------------
    # kpool_indexer_forward_host: host inputs in, host token indices out, the
    # copies of every step inside the timed region (overlapped with the kernels)
    e2e = None
    if not args.no_e2e:
        del q, k, gate, w, pool_idx, pool_score, tok, ws
        if wl.fp8:
            del pk8, pks, q8, qs
        torch.cuda.empty_cache()
        hq, hk, hg, ha, hw = (x.pin_memory() for x in (inp.q, inp.k, inp.gate, inp.ape, inp.w))
        hcu = inp.cu_seqlens if multi else None
        htok = torch.empty(T, Wd, dtype=torch.int32).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hg, ha, hw))
        h2d += hcu.numel() * 4 if multi else 0
        d2h = htok.numel() * htok.element_size()
        scratch = torch.empty(K.kpool_indexer_forward_host_scratch_size(
            T, H, D, kp, topk, hcu, wl.fp8, args.e2e_chunk_rows), dtype=torch.uint8, device=dev)

        def e2e_step():
            K.kpool_indexer_forward_host(hq, hk, hg, ha, hw, kp, topk, wl.tail, hcu, wl.fp8,
                                         args.e2e_chunk_rows, scratch=scratch, out=htok,
                                         device=dev)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if K.kpool_read_status(scratch) != 0:
            raise RuntimeError("device status after the end-to-end warm-up")
        barrier()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        n_e2e = max(2, min(args.steps, 5))
        for _ in range(n_e2e):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_e2e = a0.elapsed_time(a1) / n_e2e
        ms_e2e = job_time_ms(ms_e2e, world, dev)
        e2e = {"value": whole_job_rate(T, world, ms_e2e), "unit": UNIT, "ms_per_step": ms_e2e,
               "steps": n_e2e, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "kpool_indexer_forward_host (C ABI, pinned host buffers, copies "
                      "overlapped with the kernels in query chunks of up to %d rows)"
                      % (args.e2e_chunk_rows or 16384)}
        del hq, hk, hg, ha, hw, htok, scratch

    # ---- roofline of the dominant kernel ---------------------------------
    peaks, peak_src = load_peaks()
    pairs = sum_floor_pairs(inp.cu_seqlens, kp)
    flops = 2.0 * H * D * pairs
    achieved = flops / (t_score / 1000.0) / 1e12
    # The scoring kernel runs as one launch of tens of ms between other
    # kernels, not as a seconds-long GEMM loop under the power cap: its
    # denominator is the burst peak of its own operand type (FP8: measured in
    # this run with the same recipe as the BF16 peaks).
    fp8_peak = measure_fp8_peak(dev) if wl.fp8 and not args.no_fp8_peak else None
    if fp8_peak is not None:
        peak = fp8_peak["fp8_tflops"]
        peak_note = "fp8 e4m3 burst, measured in this run: " + fp8_peak["how"]
        sustained = fp8_peak["fp8_tflops_sustained"]
    elif wl.fp8:
        peak = 2.0 * peaks["bf16_tflops"]
        peak_note = "2 x bf16 burst (nominal E4M3/BF16 ratio; FP8 peak not measured in this run)"
        sustained = 2.0 * peaks["bf16_tflops_sustained"]
    else:
        peak = peaks["bf16_tflops"]
        peak_note = "bf16 burst (%s, MEASURED_PEAKS.json)" % peak_src
        sustained = peaks["bf16_tflops_sustained"]
    roofline = {"bound": "tensor", "kernel": "kpool_score_topk", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": recorded_traffic("kpool_score_topk", wl.name),
                "peak_source": peak_note, "peak_sustained": sustained,
                "frac_of_sustained": achieved / sustained,
                "algorithmic_flops_per_launch": flops, "causal_pairs": pairs,
                "ms_per_launch": t_score}
    if fp8_peak is not None:
        roofline["fp8_peak_measurement"] = fp8_peak
    comp_bytes = T * D * 2 * 2 + P * D * 2 + (P * (D + 4) if wl.fp8 else 0)
    side = {"compress_ms": t_compress, "compress_gbs": comp_bytes / (t_compress / 1000.0) / 1e9,
            "compress_frac_hbm": comp_bytes / (t_compress / 1000.0) / 1e9 / peaks["hbm_gbs"],
            "quantize_q_ms": t_quant if wl.fp8 else None,
            "quantize_q_gbs": (T * H * (D * 2 + D + 4)) / (t_quant / 1000.0) / 1e9
            if wl.fp8 else None,
            "expand_ms": t_expand,
            "expand_gbs": (T * Kp * 4 + T * Wd * 4) / (t_expand / 1000.0) / 1e9,
            "score_topk_ms": t_score, "score_queries_per_s": T / (t_score / 1000.0)}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rows = baseline_rows(wl, args.baseline_rows)
        dt, cores = oracle_sample(inp, rows)
        cpu = {"value": len(rows) / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "%d uniformly drawn query rows of %s (compression of all pools, "
                         "selection and expansion of those rows), %.1f s" % (len(rows), wl.name, dt)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": whole_job_rate(T, world, ms_step), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8-e4m3" if wl.fp8 else "bf16", "data": "synthetic",
            "config": bench_config(wl, inp, world),
            "scoring_tflops": achieved,
            "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks, "kernels": side,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def positioned_counts(inp):
    """Per query row: complete causal pools n_c and the document's pool count."""
    wl = inp.wl
    cu_k = inp.cu_seqlens.numpy().astype(np.int64)
    cq = inp.cu_q.numpy().astype(np.int64)
    qp = inp.q_pos.numpy().astype(np.int64)
    nc = np.empty(inp.Tq, np.int64)
    for d in range(len(qp)):
        tau = qp[d] + np.arange(cq[d + 1] - cq[d])
        nc[cq[d]:cq[d + 1]] = np.minimum((tau + 1) // wl.kpool, (cu_k[d + 1] - cu_k[d]) // wl.kpool)
    return nc


def chunk_compress_plan(inp):
    """A chunked prefill of one sequence whose chunk starts on a pool boundary
    re-compresses the chunk's keys into the pooled-key cache each step:
    (first key token, first pool).  None when the step compresses nothing
    (decode: the pooled-key cache is resident)."""
    wl = inp.wl
    if not wl.queries.startswith("chunk:") or inp.cu_seqlens.numel() != 2:
        return None
    p0 = int(inp.q_pos[0])
    if p0 % wl.kpool:
        return None
    return p0, p0 // wl.kpool


def run_positioned(args, wl, inp, K, dev, world, rank, local):
    """Decode and chunked-prefill steps: kpool_score_topk_at and
    kpool_expand_indices_at over a resident pooled-key cache (plus, for a
    chunk, the compression of the chunk's own keys into that cache)."""
    T, H, D, kp, topk, Kp = wl.T, wl.H, wl.D, wl.kpool, wl.index_topk, wl.Kp
    Tq = inp.Tq
    n_docs = inp.cu_seqlens.numel() - 1
    cu_pools_h, P = K.kpool_num_pools(inp.cu_seqlens, T, kp)
    cu_k, cp = inp.cu_seqlens.to(dev), cu_pools_h.to(dev)
    cq, qp = inp.cu_q.to(dev), inp.q_pos.to(dev)
    q, w = inp.q.to(dev), inp.w.to(dev)
    k, gate, ape = inp.k.to(dev), inp.gate.to(dev), inp.ape.to(dev)
    # the pooled-key cache: every complete pool of every document
    pk = K.kpool_compress(k, gate, ape, kp, cu_k if n_docs > 1 else None,
                          cp if n_docs > 1 else None, P)
    plan = chunk_compress_plan(inp)
    if plan is not None:
        kc, gc = k[plan[0]:], gate[plan[0]:]
        pkc = pk[plan[1]:]
    else:
        del k, gate
    pool_idx = torch.empty(Tq, Kp, dtype=torch.int32, device=dev)
    pool_score = torch.empty(Tq, Kp, dtype=torch.float32, device=dev)
    Wd = Kp * kp + kp - 1
    tok = torch.empty(Tq, Wd, dtype=torch.int32, device=dev)
    ws = K.new_workspace(Tq, H, n_docs, dev, kp, topk)
    stream = torch.cuda.current_stream(dev)
    from sparse_attention_kpool_compress_gb300 import binding as B
    L = B._lib
    sp = B._stream(dev)

    def chk(rc, name):
        if rc != 0:
            raise B.KPoolError(rc, name)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if plan is not None:
            chk(L.kpool_compress(B._ptr(kc), B._ptr(gc), B._ptr(ape), None, None, 1,
                                 kc.shape[0], D, kp, kc.shape[0] // kp, B._ptr(pkc), None, None,
                                 sp), "kpool_compress")
        if ev is not None:
            ev[1].record(stream)
        chk(L.kpool_score_topk_at(B._ptr(q), None, B._ptr(w), B._ptr(pk), None, B._ptr(cq),
                                  B._ptr(qp), B._ptr(cp), n_docs, Tq, P, H, D, kp, topk, 0,
                                  B._ptr(pool_idx), B._ptr(pool_score), B._ptr(ws), ws.numel(),
                                  sp), "kpool_score_topk_at")
        if ev is not None:
            ev[2].record(stream)
        chk(L.kpool_expand_indices_at(B._ptr(pool_idx), B._ptr(cq), B._ptr(qp), B._ptr(cu_k),
                                      B._ptr(cp), n_docs, Tq, kp, topk, int(wl.tail),
                                      B._ptr(tok), sp), "kpool_expand_indices_at")
        if ev is not None:
            ev[3].record(stream)

    launches_per_step = (1 if plan is not None else 0) + 2 + 1

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if K.kpool_read_status(ws) != 0:
        raise RuntimeError("device status %d after warm-up" % K.kpool_read_status(ws))
    nc = positioned_counts(inp)
    # algorithmic bytes of kpool_score_topk_at: each document's visible pooled
    # keys once, the queries, head weights and the selected (index, score) rows
    vis = np.zeros(n_docs, np.int64)
    cqh = inp.cu_q.numpy()
    for d in range(n_docs):
        if cqh[d + 1] > cqh[d]:
            vis[d] = nc[cqh[d + 1] - 1]
    score_bytes = int(vis.sum()) * D * 2 + Tq * H * D * 2 + Tq * H * 4 + Tq * Kp * 8
    in_bytes = score_bytes + ((T - plan[0]) * D * 4 if plan is not None else 0)
    ms_step, (t_compress, t_score, t_expand), clocks, l2_note = timed_loop(
        step, 3, args.steps, stream, in_bytes, local, barrier)
    ms_step = job_time_ms(ms_step, world, dev)
    if K.kpool_read_status(ws) != 0:
        raise RuntimeError("device status %d after the timed steps" % K.kpool_read_status(ws))

    # ---- end to end through the public API from pinned host memory --------
    e2e = None
    if not args.no_e2e:
        hq, hw = inp.q.pin_memory(), inp.w.pin_memory()
        hsrc = [hq, hw]
        if plan is not None:
            hk, hg = inp.k[plan[0]:].pin_memory(), inp.gate[plan[0]:].pin_memory()
            hsrc += [hk, hg]
        htok = torch.empty(Tq, Wd, dtype=torch.int32).pin_memory()
        dsts = [torch.empty_like(x, device=dev) for x in hsrc]
        h2d = sum(x.numel() * x.element_size() for x in hsrc)
        d2h = htok.numel() * htok.element_size()

        def e2e_step():
            for d_, h_ in zip(dsts, hsrc):
                d_.copy_(h_, non_blocking=True)
            if plan is not None:
                K.kpool_compress(dsts[2], dsts[3], ape, kp, out=pkc)
            idx, _ = K.kpool_score_topk_at(dsts[0], dsts[1], pk, kp, topk, cq, qp, cp,
                                           workspace=ws)
            tk = K.kpool_expand_indices_at(idx, kp, topk, cq, qp, cu_k, cp, wl.tail)
            htok.copy_(tk, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        n_e2e = max(2, min(args.steps, 10))
        for _ in range(n_e2e):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_e2e = job_time_ms(a0.elapsed_time(a1) / n_e2e, world, dev)
        e2e = {"value": whole_job_rate(Tq, world, ms_e2e), "unit": UNIT, "ms_per_step": ms_e2e,
               "steps": n_e2e, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    peaks, peak_src = load_peaks()
    flops = 2.0 * H * D * float(nc.sum())
    tflops = flops / (t_score / 1000.0) / 1e12
    gbs = score_bytes / (t_score / 1000.0) / 1e9
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = score_bytes / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        roofline = {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"],
                    "peak_source": "bf16 burst (%s, MEASURED_PEAKS.json)" % peak_src,
                    "frac_of_sustained": tflops / peaks["bf16_tflops_sustained"]}
    else:
        roofline = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"], "peak_source": "hbm copy (%s)" % peak_src}
    roofline.update({"kernel": "kpool_score_topk_at", "traffic": recorded_traffic(
        "kpool_score_topk_at", wl.name), "algorithmic_flops_per_launch": flops,
        "algorithmic_bytes_per_launch": score_bytes, "scoring_tflops": tflops,
        "scoring_gbs": gbs, "causal_pairs": int(nc.sum()), "ms_per_launch": t_score,
        "roofline_ms": max(t_tensor, t_hbm) * 1000.0})
    side = {"compress_ms": t_compress if plan is not None else None,
            "expand_ms": t_expand,
            "expand_gbs": (Tq * Kp * 4 + Tq * Wd * 4) / (t_expand / 1000.0) / 1e9,
            "score_topk_ms": t_score, "score_queries_per_s": Tq / (t_score / 1000.0)}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rows = positioned_rows(inp, args.baseline_rows)
        dt, cores = oracle_sample_at(inp, rows)
        cpu = {"value": len(rows) / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "%d query rows of %s (selection and expansion of those rows%s), %.1f s"
                         % (len(rows), wl.name, ", compression of the chunk's pools"
                            if plan is not None else "", dt)}
    if rank == 0:
        line = {
            "metric": METRIC, "value": whole_job_rate(Tq, world, ms_step), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": bench_config(wl, inp, world),
            "scoring_tflops": tflops,
            "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks, "kernels": side,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_sharded(args, wl, inp, dev, world, rank, local):
    """N > 1 ranks share one workload (strong scaling): each holds the rows of
    its shard (zigzag blocks of one sequence, or whole packed documents) and
    runs the query-sharded pass (sparse_attention_kpool_compress_gb300.sharding);
    one sequence exchanges pooled keys with an NCCL all-gather.  A step is one
    whole pass of every rank; its time is the max over ranks, and the job
    processes the workload's T queries per step."""
    import torch.distributed as dist
    from sparse_attention_kpool_compress_gb300 import sharding as S
    cu = inp.cu_seqlens.tolist() if inp.cu_seqlens.numel() > 2 else None
    plan = S.plan_shards(wl.T, world, rank, wl.kpool, cu)
    q, k, gate, w = (S.shard_rows(x, plan).to(dev) for x in (inp.q, inp.k, inp.gate, inp.w))
    ape = inp.ape.to(dev)
    idx = S.ShardedIndexer(plan, wl.index_topk, wl.tail, wl.fp8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        idx.forward(q, k, gate, ape, w)
        if ev is not None:
            ev[1].record(stream)

    def barrier():
        dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    in_bytes = sum(x.numel() * x.element_size() for x in (q, k, gate, w))
    ms_step, _, clocks, _ = timed_loop(step, 1, args.steps, stream, in_bytes, local, barrier)
    ms_step = job_time_ms(ms_step, world, dev)

    e2e = None
    if not args.no_e2e:
        hsrc = [x.cpu().pin_memory() for x in (q, k, gate, w)]
        dsts = [torch.empty_like(x) for x in (q, k, gate, w)]
        Wd = wl.Kp * wl.kpool + wl.kpool - 1
        htok = torch.empty(plan.local_rows, Wd, dtype=torch.int32).pin_memory()

        def e2e_step():
            for d_, h_ in zip(dsts, hsrc):
                d_.copy_(h_, non_blocking=True)
            tok = idx.forward(dsts[0], dsts[1], dsts[2], ape, dsts[3])
            htok.copy_(tok, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(2, min(args.steps, 5))
        a0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_e2e = job_time_ms(a0.elapsed_time(a1) / n_e2e, world, dev)
        e2e = {"value": wl.T / (ms_e2e / 1000.0), "unit": UNIT, "ms_per_step": ms_e2e,
               "steps": n_e2e, "h2d_bytes_per_step": sum(x.numel() * x.element_size()
                                                          for x in hsrc),
               "d2h_bytes_per_step": htok.numel() * 4,
               "api": "ShardedIndexer.forward per rank (rank 0's bytes)"}

    peaks, peak_src = load_peaks()
    flops = 2.0 * wl.H * wl.D * sum_floor_pairs(inp.cu_seqlens, wl.kpool)
    tflops = flops / (ms_step / 1000.0) / 1e12
    peak = peaks["bf16_tflops"] * (2 if wl.fp8 else 1) * world
    if rank == 0:
        line = {
            "metric": METRIC, "value": wl.T / (ms_step / 1000.0), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
            "dtype": "fp8-e4m3" if wl.fp8 else "bf16", "data": "synthetic",
            "config": dict(bench_config(wl, inp, 1),
                           parallelism="%s-%d" % (plan.layout, world)),
            "scoring_tflops": tflops, "e2e": e2e,
            # rank 0's own kernels: compress, [FP8 q cast], and per scoring call
            # the schedule, scoring and expansion kernels
            "gpu_launches": args.steps * (1 + int(wl.fp8) + 3 * (
                len(plan.segments) if plan.layout == "zigzag" else int(bool(plan.segments)))),
            "roofline": {"bound": "tensor", "kernel": "whole sharded step", "achieved": tflops,
                         "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                         "traffic": None,
                         "peak_source": "%d x %s burst (%s)" % (world, "2 x bf16" if wl.fp8
                                                                else "bf16", peak_src)},
            "cpu_baseline": None, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    dist.destroy_process_group()
    return 0


def run_projection(args):
    """The key path fused with compression (kpool_project_compress): hidden
    states to pooled keys in one kernel.  HBM-bound (the hidden states are read
    once); the roofline counts x, the weights and the pooled keys written."""
    cfg = dict(W.PROJECTION_WORKLOADS[args.workload])
    if args.T is not None:
        cfg["T"] = args.T
    T, hidden, D, kp = cfg["T"], cfg["hidden"], cfg["D"], cfg["kpool"]
    world, rank, local = dist_env()
    if args.impl == "reference":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm covers the indexer "
                          "workloads; the projection has no CPU baseline line"}), flush=True)
        return 0
    torch.cuda.set_device(local)
    import sparse_attention_kpool_compress_gb300 as K
    dev = torch.device("cuda", local)
    pi = W.make_projection_inputs(T, hidden, D, kp)
    x, w = pi.x.to(dev), pi.w_kg.to(dev)
    gamma, beta, ape = pi.gamma.to(dev), pi.beta.to(dev), pi.ape.to(dev)
    P = T // kp
    pk = torch.empty(P, D, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    from sparse_attention_kpool_compress_gb300 import binding as B
    L = B._lib
    sp = B._stream(dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        rc = L.kpool_project_compress(B._ptr(x), B._ptr(w), B._ptr(gamma), B._ptr(beta),
                                      ctypes.c_float(pi.eps), B._ptr(ape), None, None, 1, T,
                                      hidden, D, kp, P, B._ptr(pk), None, None, B._ptr(ws),
                                      ws.numel(), sp)
        if rc != 0:
            raise B.KPoolError(rc, "kpool_project_compress")
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if K.kpool_read_status(ws) != 0:
        raise RuntimeError("device status after warm-up")
    in_bytes = x.numel() * 2 + w.numel() * 2
    ms, _, clocks, l2_note = timed_loop(step, 1, args.steps, stream, in_bytes, local,
                                        lambda: None)
    peaks, peak_src = load_peaks()
    alg = T * hidden * 2 + 2 * D * hidden * 2 + P * D * 2
    gbs = alg / (ms / 1000.0) / 1e9
    flops = 2.0 * T * hidden * 2 * D
    e2e = None
    if not args.no_e2e:
        hx = pi.x.pin_memory()
        hpk = torch.empty(P, D, dtype=torch.bfloat16).pin_memory()
        xd = torch.empty_like(x)

        def e2e_step():
            xd.copy_(hx, non_blocking=True)
            K.kpool_project_compress(xd, w, gamma, beta, pi.eps, ape, kp, workspace=ws)
            hpk.copy_(pk, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(5):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        me = a0.elapsed_time(a1) / 5
        e2e = {"value": T / (me / 1000.0), "unit": "tokens/s", "ms_per_step": me, "steps": 5,
               "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hpk.numel() * 2}
    line = {
        "metric": "KPool key path fused with compression, tokens/s", "value": T / (ms / 1000.0),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "desc": cfg["desc"], "T": T, "hidden": hidden,
                   "D": D, "kpool": kp, "parallelism": "single", "l2": l2_note},
        "e2e": e2e, "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "kernel": "kpool_project_compress", "achieved": gbs,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "traffic": None, "peak_source": "hbm copy (%s)" % peak_src,
                     "algorithmic_bytes_per_launch": alg, "tensor_tflops": flops / ms / 1e9},
        "cpu_baseline": None, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def sum_floor_pairs(cu_seqlens, kp):
    cs = [int(x) for x in cu_seqlens]
    return sum(sum_floor(b - a, kp) for a, b in zip(cs[:-1], cs[1:]))


if __name__ == "__main__":
    sys.exit(main())
