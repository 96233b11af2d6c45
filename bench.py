#!/usr/bin/env python3
"""Benchmark of the attention forward on GB300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2] [--impl reference]

A step is one attention forward (the whole hot path: one launch of the
persistent kernel) over the workload's synthetic batch. The default workload
is the bf16 B=4 H=16 Sq=Sk=8192 D=128 non-causal forward. Inputs are larger
than L2 (384 MiB of Q/K/V), so no L2 flush runs between steps.

``value`` is TFLOP/s (4*B*H*Sq*Sk*D, halved for causal) with inputs resident
in HBM, timed with CUDA events on the launching stream; ``e2e`` is the same
metric through the C ABI with the inputs copied from pinned host memory and
the outputs copied back inside the timed region. ``roofline`` compares the
kernel with the measured dense bf16 tensor-core peak; ``cpu_baseline`` times
the fp64 oracle on the host cores on a bounded sample of the same workload.

Paged workloads (``--workload p1`` / ``p2``): one ``fa_fwd_paged`` call over a
K/V cache of shuffled 16-key pages (p2, decode, with automatic key ranges and
an HBM roofline: one read of the cache).

Backward workloads (``--workload b1`` / ``b2``): a step is one ``fa_bwd``
call (row constants, dK/dV kernel, dQ kernel) for O, LSE from one forward run
before timing; the metric counts 2.5x the forward's FLOPs (the five matrix
products of the gradient) and ``e2e`` copies Q, K, V, O, dO, LSE in and dQ,
dK, dV out every step.

``--impl reference`` times the oracle itself as the reference arm (each step
a bounded sample of the workload) and prints the same line with
"impl": "reference".

With N > 1 (torchrun, one rank per GPU) every rank runs its own copy of the
workload (weak scaling: the forward shards over batch x heads with no data
exchange); ``value`` = FLOPs of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s on 1 GB300 and % of measured dense tensor-core ceiling"
METRIC_BWD = "attention bwd TFLOP/s (2.5x forward FLOPs) on 1 GB300 and % of measured dense tensor-core ceiling"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def csrc_digest() -> str:
    from exact_attention_forward_tiled_gb300 import build as fb
    h = hashlib.sha256()
    for d in (fb.CSRC, fb.INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = csrc_digest()
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(tok.split("=", 1) for tok in line.split())
            if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("csrc") == digest:
                return float(kv["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            self.out = ""
            return
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        top = max(r[0] for r in rows)
        loaded = [r for r in rows if r[0] >= 0.5 * top] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded)}


def _best_tflops(torch, fn, flops, reps=8):
    for _ in range(3):
        fn()
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        best = max(best, flops / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    return best


def gemm_ceiling(torch, dev):
    """Dense bf16 GEMM TFLOP/s measured in this run (cuBLAS through torch),
    8192^3, best of 8 (burst)."""
    n = 8192
    a = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    b = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    best = _best_tflops(torch, lambda: torch.matmul(a, b), 2 * n ** 3)
    del a, b
    return best


def fp8_gemm_ceiling(torch, dev):
    """Dense e4m3 x e4m3 GEMM TFLOP/s (bf16 output, unit scales) measured in
    this run through torch._scaled_mm (cuBLASLt), 8192^3, best of 8 (burst);
    None when this torch build cannot run it."""
    n = 8192
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()   # column-major second operand
        one = torch.ones((), device=dev)
        best = _best_tflops(torch, lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one,
                                                            out_dtype=torch.bfloat16), 2 * n ** 3)
        del a, b
        return best
    except (RuntimeError, AttributeError, TypeError):
        return None


def oracle_sample(w, inputs, seconds=10.0, max_rows=None):
    """Time the fp64 oracle on a bounded sample of the workload: whole
    (sequence, head) pairs in order until the sample has taken ``seconds``
    (or, with ``max_rows``, that many rows of the first pair)."""
    from oracle import oracle as orc
    import numpy as np
    if w.varlen:
        cu = inputs["cu_seqlens_q"].cpu().tolist()
        bounds = [((cu[b], cu[b + 1]), (cu[b], cu[b + 1])) for b in range(w.B)]
    else:
        bounds = [((b * w.Sq, (b + 1) * w.Sq), (b * w.Sk, (b + 1) * w.Sk)) for b in range(w.B)]
    scale = w.D ** -0.5
    spent, pairs, rows, heads = 0.0, 0, 0, 0
    for b, ((s0, s1), (k0, k1)) in enumerate(bounds):
        for h in range(w.H):
            L = s1 - s0
            if L == 0:
                continue
            q = orc._f64(inputs["q"][s0:s1, h, :])
            k = orc._f64(inputs["k"][k0:k1, h, :])
            v = orc._f64(inputs["v"][k0:k1, h, :])
            pos = np.arange(L) if max_rows is None else np.arange(min(L, max_rows))
            t0 = time.perf_counter()
            orc.attention_head(q[pos], pos, k, v, L, scale, w.causal)
            spent += time.perf_counter() - t0
            pairs += orc.visible_pairs(pos, k1 - k0, L, w.causal)
            rows += len(pos)
            heads += 1
            if spent >= seconds or max_rows is not None:
                break
        if spent >= seconds or max_rows is not None:
            break
    flops = 4.0 * pairs * w.D     # the same convention as the GPU metric, per visible pair
    return {"value": flops / spent / 1e12, "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"{rows} query rows ({heads} whole (sequence, head) pairs) of {w.name}, "
                      f"fp64 C oracle with OpenMP, {spent:.2f} s",
            "seconds": spent, "rows": rows}


def oracle_bwd_sample(w, inputs, seconds=10.0, rows=None):
    """Time the oracle's gradients on a bounded sample of a backward workload:
    the leading ``rows`` x ``rows`` square (queries and keys) of (sequence,
    head) pairs in order, whole-matrix fp64 numpy, until ``seconds`` pass. The
    square is sized from a small probe so one pair takes about a second."""
    from oracle import oracle as orc
    import numpy as np
    scale = w.D ** -0.5
    if rows is None:
        n0 = min(512, w.Sq)
        t0 = time.perf_counter()
        orc.attention_backward_head(*(orc._f64(inputs[t][:n0, 0, :]) for t in ("q", "k", "v", "do")), scale,
                                    w.causal)
        dt = max(time.perf_counter() - t0, 1e-4)
        rows = int(min(w.Sq, max(256, n0 * (1.0 / dt) ** 0.5)))
    spent, flops, pairs = 0.0, 0.0, 0
    for b in range(w.B):
        for h in range(w.H):
            s0 = b * w.Sq
            args = [orc._f64(inputs[t][s0:s0 + rows, h, :]) for t in ("q", "k", "v", "do")]
            t0 = time.perf_counter()
            orc.attention_backward_head(*args, scale, w.causal)
            spent += time.perf_counter() - t0
            flops += 10.0 * rows * rows * w.D * (0.5 if w.causal else 1.0)
            pairs += 1
            if spent >= seconds:
                break
        if spent >= seconds:
            break
    return {"value": flops / spent / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{pairs} (sequence, head) pairs of {w.name} cut to their first {rows} queries and keys, "
                      f"fp64 numpy gradients (BLAS on all host cores), {spent:.2f} s; FLOPs counted as "
                      f"2.5x the forward's",
            "seconds": spent, "rows": rows}


def max_over_ranks(ms: float, device=None) -> float:
    """The slowest rank's time (the job finishes when its last rank does).
    Single process: the value itself. Uses whatever backend the process group
    was started with (NCCL with a CUDA device on the GPU machine, gloo on CPU)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Weak scaling: every rank processes its own copy of the workload, so the
    job's throughput is all ranks' units over the slowest rank's time."""
    return world * units_per_rank / (ms_per_step * 1e-3) / 1e12


def run_reference(args):
    """The oracle as the reference arm: each step a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import torch  # noqa: F401
    from exact_attention_forward_tiled_gb300 import workloads
    from oracle import oracle as orc
    orc.build()
    w = workloads.WORKLOADS[args.workload]
    inputs = workloads.make_inputs(w, device="cpu")
    vals = []
    if w.backward:
        # one step = the gradients of the first (sequence, head) cut to a
        # square that takes ~1 s
        probe = oracle_bwd_sample(w, inputs, seconds=0.0)
        for i in range(args.warmup + args.steps):
            r = oracle_bwd_sample(w, inputs, seconds=0.0, rows=probe["rows"])
            if i >= args.warmup:
                vals.append(r)
    else:
        # one step = the rows of the first (sequence, head) that take ~1 s
        probe = oracle_sample(w, inputs, seconds=0.0, max_rows=256)
        rows = max(16, int(256 * 1.0 / max(probe["seconds"], 1e-3)))
        for i in range(args.warmup + args.steps):
            r = oracle_sample(w, inputs, seconds=1e9, max_rows=rows)
            if i >= args.warmup:
                vals.append(r)
    tot_s = sum(r["seconds"] for r in vals)
    value = statistics.mean(r["value"] for r in vals)
    line = {"impl": "reference", "metric": METRIC_BWD if w.backward else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / len(vals),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "Sq": w.Sq, "Sk": w.Sk,
                                            "D": w.D, "causal": w.causal},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": vals[0]["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="c2")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's number of sequences (smaller profiling cases)")
    ap.add_argument("--page-size", type=int, default=None,
                    help="paged workloads: override the page size; 0 runs the same shapes with contiguous K/V "
                         "through fa_fwd")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    from exact_attention_forward_tiled_gb300 import accounting as A
    from exact_attention_forward_tiled_gb300 import api, workloads
    from exact_attention_forward_tiled_gb300 import build as fb

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        fb.build()
    if world > 1:
        dist.barrier()
    api.lib()

    w = workloads.WORKLOADS[args.workload]
    from dataclasses import replace
    if args.batch is not None and not w.varlen:
        w = replace(w, B=args.batch, name=f"{w.name}_B{args.batch}")
    if args.page_size is not None and w.page_size:
        w = replace(w, page_size=args.page_size,
                    name=w.name.rsplit("_page", 1)[0] + (f"_page{args.page_size}" if args.page_size else "_contiguous"))
    fp8 = w.dtype == "fp8"
    inputs = workloads.make_inputs(w, device=dev)
    q, k, v = inputs["q"], inputs["k"], inputs["v"]
    scale = w.D ** -0.5
    stream = torch.cuda.current_stream(dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16 if fp8 else q.dtype, device=dev)
    if w.varlen:
        cu = inputs["cu_seqlens_q"]
        lens = inputs["lengths"].tolist()
        lse = torch.empty((w.H, q.shape[0]), device=dev, dtype=torch.float32)
        Sq = Sk = inputs["max_seqlen"]
        flops = A.attention_flops(w.H, w.D, lens, lens, w.causal)
        extra = dict(cu_seqlens_q=cu, cu_seqlens_k=cu, total_q=q.shape[0], total_k=k.shape[0])
    else:
        lse = torch.empty((w.B, w.H, w.Sq), device=dev, dtype=torch.float32)
        Sq, Sk = w.Sq, w.Sk
        flops = A.attention_flops(w.H, w.D, [w.Sq] * w.B, [w.Sk] * w.B, w.causal)
        if w.Sq != w.Sk:   # count the visible pairs exactly (bottom-right causal mask)
            flops = A.visible_pair_flops(w.H, w.D, [w.Sq] * w.B, [w.Sk] * w.B, w.causal)
        extra = {}

    # one step = the whole hot path; for fp8 the prep kernel then the attention;
    # for a backward workload one fa_bwd call (row constants, dK/dV, dQ).
    # hot_path(ins, outs, stream) returns the list of its launches; `ins` are
    # the step's inputs (copied from the host in the end-to-end loop), `outs`
    # its results (copied back).
    ins, outs = [q, k, v], [o, lse]
    if w.backward:
        do = inputs["do"]
        api.attention_forward(q, k, v, causal=w.causal, scale=scale, batch=w.B, out=o, lse=lse)
        ins = [q, k, v, o, do, lse]   # the order of fa_bwd's arguments
        outs = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
        ws_bytes = api.fa_bwd_workspace_size(w.H, q.shape[0])
        bwd_ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        flops = A.attention_bwd_flops(w.H, w.D, [w.Sq] * w.B, [w.Sk] * w.B, w.causal)

        def hot_path(i_, o_, st):
            return [lambda: api.fa_bwd(*i_, *o_, w.B, w.H, Sq, Sk, w.D, scale, w.causal, workspace=bwd_ws,
                                       workspace_bytes=ws_bytes, stream=st)]
        names = ["fa_bwd (bwd_prep_kernel + fa_bwd_kernel dK/dV + fa_bwd_kernel dQ)" if w.D <= 128 else
                 "fa_bwd (bwd_prep_kernel + fa_bwd_kernel dV + fa_bwd_kernel dK + fa_bwd_kernel dQ)"]
    elif w.page_size:
        kc, vc, table, seqlens = (inputs[n] for n in ("k_cache", "v_cache", "block_table", "seqlens_k"))
        max_pages = table.shape[1]
        splits = 0 if w.Sq == 1 else 1   # decode: automatic key ranges
        ws_bytes = (api.fa_fwd_splitkv_workspace_size(w.B, w.H, w.Sq, max_pages * w.page_size, w.D, splits)
                    if splits != 1 else 0)
        paged_ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        ins = [q]   # the K/V cache stays resident on the device, as in serving

        def hot_path(i_, o_, st):
            return [lambda: api.fa_fwd_paged(i_[0], kc, vc, table, seqlens, *o_, w.B, w.H, w.Sq, w.D, kc.shape[0],
                                             w.page_size, max_pages, scale, w.causal, splits, paged_ws, ws_bytes,
                                             stream=st)]
        names = ["fa_fwd_kernel (paged)" + (" + splitkv_merge_kernel" if splits != 1 else "")]
    elif fp8:
        prep = api.fp8_prepare(q, k, v, inputs["sigma"], batch=w.B, stream=stream)

        def hot_path(i_, o_, st):
            qq, kk, vv = i_
            return [lambda: api.fa_fp8_prep(qq, kk, vv, prep["q8"], prep["k8"], prep["v8"], prep["q_scale"],
                                            prep["k_scale"], prep["v_scale"], inputs["sigma"], w.B, w.H, Sq, Sk,
                                            w.D, stream=st),
                    lambda: api.fp8_attention_forward(prep, causal=w.causal, scale=scale, out=o_[0], lse=o_[1],
                                                      stream=st)]
        names = ["fp8_prep_kernel", "fa_fwd_kernel"]
    elif w.splitkv:
        ws_bytes = api.fa_fwd_splitkv_workspace_size(w.B, w.H, Sq, Sk, w.D, 0)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

        def hot_path(i_, o_, st):
            return [lambda: api.fa_fwd_splitkv(*i_, *o_, w.B, w.H, Sq, Sk, w.D, scale, w.causal, 0,
                                               workspace, ws_bytes, stream=st)]
        names = ["fa_fwd_kernel+splitkv_merge_kernel"]
    else:
        def hot_path(i_, o_, st):
            return [lambda: api.fa_fwd(*i_, *o_, w.B, w.H, Sq, Sk, w.D, scale, w.causal, stream=st, **extra)]
        names = ["fa_fwd_kernel"]
    kernels = list(zip(names, hot_path(ins, outs, stream)))

    def step():
        for _, fn in kernels:
            fn()

    for _ in range(args.warmup):
        step()
    api.fa_get_device_status(stream)
    ceiling = gemm_ceiling(torch, dev)
    ceiling8 = fp8_gemm_ceiling(torch, dev) if fp8 else None

    def timed(fn, steps, per_kernel=False):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ev = lambda: torch.cuda.Event(enable_timing=True)
        e0, e1 = ev(), ev()
        marks = []
        e0.record(stream)
        for _ in range(steps):
            if per_kernel:
                m = [ev() for _ in range(len(kernels) + 1)]
                m[0].record(stream)
                for j, (_, kf) in enumerate(kernels):
                    kf()
                    m[j + 1].record(stream)
                marks.append(m)
            else:
                fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        ms = max_over_ranks(e0.elapsed_time(e1), dev)
        per = [sum(m[j].elapsed_time(m[j + 1]) for m in marks) / max(1, len(marks))
               for j in range(len(kernels))] if per_kernel else None
        return ms, per

    with ClockSampler(local) as clk:
        total_ms, per_kernel = timed(step, args.steps, per_kernel=True)
    api.fa_get_device_status(stream)
    ms_per_step = total_ms / args.steps
    value = job_value(flops, world, ms_per_step)

    # end to end through the C ABI from pinned host buffers: every step copies
    # its inputs in and its results out. Copies and compute of neighbouring
    # steps overlap (H2D and D2H on their own streams, two sets of device
    # buffers), as a serving loop would run them.
    in_host = [t.cpu().pin_memory() for t in ins]
    out_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d_st, d2h_st = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = [(ins, outs), ([torch.empty_like(t) for t in ins], [torch.empty_like(t) for t in outs])]
    runs = [hot_path(i_, o_, stream) for i_, o_ in sets]
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_ready = [ev(), ev()]
    out_ready = [ev(), ev()]
    out_free = [ev(), ev()]
    in_free = [ev(), ev()]
    for e_ in in_free + out_free:
        e_.record(stream)

    def e2e_loop(steps):
        for i in range(steps):
            b = i % 2
            i_dev, o_dev = sets[b]
            h2d_st.wait_event(in_free[b])
            with torch.cuda.stream(h2d_st):
                for d_, h_ in zip(i_dev, in_host):
                    d_.copy_(h_, non_blocking=True)
            in_ready[b].record(h2d_st)
            stream.wait_event(in_ready[b])
            stream.wait_event(out_free[b])
            for fn in runs[b]:
                fn()
            in_free[b].record(stream)
            out_ready[b].record(stream)
            d2h_st.wait_event(out_ready[b])
            with torch.cuda.stream(d2h_st):
                for h_, d_ in zip(out_host, o_dev):
                    h_.copy_(d_, non_blocking=True)
            out_free[b].record(d2h_st)

    e2e_loop(3)
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, min(args.steps, 50))
    if world > 1:
        dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(h2d_st)
    e2e_loop(e2e_steps)
    d2h_st.wait_stream(h2d_st)
    d2h_st.wait_stream(stream)
    t1.record(d2h_st)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), dev) / e2e_steps
    api.fa_get_device_status(stream)
    h2d = sum(t.numel() * t.element_size() for t in in_host)
    d2h = sum(t.numel() * t.element_size() for t in out_host)

    peaks, peak_src = load_peaks()
    attn_ms = per_kernel[-1]
    achieved = flops / (attn_ms * 1e-3) / 1e12
    if fp8 and ceiling8:
        peak = ceiling8
        peak_note = ("e4m3 dense GEMM 8192^3 (torch._scaled_mm, cuBLASLt, burst) measured in this run; the "
                     f"{peak_src} bf16 burst x 2 (nominal fp8/bf16 ratio) would be {peaks['bf16_tflops'] * 2.0:.1f}")
    elif fp8:
        peak = peaks["bf16_tflops"] * 2.0
        peak_note = (f"{peak_src} bf16 dense GEMM (burst) x 2, the nominal fp8/bf16 dense ratio "
                     "(4.5 / 2.25 PFLOP/s); no e4m3 GEMM could be timed in this run")
    else:
        peak = peaks["bf16_tflops"]
        peak_note = f"{peak_src} bf16 dense GEMM (burst), MEASURED_PEAKS.json"
    kern = "fa_fwd_kernel"
    if w.backward:
        kern = "fa_bwd"
        peak_note += ("; achieved = algorithmic backward FLOPs (5 matrix products, 2.5x the forward's) over "
                      "the whole fa_bwd call (3 kernels; the dQ kernel recomputes S and dP, 7 products run)")
    if w.splitkv or (w.page_size and w.Sq == 1):
        peak_note += "; achieved covers the attention and the merge kernel of each call"
    line = {
        "metric": METRIC_BWD if w.backward else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if fp8 else w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Sq": Sq, "Sk": Sk, "D": w.D,
                   "causal": w.causal, "varlen": w.varlen, "scale": scale,
                   "l2": "inputs larger than L2 (no flush between steps)",
                   "inputs": "Q,K,V iid N(0,1) fp32 -> %s, seed %d%s" % (
                       "bf16" if fp8 else w.dtype, w.seed,
                       ", 0.1%% N(0,10^2) outliers in 4 columns, prep + attention per step" if fp8 else
                       (", dO iid N(0,1); O, LSE from one forward before timing; one fa_bwd per step"
                        if w.backward else ""))},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": committed_traffic(kern, w.name),
                     "peak_source": peak_note, "kernel": kern, "kernel_ms": attn_ms},
        "ceiling_in_run": {"bf16_gemm_tflops": ceiling,
                           **({"fp8_gemm_tflops": ceiling8} if fp8 else {}),
                           "frac": achieved / ((ceiling8 or 2.0 * ceiling) if fp8 else ceiling)},
        "e2e": {"value": job_value(flops, world, e2e_ms), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "note": ("pinned host -> device copy of Q, K, V, O, LSE, dO and device -> host copy of dQ, "
                         "dK, dV every step" if w.backward else
                         "pinned host -> device copy of Q and device -> host copy of O, LSE every step; the "
                         "paged K/V cache stays resident" if w.page_size else
                         "pinned host -> device copy of Q, K, V and device -> host copy of O, LSE every step")
                        + "; copies of neighbouring steps overlap compute (two buffer sets, H2D / D2H streams)"},
        "gpu_launches": args.steps * ((4 if w.D == 256 else 3) if w.backward
                                      else 2 if (w.splitkv or (w.page_size and w.Sq == 1))
                                      else len(kernels)),
        "clocks": clk.summary(),
    }
    if w.page_size and w.Sq == 1:
        # decode: one query per sequence; the bound is reading the cache once
        kvb = A.paged_kv_bytes(w.H, w.D, [w.Sk] * w.B)
        gbs = kvb / (attn_ms * 1e-3) / 1e9
        line["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": gbs / peaks["hbm_gbs"], "traffic": committed_traffic(kern, w.name),
                            "peak_source": f"{peak_src} HBM copy bandwidth, MEASURED_PEAKS.json; achieved = one "
                                           "read of every cached K and V row over the attention + merge call",
                            "kernel": kern, "kernel_ms": attn_ms, "bytes": kvb}
    if fp8:
        pb = A.prep_bytes(w.H, w.D, w.B, w.Sq)
        gbs = pb / (per_kernel[0] * 1e-3) / 1e9
        line["prep_roofline"] = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": gbs / peaks["hbm_gbs"], "kernel": "fp8_prep_kernel",
                                 "kernel_ms": per_kernel[0], "bytes": pb,
                                 "traffic": committed_traffic("fp8_prep_kernel", w.name)}
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        host = {"q": q.cpu(), "k": k.cpu(), "v": v.cpu(), "cu_seqlens_q": inputs["cu_seqlens_q"]}
        if w.backward:
            host["do"] = inputs["do"].cpu()
            cb = oracle_bwd_sample(w, host, seconds=args.cpu_seconds)
        else:
            cb = oracle_sample(w, host, seconds=args.cpu_seconds)
            # the same oracle on one host thread, over the first 512 rows of
            # the first (sequence, head) pair
            from oracle import oracle as orc
            n_thr = orc.num_threads()
            orc.set_num_threads(1)
            try:
                one = oracle_sample(w, host, seconds=0.0, max_rows=512)
            finally:
                orc.set_num_threads(n_thr)
            cb["value_1_thread"] = one["value"]
            cb["sample_1_thread"] = one["sample"].replace("with OpenMP", "on 1 thread")
        cb.pop("seconds")
        cb.pop("rows")
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
