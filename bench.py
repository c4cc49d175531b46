#!/usr/bin/env python
"""Throughput of Attention Matching KV compaction on B300.

One step = one kvc_compact call over every head of the workload (all steps
of the compaction: logits/lse/outputs, key scores, top-t, gather, mass
matrix, NNLS for beta, least squares for C_v), inputs resident in HBM.
Metric: compacted head-tokens per second = sum over heads of T / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]
                  [--layers L] [--select rms|omp|tam]

The default workload is the largest one that fits one GPU: the 32-layer x
8-KV-head Llama-3-8B-shaped cache (256 heads, T = 32768, n = 8192,
t = 655).  --layers L keeps the first L layers of a multi-layer workload
(same per-head shapes; for profiler captures of a bounded size).

N > 1 runs one independent replica per GPU (launched by torch.distributed.run):
heads are independent, so each rank compacts its own sequences with no
collective on the data path; only the timing barrier and a max-reduction of
the step time cross ranks (weak scaling).

--impl reference times the float64 CPU oracle (the only other
implementation of this method that exists) on the host cores, one head per
step, in the same metric.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import WORKLOADS, budgets as make_budgets  # noqa: E402

# fp32 FFMA peak of a B300 (148 SMs x 128 lanes x 2 flop x 2032 MHz), for
# kernels that run on the CUDA cores.
SIMT_F32_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            j = json.load(fh)
        return j, "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


# --------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.lines: list[str] = []
        self.proc = None
        self.th = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 3.0:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- work model
def stage_work(w, buds):
    """Algorithmic work per stage for one call: (kind, amount, unit).

    flops count a multiply-add as 2; symmetric Grams count only the distinct
    entries; bytes are the minimum the stage must move through HBM."""
    H, n, T, d = w.H, w.n, w.T, w.d
    b_in = 2 if w.dtype == "bf16" else 4
    t = [int(x) for x in buds]
    st = sum(t)
    return {
        "v_f16": ("bytes", 2.0 * 2 * T * d * H),        # reads V (bf16), writes fp16 once
        "attn_fwd": ("flops", 4.0 * n * T * d * H),
        "colscore": ("flops", 2.0 * n * T * d * H),
        "select": ("bytes", 4.0 * T * H + 4.0 * st),
        "gather": ("bytes", 2.0 * st * d * b_in + st * d * (b_in + 4) + 4.0 * st),
        "masslogits": ("flops", 2.0 * n * d * st),
        "gram_a": ("flops", float(sum(n * ti * (ti + 1) for ti in t))),
        # the inversions count the method's work, a factorisation of the t x t
        # system (t^3 / 3), not the explicit inverse's t^3
        "inv_h": ("flops", float(sum(float(ti) ** 3 / 3.0 for ti in t))),
        "gram_x": ("flops", float(sum(n * ti * (ti + 1) for ti in t))),
        "xto": ("flops", 2.0 * n * d * st),
        "chol_m": ("flops", float(sum(ti ** 3 / 3.0 for ti in t))),
        "cholsolve": ("flops", float(sum(2.0 * ti * ti * d for ti in t))),
        "inv_m": ("flops", float(sum(float(ti) ** 3 / 3.0 for ti in t))),
        "apply_minv": ("flops", float(sum(2.0 * ti * ti * d for ti in t))),
    }


# MUFU ex2 rate of a B300: 148 SMs x 32 per clock x 2032 MHz (Blackwell
# Ultra doubled the special-function rate for attention; a probe of
# independent ex2.approx chains sustained 29.8 per SM per clock).  The
# attention passes take one exponential per logit and are co-bound by it.
MUFU_PEAK_TEXP = 148 * 32 * 2.032e9 / 1e12


def tensor_stages(w) -> set[str]:
    """Stages that run on the tensor cores (bf16 operands, fp32 accumulation)
    for this workload; the others run on the CUDA cores (fp32 FFMA) or are
    memory-bound.  The Gram products and C_v = M^{-1} R run on the tensor
    cores for every input dtype (their fp32 operands are split into bf16
    terms)."""
    grams = {"gram_a", "gram_x", "xto", "apply_minv"}
    return grams | ({"attn_fwd", "colscore", "masslogits"} if w.dtype == "bf16" else set())


TENSOR_STAGES: set[str] = set()


def roofline_for(stage, per_launch_ms, work, peaks, peak_src, traffic):
    kind, amount = work
    if kind == "bytes":
        ach = amount / (per_launch_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(ach, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic, "kernel": stage,
                "peak_source": f"{peak_src} hbm_gbs"}
    ach = amount / (per_launch_ms * 1e-3) / 1e12
    if stage in TENSOR_STAGES:
        pk = peaks["bf16_tflops"]
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": pk, "unit": "TFLOP/s",
                "frac": round(ach / pk, 4), "traffic": traffic, "kernel": stage,
                "peak_source": f"{peak_src} bf16_tflops (burst)"}
    return {"bound": "alu", "achieved": round(ach, 3), "peak": round(SIMT_F32_PEAK_TFLOPS, 2), "unit": "TFLOP/s",
            "frac": round(ach / SIMT_F32_PEAK_TFLOPS, 4), "traffic": traffic, "kernel": stage,
            "peak_source": "derived fp32 FFMA peak 148 SM x 128 lanes x 2 x 2032 MHz"}


# --------------------------------------------------------------- CPU oracle
def time_oracle(w, heads, buds):
    """Seconds per head of the float64 oracle, and the BLAS threads it used."""
    import numpy as np
    import oracle
    from workloads import forced_mask, head_inputs
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"] or [1])
    except Exception:  # noqa: BLE001
        cores = 1
    # BLAS threads cannot exceed the cores this process may run on
    cores = min(cores, len(os.sched_getaffinity(0)))
    forced = forced_mask(w) if (w.keep_first or w.keep_last) else None
    times = []
    for h in heads:
        x = head_inputs(w, h, with_test=False)
        Q, K, V = (oracle.decode(x[k], w.dtype) for k in "QKV")
        t0 = time.perf_counter()
        oracle.compact_head(Q, K, V, int(buds[h]), forced=forced)
        times.append(time.perf_counter() - t0)
    return times, cores


def config_dict(w, buds, world, select="rms"):
    if select == "tam":
        select = f"tam (window {TAM_WINDOW}, c {TAM_C:g}, {max(1, w.segments)} segments, no forced keys)"
    return {"workload": w.name, "heads_per_gpu": w.H, "n": w.n, "T": w.T, "d": w.d, "key_selection": select,
            "t": (w.t if w.t is not None else f"nonuniform mean {float(sum(buds)) / len(buds):.1f}"),
            "input_dtype": w.dtype, "keep_first": w.keep_first, "keep_last": w.keep_last,
            "l2": "flushed between steps (256 MiB write)", "parallelism": f"replicas x{world}"}


# --------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return 0
    w = WORKLOADS[args.config]
    buds = make_budgets(w)
    n_steps = args.warmup + args.steps
    heads = [i % w.H for i in range(n_steps)]
    times, cores = time_oracle(w, heads, buds)
    timed = times[args.warmup:]
    sec = sum(timed)
    value = w.T * len(timed) / sec
    line = {
        "impl": "reference", "metric": "compacted KV head-tokens/sec", "value": round(value, 2),
        "unit": "head-tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sec / len(timed), 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator, workload shapes of the pages)",
        "config": config_dict(w, buds, 1),
        "cpu_baseline": {"value": round(value, 2), "unit": "head-tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"one KV head per step ({len(timed)} timed heads of {w.H})"},
        "e2e": {"value": round(value, 2), "unit": "head-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- sharding
def rank_workload(base, rank: int, world: int):
    """The workload replica of `rank`: the same shapes, its own sequences.

    Heads are independent problems, so N ranks compact N disjoint sets of
    sequences (weak scaling) and exchange nothing on the data path."""
    import dataclasses
    if world <= 1:
        return base
    return dataclasses.replace(base, seq_offset=base.seq_offset + rank * base.seqs)


def limit_layers(w, layers):
    """The first `layers` layers of a multi-layer workload (None: all)."""
    import dataclasses
    if not layers or layers >= w.layers:
        return w
    return dataclasses.replace(w, layers=layers, name=f"{w.name}-first{layers}layers")


def oracle_sample(w):
    """Heads the CPU baseline times: every head of a workload of at most 8,
    else 4 heads evenly spaced over the flat head index (so over sequences,
    layers and KV heads), whose mean time stands for every head."""
    if w.H <= 8:
        return list(range(w.H))
    return [round(i * (w.H - 1) / 3) for i in range(4)]


def max_over_ranks(x: float, dist, device) -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# thought-aware leg (--select tam): window of the last 128 tokens, pivot factor 16
TAM_WINDOW = 128
TAM_C = 16.0


# --------------------------------------------------------------- decode leg
def measure_decode(kvc, w, inputs, K, V, Ck, beta, Cv, offsets, total, flush, stream, dev, dist, reps=20):
    """One decoded token per query head (n_q = the GQA group) read through
    kvc_attend: over the compacted cache (t_h keys with bias) and over the
    full cache (T keys, bias 0, values in fp32 like C_v), L2 flushed before
    every call.  Both are HBM streams; returns times, speedup and the
    fraction of the measured HBM bandwidth each reaches."""
    import numpy as np
    import torch

    nq = max(1, w.gqa)
    qt = inputs["Qt"][:, :nq]
    qt = np.ascontiguousarray(qt)
    Qd = torch.from_numpy(qt.view(np.int16) if w.dtype == "bf16" else qt)
    if w.dtype == "bf16":
        Qd = Qd.view(torch.bfloat16)
    Qd = Qd.to(dev)
    H, T, d = w.H, w.T, w.d
    Kf = K.view(H * T, d)
    Vf = V.view(H * T, d).float()
    bf = torch.zeros(H * T, dtype=torch.float32, device=dev)
    of = torch.arange(H + 1, dtype=torch.int32, device=dev) * T
    O = torch.empty(H, nq, d, dtype=torch.float32, device=dev)
    st = torch.empty(H, dtype=torch.int32, device=dev)
    prob = kvc.make_problem(H, nq, 1, d, kvc.DTYPE_BF16 if w.dtype == "bf16" else kvc.DTYPE_F32, 1)

    def timed(ck, b, cv, off):
        for _ in range(3):
            if kvc.attend(prob, Qd, nq, ck, b, cv, off, O, st, 0.0, stream):
                raise RuntimeError("kvc_attend refused the call")
        ms = 0.0
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            kvc.attend(prob, Qd, nq, ck, b, cv, off, O, st, 0.0, stream)
            e1.record(stream)
            e1.synchronize()
            ms += e0.elapsed_time(e1)
        if not bool((st == 0).all()):
            raise RuntimeError("kvc_attend head status not OK")
        return ms / reps

    comp_ms = max_over_ranks(timed(Ck, beta, Cv, offsets), dist, dev)
    full_ms = max_over_ranks(timed(Kf, bf, Vf, of), dist, dev)
    b_in = 2 if w.dtype == "bf16" else 4
    per_key = d * (b_in + 4) + 4
    io = H * nq * d * (b_in + 4)
    comp_bytes = total * per_key + io
    full_bytes = H * T * per_key + io
    peaks, src = _peaks()
    return {
        "n_q": nq, "keys_compacted": int(total), "keys_full": H * T,
        "compacted_us": round(comp_ms * 1e3, 2), "full_us": round(full_ms * 1e3, 2),
        "speedup": round(full_ms / comp_ms, 2),
        "compacted_hbm_frac": round(comp_bytes / (comp_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "full_hbm_frac": round(full_bytes / (full_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "peak_source": f"{src} hbm_gbs",
        "what": "kvc_attend, one decoded token per query head, compacted cache vs full cache (bias 0, fp32 values)",
    }


# --------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import kv_cache_compaction_03_b300 as kvc
    from workloads.batch import generate

    w = rank_workload(limit_layers(WORKLOADS[args.config], args.layers), rank, world)
    TENSOR_STAGES.clear()
    TENSOR_STAGES.update(tensor_stages(w))
    buds = make_budgets(w)
    inputs = generate(w)                     # spawn pool, before any CUDA call

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)

    def dev_tensor(a):
        t = torch.from_numpy(a.view(np.int16) if w.dtype == "bf16" else a)
        if w.dtype == "bf16":
            t = t.view(torch.bfloat16)
        return t.to(dev)

    Q, K, V = dev_tensor(inputs["Q"]), dev_tensor(inputs["K"]), dev_tensor(inputs["V"])
    b_dev = torch.from_numpy(buds.astype(np.int32)).to(dev)
    offsets = torch.zeros(w.H + 1, dtype=torch.int32, device=dev)
    offsets[1:] = torch.cumsum(b_dev.to(torch.int64), 0).to(torch.int32)
    total = int(buds.sum())
    max_t = int(buds.max())
    prob = kvc.make_problem(w.H, w.n, w.T, w.d, kvc.DTYPE_BF16 if w.dtype == "bf16" else kvc.DTYPE_F32, max_t)
    flags = kvc.FLAG_STAGE_TIMING | (kvc.FLAG_SELECT_OMP if args.select == "omp" else 0)
    tam = args.select == "tam"
    prm = kvc.default_params(keep_first=0 if tam else w.keep_first, keep_last=0 if tam else w.keep_last, flags=flags)
    if tam:
        from workloads import segment_bounds, window_queries
        win = np.stack([window_queries(w, h, TAM_WINDOW) for h in range(w.H)])
        Qw = dev_tensor(win)
        seg_bounds = torch.from_numpy(segment_bounds(w)).to(dev)
        nseg = seg_bounds.numel() - 1
        seg_out = torch.empty(w.H, nseg, dtype=torch.int32, device=dev)
        piv_out = torch.empty(w.H, w.T, dtype=torch.uint8, device=dev)
        ws_bytes = kvc.workspace_size_tam(prob, prm, TAM_WINDOW, nseg)
    else:
        ws_bytes = kvc.workspace_size(prob, prm)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    idx = torch.empty(total, dtype=torch.int32, device=dev)
    Ck = torch.empty(total, w.d, dtype=tdt, device=dev)
    beta = torch.empty(total, dtype=torch.float32, device=dev)
    Cv = torch.empty(total, w.d, dtype=torch.float32, device=dev)
    status = torch.empty(w.H, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if tam:
            rc = kvc.compact_tam(prob, prm, Q, K, V, Qw, TAM_WINDOW, seg_bounds, nseg, TAM_C, b_dev, offsets, idx, Ck,
                                 beta, Cv, status, seg_out, piv_out, ws, ws_bytes, stream)
        else:
            rc = kvc.compact(prob, prm, Q, K, V, b_dev, offsets, idx, Ck, beta, Cv, status, ws, ws_bytes, stream)
        if rc:
            raise kvc.KvcError(rc, "kvc_compact")

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st_host = status.cpu().numpy()
    if not np.all(st_host == 0):
        raise RuntimeError(f"head status not OK after warm-up: {st_host.tolist()}")

    sampler = ClockSampler(local_rank)
    sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms, stage_acc, launches = [], {}, 0
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        stages, nl = kvc.stage_times()          # waits for this step's last stage
        launches += nl
        e1.synchronize()
        step_ms.append(e0.elapsed_time(e1))
        for name, ms, cnt in stages:
            a = stage_acc.setdefault(name, [0.0, 0])
            a[0] += ms
            a[1] += cnt
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    ms_per_step = total_ms / args.steps
    value = world * w.H * w.T / (ms_per_step * 1e-3)

    # ---- end to end: pinned host inputs in, compacted cache out, every step.
    # Serial: copy in, compact, copy out, one step after the other.  Pipelined
    # (the headline, as a serving loop runs): two buffer sets; step i+1's
    # inputs go in on a copy stream and step i's results come out on an output
    # stream while step i compacts.  Every step still moves its own inputs in
    # and its own results out.
    hQ, hK, hV = (torch.from_numpy(inputs[k].view(np.int16) if w.dtype == "bf16" else inputs[k]).pin_memory()
                  for k in "QKV")
    hb = torch.from_numpy(buds.astype(np.int32)).pin_memory()
    o_idx = torch.empty(total, dtype=torch.int32).pin_memory()
    o_Ck = torch.empty(total * w.d * (2 if w.dtype == "bf16" else 4), dtype=torch.uint8).pin_memory()
    o_beta = torch.empty(total, dtype=torch.float32).pin_memory()
    o_Cv = torch.empty(total, w.d, dtype=torch.float32).pin_memory()
    o_st = torch.empty(w.H, dtype=torch.int32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hQ, hK, hV, hb))
    d2h = sum(x.numel() * x.element_size() for x in (o_idx, o_Ck, o_beta, o_Cv, o_st))
    bufs = [dict(Q=Q, K=K, V=V, b=b_dev, idx=idx, Ck=Ck, beta=beta, Cv=Cv, st=status)]
    bufs.append({k: torch.empty_like(v) for k, v in bufs[0].items()})

    def raw(t):
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t

    def copy_in(bq):
        raw(bq["Q"]).copy_(hQ, non_blocking=True)
        raw(bq["K"]).copy_(hK, non_blocking=True)
        raw(bq["V"]).copy_(hV, non_blocking=True)
        bq["b"].copy_(hb, non_blocking=True)

    def copy_out(bq):
        o_idx.copy_(bq["idx"], non_blocking=True)
        o_Ck.copy_(bq["Ck"].view(torch.uint8).view(-1), non_blocking=True)
        o_beta.copy_(bq["beta"], non_blocking=True)
        o_Cv.copy_(bq["Cv"], non_blocking=True)
        o_st.copy_(bq["st"], non_blocking=True)

    def step_on(bq):
        if tam:
            rc = kvc.compact_tam(prob, prm, bq["Q"], bq["K"], bq["V"], Qw, TAM_WINDOW, seg_bounds, nseg, TAM_C,
                                 bq["b"], offsets, bq["idx"], bq["Ck"], bq["beta"], bq["Cv"], bq["st"], seg_out,
                                 piv_out, ws, ws_bytes, stream)
        else:
            rc = kvc.compact(prob, prm, bq["Q"], bq["K"], bq["V"], bq["b"], offsets, bq["idx"], bq["Ck"], bq["beta"],
                             bq["Cv"], bq["st"], ws, ws_bytes, stream)
        if rc:
            raise kvc.KvcError(rc, "kvc_compact")

    serial_ms = []
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_in(bufs[0])
        step_on(bufs[0])
        copy_out(bufs[0])
        e1.record(stream)
        e1.synchronize()
        serial_ms.append(e0.elapsed_time(e1))
    if not np.all(o_st.numpy() == 0):
        raise RuntimeError("head status not OK in the end-to-end loop")

    cps, outs = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    flush.zero_()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cps.wait_event(e0)
    with torch.cuda.stream(cps):
        copy_in(bufs[0])
    ev_in[0].record(cps)
    for i in range(args.steps):
        cur, nxt = i % 2, (i + 1) % 2
        if i + 1 < args.steps:
            if i >= 1:
                cps.wait_event(ev_done[nxt])          # step i-1 has finished reading that set
            with torch.cuda.stream(cps):
                copy_in(bufs[nxt])
            ev_in[nxt].record(cps)
        stream.wait_event(ev_in[cur])
        if i >= 2:
            stream.wait_event(ev_out[cur])            # step i-2's results are out
        step_on(bufs[cur])
        ev_done[cur].record(stream)
        outs.wait_event(ev_done[cur])
        with torch.cuda.stream(outs):
            copy_out(bufs[cur])
        ev_out[cur].record(outs)
    stream.wait_stream(outs)
    e1.record(stream)
    e1.synchronize()
    pipe_total = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    if not np.all(o_st.numpy() == 0):
        raise RuntimeError("head status not OK in the pipelined end-to-end loop")
    e2e_value = world * w.H * w.T / (pipe_total / args.steps * 1e-3)
    serial_value = world * w.H * w.T / (max_over_ranks(sum(serial_ms), dist, dev) / args.steps * 1e-3)

    # ---- decode: kvc_attend over the compacted cache vs over the full cache
    decode = measure_decode(kvc, w, inputs, K, V, Ck, beta, Cv, offsets, total, flush, stream, dev, dist)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = _peaks()
    work = stage_work(w, buds)
    per_stage = {}
    for name, (ms, cnt) in stage_acc.items():
        entry = {"ms_per_step": round(ms / args.steps, 4), "share": round(ms / max(1e-9, sum(a[0] for a in stage_acc.values())), 4),
                 "launches_per_step": cnt // args.steps}
        if name in work:
            r = roofline_for(name, ms / args.steps, work[name], peaks, peak_src, None)
            entry.update({"bound": r["bound"], "achieved": r["achieved"], "unit": r["unit"], "frac": r["frac"]})
        if name in ("attn_fwd", "colscore"):
            texp = w.H * w.n * w.T / (ms / args.steps * 1e-3) / 1e12
            entry["exp_frac_of_mufu"] = round(texp / MUFU_PEAK_TEXP, 4)
        per_stage[name] = entry
    dom = max((n for n in stage_acc if n in work), key=lambda n: stage_acc[n][0])
    traffic = _traffic_for(dom, args.config)
    roof = roofline_for(dom, stage_acc[dom][0] / args.steps, work[dom], peaks, peak_src, traffic)

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sample_heads = oracle_sample(w)
        times, cores = time_oracle(w, sample_heads, buds)
        per_head = sum(times) / len(times)
        extra = "" if len(times) == w.H else f"; {w.H} x the mean per-head time (extrapolated)"
        cpu = {"value": round(w.T / per_head, 2), "unit": "head-tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"heads {sample_heads} of {w.H}, {per_head:.2f} s per head (float64 numpy){extra}"}

    line = {
        "metric": "compacted KV head-tokens/sec", "value": round(value, 1), "unit": "head-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if TENSOR_STAGES else "f32",
        "solver_dtype": "f32",
        "data": "synthetic (seeded generator, workload shapes of the pages)",
        "config": config_dict(w, buds, world, args.select),
        "e2e": {"value": round(e2e_value, 1), "unit": "head-tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "how": "pipelined: step i+1's inputs copied in and step i's results copied out on their own streams "
                       "while step i compacts (two buffer sets); L2 not flushed inside this loop",
                "serial_value": round(serial_value, 1)},
        "gpu_launches": int(launches),
        "roofline": roof,
        "stages": per_stage,
        "cpu_baseline": cpu,
        "decode": decode,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def _traffic_for(stage, cfg):
    """DRAM bytes per call of `stage` from the committed ncu summaries
    (profiles/traffic_*.txt: lines "stage configN bytes"), if any."""
    pdir = os.path.join(ROOT, "profiles")
    try:
        names = sorted(f for f in os.listdir(pdir) if f.startswith("traffic_") and f.endswith(".txt"))
    except OSError:
        return None
    for name in names:
        try:
            with open(os.path.join(pdir, name)) as fh:
                for line in fh:
                    parts = line.split()
                    if line.startswith("#") or len(parts) != 3:
                        continue
                    if parts[0] == stage and parts[1] == f"config{cfg}":
                        return int(parts[2])
        except (OSError, ValueError):
            continue
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=3, choices=sorted(WORKLOADS))
    ap.add_argument("--layers", type=int, default=0,
                    help="keep only the first L layers of a multi-layer workload (profiling captures)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--select", default="rms", choices=["rms", "omp", "tam"],
                    help="key selection: highest RMS attention (default), orthogonal matching pursuit, or "
                         "thought-aware segment budgets with pivots (window of the last 128 tokens, c = 16)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
