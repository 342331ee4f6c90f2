#!/usr/bin/env python
"""Benchmark of the attention core under selective activation recomputation.

One step = forward (S = QK^T with causal mask and scale, softmax, softmax
dropout, O = P_d V, LSE) plus the recompute-backward (dQ with the row
statistics, then dK/dV) over one batch of synthetic bf16 inputs of the named workload, through the
library's C ABI.  Default workload: the GPT-3-style 175B layer, one
tensor-parallel rank's shard (b=2, 12 local heads, s=2048, d_head=128,
causal, p=0.1).

Prints one JSON line (rank 0).  Metric: combined fwd + recompute-bwd
TFLOP/s with algorithmic FLOPs 14 d b h s(s+1)/2 (fwd 4, bwd 10: the
recomputed QK^T plus dV, dP, dQ, dK), and its share of the measured dense
BF16 tensor peak.

--impl reference runs the CPU oracle on the host cores instead (rank 0 only),
each step a bounded sample (query and key rows) of the same workload.

Multi-GPU (torchrun): every rank runs its own replica of the workload (the
core shards by independent heads; no collective on the data path), so work
per GPU is fixed ("scaling": "weak") and value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024


def _flops(w) -> dict:
    pairs = w["s"] * (w["s"] + 1) // 2
    u = w["d"] * pairs * w["b"] * w["h_q"]
    return {"fwd": 4 * u, "bwd": 10 * u, "total": 14 * u, "model": 12 * u,
            # algorithmic FLOPs of each kernel's launch: the backward's 10 d per pair
            # (recomputed S, dP, dV, dQ, dK) split between its two kernels, the
            # recomputed S and dP that both need counted half to each
            "k_fwd": 4 * u, "k_dkdv": 6 * u, "k_dq": 4 * u}


def job_ms(ms: float, dist, device) -> float:
    """The job's time: the slowest rank's (max over ranks; one rank: its own)."""
    if dist is None:
        return ms
    import torch
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_tflops(units_per_rank_step: float, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed (each rank runs the
    same workload on its own inputs) over the job's time."""
    return units_per_rank_step * steps * world / (ms / 1e3) / 1e12


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"bf16_tflops": float(pk["bf16_tflops"]), "hbm_gbs": float(pk["hbm_gbs"]),
                "source": "measured"}
    return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "source": "fallback"}


def _strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines (the kernel sources
    hold no string literal with a comment marker in it)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip())


def _csrc_hash() -> str:
    """Hash of the kernel sources, comments aside: a profile taken on them stays
    valid until their code changes."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_core_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            h.update(fn.encode())
            h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()[:12]


def _traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/traffic.txt, if taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = _csrc_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload and parts[3] == cur:
                return int(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the GPU is busy."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.dev = dev_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _workload(name):
    from attention_core_gb300.inputs import WORKLOADS
    w = dict(WORKLOADS[name])
    w["name"] = name
    return w


def _config(w, extra=None):
    c = {"workload": w["name"], "b": w["b"], "h_q": w["h_q"], "h_kv": w["h_kv"], "s": w["s"],
         "d_head": w["d"], "causal": True, "p_drop": w["p_drop"]}
    if extra:
        c.update(extra)
    return c


# ------------------------------------------------------------- CPU oracle --

def _oracle_sample(w, budget_s: float, seed: int):
    """Time the oracle on a bounded sample of the workload: forward and dQ for a
    set R of query rows, dK/dV for a set C of key rows, all of one KV group.
    The 14 d FLOPs of each causal pair (i, j) are credited as 10 d to query row
    i (QK^T and P.V forward; QK^T, dP and dQ backward) and 4 d to key row j (dV,
    dK), so whole rows of both sets add up to the workload's count.
    Returns (seconds, credited flops, threads, description)."""
    import numpy as np

    import oracle
    from attention_core_gb300.inputs import random_inputs
    s, d, g = w["s"], w["d"], w["h_q"] // w["h_kv"]
    t = random_inputs(1, g, 1, s, d, seed=seed)
    q, k, v, dout = (x.double().numpy() for x in (t.q, t.k, t.v, t.dout))
    pr = oracle.Problem(b=1, h_q=g, h_kv=1, s=s, d=d, causal=True, p_drop=w["p_drop"], seed=seed)
    oracle.build()

    def run(n):
        rows = np.arange(n, dtype=np.int64) * 7919 % s            # spread over the sequence
        heads = np.arange(n, dtype=np.int64) % g
        krows = np.linspace(s - max(1, s // 16), s - 1, max(1, n // 4)).astype(np.int64)
        kheads = np.zeros(len(krows), dtype=np.int64)
        t0 = time.perf_counter()
        oracle.fwd_rows(pr, q, k, v, heads, rows)
        oracle.dq_rows(pr, q, k, v, dout, heads, rows)
        oracle.dkdv_rows(pr, q, k, v, dout, kheads, krows)
        dt = time.perf_counter() - t0
        flops = 10 * d * int((rows + 1).sum()) + 4 * d * g * int((s - krows).sum())
        return dt, flops, f"{n} query rows and {len(krows)} key rows of one KV group"

    n = 32
    dt, flops, desc = run(n)
    while dt < budget_s / 2 and n < 512 * s * g:
        n = int(n * min(16.0, max(2.0, budget_s / max(dt, 1e-3))))
        dt, flops, desc = run(n)
    return dt, flops, len(os.sched_getaffinity(0)), desc


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup):
        _oracle_sample(w, per_step, seed=1 + i)
    tot_t, tot_f, threads, desc = 0.0, 0, 1, ""
    for i in range(args.steps):
        dt, fl, threads, desc = _oracle_sample(w, per_step, seed=100 + i)
        tot_t += dt
        tot_f += fl
    val = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": "attn-core fwd+recompute-bwd TFLOP/s", "value": val,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w, {"sample_per_step": desc}),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc + " per step", "cpu": _cpu_model()},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU ----

def run_ours(args, w):
    import secrets

    import torch

    import attention_core_gb300 as ac
    from attention_core_gb300 import build as lib_build
    from attention_core_gb300.inputs import random_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    if rank == 0:
        lib_build.build()
    if dist is not None:
        dist.barrier()
    ac.load_library()

    b, hq, hkv, s, d, p = w["b"], w["h_q"], w["h_kv"], w["s"], w["d"], w["p_drop"]
    fl = _flops(w)
    seed = secrets.randbits(63)
    base = random_inputs(b, hq, hkv, s, d, seed=rank)
    per_set = 2 * (4 * b * hq * s * d + 4 * b * hkv * s * d) + 4 * b * hq * s
    pr = ac.Params(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=True, p_drop=p, seed=seed)
    ws_bytes = ac.attn_core_bwd_workspace_bytes(pr)
    per_set += ws_bytes
    n_sets = max(1, math.ceil(3 * L2_BYTES / per_set))
    sets = []
    for i in range(n_sets):
        q, k, v, g = (x.to(dev) for x in (base.q, base.k, base.v, base.dout))
        sets.append({
            "q": q, "k": k, "v": v, "dout": g, "o": torch.empty_like(q),
            "lse": torch.empty((b, hq, s), dtype=torch.float32, device=dev),
            "dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
            "ws": torch.empty(ws_bytes, dtype=torch.uint8, device=dev)})
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def step(ts, ev_ptr=0, on=None):
        sh = (on if on is not None else stream).cuda_stream
        pr.dev_status = status.data_ptr()
        pr.timing_events = ev_ptr
        rc = ac.attn_core_fwd(pr, ts["q"].data_ptr(), ts["k"].data_ptr(), ts["v"].data_ptr(),
                              ts["o"].data_ptr(), ts["lse"].data_ptr(), sh)
        if rc:
            raise ac.AttnCoreError(rc, "attn_core_fwd")
        pr.timing_events = ev_ptr + 2 * ctypes.sizeof(ctypes.c_void_p) if ev_ptr else 0
        rc = ac.attn_core_bwd_recompute(
            pr, ts["q"].data_ptr(), ts["k"].data_ptr(), ts["v"].data_ptr(), ts["o"].data_ptr(),
            ts["lse"].data_ptr(), ts["dout"].data_ptr(), ts["dq"].data_ptr(),
            ts["dk"].data_ptr(), ts["dv"].data_ptr(), ts["ws"].data_ptr(), ws_bytes, sh)
        if rc:
            raise ac.AttnCoreError(rc, "attn_core_bwd_recompute")

    for i in range(args.warmup):
        step(sets[i % n_sets])
    torch.cuda.synchronize(dev)

    # per-kernel events (fwd, dq, dkdv: 6 per timed step) on every EVERY-th step of
    # the timed region: an event between two launches costs about 2 us of GPU
    # time, so recording them on every step would slow the very loop they time
    K = args.steps
    NE = 6
    EVERY = 4
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(NE * K)]
    for e in evs:              # torch creates the CUDA event at its first record
        e.record(stream)
    torch.cuda.synchronize(dev)
    ev_arr = (ctypes.c_void_p * (NE * K))(*[e.cuda_event for e in evs])
    ev_base = ctypes.addressof(ev_arr)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    t_start.record(stream)
    for i in range(K):
        step(sets[i % n_sets], ev_base + NE * i * ctypes.sizeof(ctypes.c_void_p) if i % EVERY == 0 else 0)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} during the timed region")
    elapsed_ms = job_ms(t_start.elapsed_time(t_end), dist, dev)

    names = ["fwd", "dq", "dkdv"]
    kt = {n: [] for n in names}
    for i in range(0, K, EVERY):
        for j, n in enumerate(names):
            kt[n].append(evs[NE * i + 2 * j].elapsed_time(evs[NE * i + 2 * j + 1]))
    kavg = {n: sum(v) / len(v) for n, v in kt.items()}
    fwd_ms = kavg["fwd"]
    bwd_ms = kavg["dkdv"] + kavg["dq"]

    pk = _peaks()
    value = job_tflops(fl["total"], K, world, elapsed_ms)
    dom = max(("fwd", "dkdv", "dq"), key=lambda n: kavg[n])
    dom_flops = fl["k_" + dom]
    achieved = dom_flops / (kavg[dom] / 1e3) / 1e12
    kname = {"fwd": "attn_fwd_kernel", "dkdv": "attn_bwd_dkdv_kernel", "dq": "attn_bwd_dq_kernel"}[dom]

    # the same steps captured once into a CUDA graph and replayed (no per-kernel
    # events: they cannot be captured)
    graph = None
    if not args.no_graph:
        graph = _graph_replay(args, sets, step, n_sets, dev, fl, world, dist, status)

    # the dropout + residual add + layer norm block of the same layer (its own field)
    dal = None
    if not args.no_dal and rank == 0:
        dal = _dal_measure(dev, stream)

    # the layer around the core: recompute overhead of the core against the whole layer
    layer_study = None
    if not args.no_layer and rank == 0:
        layer_study = _layer_study(dev, stream)

    # every workload configuration, timed in this run
    per_config = None
    if not args.no_per_config and rank == 0:
        per_config = _per_config(dev, stream)

    # a packed batch of mixed lengths, one launch per kernel
    varlen = None
    if not args.no_varlen and rank == 0:
        varlen = _varlen_bench(dev, stream)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(args, w, pr, base, dev, stream, ws_bytes, fl, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, cflops, threads, desc = _oracle_sample(w, args.cpu_seconds, seed=7)
        cpu = {"value": cflops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{desc} ({dt:.1f} s)", "cpu": _cpu_model()}

    if rank == 0:
        line = {
            "metric": "attn-core fwd+recompute-bwd TFLOP/s", "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": elapsed_ms / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": _config(w, {"philox_seed": seed, "l2": f"{n_sets} rotating input sets of "
                                  f"{per_set / 2**20:.0f} MiB (> L2)", "parallelism":
                                  f"replicas x{world}" if world > 1 else "single GPU"}),
            "pct_of_bf16_peak": 100.0 * value / world / pk["bf16_tflops"],
            "fwd_tflops": fl["fwd"] / (fwd_ms / 1e3) / 1e12,
            "bwd_tflops": fl["bwd"] / (bwd_ms / 1e3) / 1e12,
            "model_flops_tflops": fl["model"] * K * world / (elapsed_ms / 1e3) / 1e12,
            "kernel_ms": {n: round(v, 4) for n, v in kavg.items()},
            "wall_ms_per_step": wall / K * 1e3,
            "roofline": {"bound": "tensor", "kernel": kname, "achieved": achieved,
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / pk["bf16_tflops"],
                         "peak_source": pk["source"] + " (burst)",
                         "traffic": _traffic(kname, w["name"])},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "cuda_graph": graph,
            "dropout_add_ln": dal,
            "layer_study": layer_study,
            "per_config": per_config,
            "varlen": varlen,
            "bwd_workspace_bytes": ws_bytes,
            "gpu_launches": 3 * K,
            "kernel_ms_sampled": f"per-kernel events on every {EVERY}th timed step ({len(kt['fwd'])} samples)",
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


PER_CONFIG = ["tiny", "gpt22b", "gpt175b", "gpt530b", "llama70b_p0", "llama70b_p01"]


def _core_bytes(w) -> dict:
    """Algorithmic HBM bytes of one step: the forward reads Q, K, V and writes
    O and the LSE; the backward reads Q, K, V, O, dO and the LSE and writes dQ,
    dK, dV (bf16 tensors, fp32 LSE)."""
    q = 2 * w["b"] * w["h_q"] * w["s"] * w["d"]
    kv = 2 * w["b"] * w["h_kv"] * w["s"] * w["d"]
    lse = 4 * w["b"] * w["h_q"] * w["s"]
    return {"fwd": q + 2 * kv + q + lse, "bwd": 3 * q + 2 * kv + lse + q + 2 * kv}


def _per_config(dev, stream, steps: int = 20, warmup: int = 3):
    """Every workload configuration, timed in this run: the whole step with
    events around `steps` back-to-back steps, and each kernel with the ABI's
    timing events on a second pass of `steps` steps.  Inputs rotate over sets
    larger than L2 in total.  TFLOP/s are algorithmic (fwd 4 d, bwd 10 d per
    visible pair); the tiny configuration is latency-bound and also reports
    its algorithmic bytes over the step time."""
    import torch

    import attention_core_gb300 as ac
    from attention_core_gb300.inputs import random_inputs
    pk = _peaks()
    out = {}
    for name in PER_CONFIG:
        w = _workload(name)
        b, hq, hkv, s, d, p = w["b"], w["h_q"], w["h_kv"], w["s"], w["d"], w["p_drop"]
        fl = _flops(w)
        pr = ac.Params(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=True, p_drop=p, seed=0x5EED + len(out))
        ws_bytes = ac.attn_core_bwd_workspace_bytes(pr)
        base = random_inputs(b, hq, hkv, s, d, seed=PER_CONFIG.index(name))
        per_set = 2 * (4 * b * hq * s * d + 4 * b * hkv * s * d) + 4 * b * hq * s + ws_bytes
        n_sets = max(1, math.ceil(3 * L2_BYTES / per_set))
        sets = []
        for _ in range(n_sets):
            q, k, v, g = (x.to(dev) for x in (base.q, base.k, base.v, base.dout))
            sets.append(dict(q=q, k=k, v=v, g=g, o=torch.empty_like(q),
                             lse=torch.empty((b, hq, s), dtype=torch.float32, device=dev),
                             dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                             ws=torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)))
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        pr.dev_status = status.data_ptr()
        sh = stream.cuda_stream

        def step(t, ev=0):
            pr.timing_events = ev
            rc = ac.attn_core_fwd(pr, t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), t["o"].data_ptr(),
                                  t["lse"].data_ptr(), sh)
            if rc:
                raise ac.AttnCoreError(rc, "attn_core_fwd")
            pr.timing_events = ev + 2 * ctypes.sizeof(ctypes.c_void_p) if ev else 0
            rc = ac.attn_core_bwd_recompute(pr, t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                                            t["o"].data_ptr(), t["lse"].data_ptr(), t["g"].data_ptr(),
                                            t["dq"].data_ptr(), t["dk"].data_ptr(), t["dv"].data_ptr(),
                                            t["ws"].data_ptr(), ws_bytes, sh)
            if rc:
                raise ac.AttnCoreError(rc, "attn_core_bwd_recompute")

        for i in range(warmup):
            step(sets[i % n_sets])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for i in range(steps):
            step(sets[i % n_sets])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(6 * steps)]
        for e in evs:
            e.record(stream)
        torch.cuda.synchronize(dev)
        arr = (ctypes.c_void_p * len(evs))(*[e.cuda_event for e in evs])
        for i in range(steps):
            step(sets[i % n_sets], ctypes.addressof(arr) + 6 * i * ctypes.sizeof(ctypes.c_void_p))
        torch.cuda.synchronize(dev)
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item()):#x} in configuration {name}")
        kms = {}
        for j, kn in enumerate(("fwd", "dq", "dkdv")):
            kms[kn] = sum(evs[6 * i + 2 * j].elapsed_time(evs[6 * i + 2 * j + 1]) for i in range(steps)) / steps
        fwd_ms, bwd_ms = kms["fwd"], kms["dq"] + kms["dkdv"]
        tf = fl["total"] / (ms / 1e3) / 1e12
        entry = {"b": b, "h_q": hq, "h_kv": hkv, "s": s, "d_head": d, "p_drop": p,
                 "ms_per_step": ms, "kernel_ms": {k: round(v, 4) for k, v in kms.items()},
                 "fwd_tflops": fl["fwd"] / (fwd_ms / 1e3) / 1e12,
                 "bwd_tflops": fl["bwd"] / (bwd_ms / 1e3) / 1e12,
                 "combined_tflops": tf, "pct_of_bf16_peak": 100.0 * tf / pk["bf16_tflops"],
                 "bwd_workspace_bytes": ws_bytes, "steps": steps, "input_sets": n_sets}
        if name == "tiny":
            cb = _core_bytes(w)
            entry["gbs"] = (cb["fwd"] + cb["bwd"]) / (ms / 1e3) / 1e9
            entry["pct_of_hbm"] = 100.0 * entry["gbs"] / pk["hbm_gbs"]
        out[name] = entry
        del sets
        torch.cuda.empty_cache()
    return out


def _dal_measure(dev, stream, iters: int = 30):
    """Dropout + residual add + layer norm at the 175B layer's residual boundary
    (s * b = 4096 tokens of h = 12288, p = 0.1): forward and backward, each timed
    alone with CUDA events on its stream, inputs (100 MB per tensor) larger than
    L2.  Algorithmic bytes: forward reads x and the residual and writes z and y
    (8 n h) plus mean, rstd, gamma and beta; backward reads dy, z and dz_next and
    writes dx and d_residual (10 n h) plus mean, rstd, gamma, dgamma and dbeta."""
    import secrets

    import torch

    import attention_core_gb300 as ac
    from attention_core_gb300.inputs import DAL_WORKLOADS, dal_inputs
    w = DAL_WORKLOADS["gpt175b"]
    n, h, p = w["n_rows"], w["hidden"], w["p_drop"]
    t = dal_inputs(n, h, seed=11)
    x, r, dy, dzn = (v.to(dev) for v in (t.x, t.residual, t.dy, t.dz_next))
    g, b = t.gamma.to(dev), t.beta.to(dev)
    kw = dict(p_drop=p, seed=secrets.randbits(63), offset=0)
    z, y, mean, rstd = ac.dropout_add_ln_fwd(x, r, g, b, **kw)
    ws = torch.empty(ac.attn_core_dropout_add_ln_bwd_workspace_bytes(ac.DalParams(n, h, p)),
                     dtype=torch.uint8, device=dev)
    fwd_bytes = 8 * n * h + 8 * n + 8 * h
    bwd_bytes = 10 * n * h + 8 * n + 12 * h
    pk = _peaks()
    out = {"workload": f"{n} tokens x hidden {h} (175B layer, s=2048, b=2), p={p}"}
    for name, fn, nbytes in (
            ("fwd", lambda: ac.dropout_add_ln_fwd(x, r, g, b, **kw), fwd_bytes),
            ("bwd", lambda: ac.dropout_add_ln_bwd(dy, z, mean, rstd, g, dz_next=dzn, workspace=ws, **kw),
             bwd_bytes)):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        torch.cuda.synchronize()
        for e0, e1 in evs:
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = sorted(e0.elapsed_time(e1) for e0, e1 in evs)[iters // 2]
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"us": ms * 1e3, "roofline": {
            "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / pk["hbm_gbs"], "peak_source": pk["source"], "bytes": nbytes,
            "traffic": _traffic("dal_" + name + "_kernel", "gpt175b_dal")}}
    return out


VARLEN = {"n_seq": 64, "min_len": 64, "max_len": 4096, "h_q": 12, "h_kv": 12, "d": 128, "p_drop": 0.1,
          "len_seed": 64}


def _varlen_bench(dev, stream, steps: int = 20, warmup: int = 3):
    """A packed batch of mixed lengths, one launch per kernel: 64 sequences of
    lengths drawn uniformly from 64 .. 4096 (seeded), heads shaped as the 175B
    shard (12 heads of 128, causal, p = 0.1).  Forward and backward are timed
    with events around each call over `steps` steps; TFLOP/s are algorithmic
    (fwd 4 d, bwd 10 d per visible pair, summed over the sequences)."""
    import random

    import torch

    import attention_core_gb300 as ac
    pk = _peaks()
    c = VARLEN
    rng = random.Random(c["len_seed"])
    lens = [rng.randint(c["min_len"], c["max_len"]) for _ in range(c["n_seq"])]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    total, hq, hkv, d = cu[-1], c["h_q"], c["h_kv"], c["d"]
    gen = torch.Generator(device="cpu").manual_seed(c["len_seed"])
    q, g = (torch.randn((total, hq, d), generator=gen).to(torch.bfloat16).to(dev) for _ in range(2))
    k, v = (torch.randn((total, hkv, d), generator=gen).to(torch.bfloat16).to(dev) for _ in range(2))
    o, dq = torch.empty_like(q), torch.empty_like(q)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    lse = torch.empty((hq, total), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pr = ac.Params(b=1, h_q=hq, h_kv=hkv, s=1, d=d, causal=True, p_drop=c["p_drop"], seed=0x7A12,
                   dev_status=status.data_ptr())
    tq, _, cq_dev, _ = ac._device_tables(cu, None, dev)
    ws_bytes = ac.attn_core_bwd_varlen_workspace_bytes(pr, cu, None, cu_q_dev=cq_dev)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    sh = stream.cuda_stream

    def fwd():
        rc = ac.attn_core_fwd_varlen(pr, cu, None, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), sh, cu_q_dev=cq_dev)
        if rc:
            raise ac.AttnCoreError(rc, "attn_core_fwd_varlen")

    def bwd():
        rc = ac.attn_core_bwd_varlen(pr, cu, None, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), g.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                     ws.data_ptr(), ws_bytes, sh, cu_q_dev=cq_dev)
        if rc:
            raise ac.AttnCoreError(rc, "attn_core_bwd_varlen")

    for _ in range(warmup):
        fwd()
        bwd()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(3 * steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        evs[3 * i].record(stream)
        fwd()
        evs[3 * i + 1].record(stream)
        bwd()
        evs[3 * i + 2].record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} in the packed batch")
    fwd_ms = sum(evs[3 * i].elapsed_time(evs[3 * i + 1]) for i in range(steps)) / steps
    bwd_ms = sum(evs[3 * i + 1].elapsed_time(evs[3 * i + 2]) for i in range(steps)) / steps
    u = sum(n * (n + 1) // 2 for n in lens) * d * hq
    tf = 14 * u / ((fwd_ms + bwd_ms) / 1e3) / 1e12
    return {"n_seq": c["n_seq"], "lengths": f"uniform {c['min_len']}..{c['max_len']} (seed {c['len_seed']})",
            "total_tokens": total, "max_len": max(lens), "h_q": hq, "h_kv": hkv, "d_head": d, "causal": True,
            "p_drop": c["p_drop"], "ms_per_step": fwd_ms + bwd_ms, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_tflops": 4 * u / (fwd_ms / 1e3) / 1e12, "bwd_tflops": 10 * u / (bwd_ms / 1e3) / 1e12,
            "combined_tflops": tf, "pct_of_bf16_peak": 100.0 * tf / pk["bf16_tflops"],
            "launches_per_step": 3, "bwd_workspace_bytes": ws_bytes, "steps": steps,
            "l2": f"{(2 * total * (hq + hkv) * d * 2) / 2**20:.0f} MiB of inputs (> L2)"}


def _layer_study(dev, stream, iters: int = 10):
    """One 175B-shaped layer shard (b=2, s=2048, h=12288, 12 local heads of 128,
    MLP width 6144, p=0.1) through attention_core_gb300.layer, three training
    steps each timed (median of `iters` CUDA-event timings on the stream):
      none       -- no recomputation: the core keeps its probabilities, mask and
                    dropout output (layer.StoredCore, 5 a s^2 b bytes) and the
                    backward reads them;
      selective  -- this library's core: the forward keeps Q, K, V, O and the
                    LSE, and the backward recomputes scores, probabilities and
                    mask on chip;
      full       -- only the layer input is kept: the backward reruns the whole
                    layer forward first (layer.backward_full).
    The overheads are ratios of these measured step times to the step without
    recomputation."""
    import torch

    import attention_core_gb300 as ac
    from attention_core_gb300 import layer
    sh = layer.LayerShape(b=2, s=2048, h=12288, a=12, d=128, ffn=6144, p_drop=0.1)
    w = layer.init_weights(sh, seed=3, device=dev)
    gen = torch.Generator(device="cpu").manual_seed(4)
    y_in, r_in, dy2, dz2 = (torch.randn((sh.n, sh.h), generator=gen).to(torch.bfloat16).to(dev)
                            for _ in range(4))
    seed = 12345

    def timed(fn):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        torch.cuda.synchronize()
        for e0, e1 in evs:
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return sorted(e0.elapsed_time(e1) for e0, e1 in evs)[iters // 2]

    stored = layer.StoredCore(sh)
    _, _, ctx = layer.forward(sh, w, y_in, r_in, seed=seed)
    fwd_ms = timed(lambda: layer.forward(sh, w, y_in, r_in, seed=seed))
    bwd_ms = timed(lambda: layer.backward(sh, w, ctx, dy2, dz2))
    core_ms = timed(lambda: ac.fwd(ctx["q"], ctx["k"], ctx["v"], **ctx["core"]))
    del ctx
    _, _, ctx_n = layer.forward(sh, w, y_in, r_in, seed=seed, stored=stored)
    fwd_none_ms = timed(lambda: layer.forward(sh, w, y_in, r_in, seed=seed, stored=stored))
    bwd_none_ms = timed(lambda: layer.backward(sh, w, ctx_n, dy2, dz2))
    del ctx_n
    bwd_full_ms = timed(lambda: layer.backward_full(sh, w, y_in, r_in, dy2, dz2, seed=seed))
    step_none = fwd_none_ms + bwd_none_ms
    step_sel = fwd_ms + bwd_ms
    step_full = fwd_ms + bwd_full_ms
    sb = ac.stored_bytes(sh.b, sh.a, sh.a, sh.s, sh.d)
    return {"workload": "175B layer shard: b=2, s=2048, h=12288, 12 local heads of 128, MLP 6144, "
                        "p=0.1; GEMMs by cuBLAS (torch.matmul), the rest by this library; the "
                        "no-recomputation core materialised with cuBLAS and PyTorch softmax/dropout",
            "step_ms": {"none": step_none, "selective": step_sel, "full": step_full},
            "fwd_ms": {"none": fwd_none_ms, "selective": fwd_ms, "full": fwd_ms},
            "bwd_ms": {"none": bwd_none_ms, "selective": bwd_ms, "full": bwd_full_ms},
            "core_fwd_ms": core_ms,
            "overhead_selective": step_sel / step_none - 1.0,
            "overhead_full": step_full / step_none - 1.0,
            "full_over_selective": step_full / step_sel - 1.0,
            "gemm_fwd_tflops": sh.gemm_flops_fwd() / (fwd_ms / 1e3) / 1e12,
            "activation_bytes_per_layer": {k: sb[k] for k in ("layer_none", "layer_selective", "layer_full")}}


def _graph_replay(args, sets, step, n_sets, dev, fl, world, dist, status):
    """The timed loop's steps (one per rotating input set) captured once into a
    CUDA graph and replayed, as a training loop that captures its step would run
    them: the launches go back to back without host round trips.  Timed with
    events on the replay stream around whole replays, inputs resident."""
    import torch
    side = torch.cuda.Stream(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        for i in range(n_sets):
            step(sets[i], on=side)
        side.synchronize()
        with torch.cuda.graph(g, stream=side):
            for i in range(n_sets):
                step(sets[i], on=side)
        for _ in range(3):
            g.replay()
        side.synchronize()
        reps = max(1, args.steps // n_sets)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        e0.record(side)
        for _ in range(reps):
            g.replay()
        e1.record(side)
        side.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} during the graph replays")
    ms = job_ms(e0.elapsed_time(e1), dist, dev)
    steps = reps * n_sets
    return {"value": job_tflops(fl["total"], steps, world, ms), "unit": "TFLOP/s",
            "steps": steps, "ms_per_step": ms / steps, "gpu_launches": 3 * steps}


def _e2e(args, w, pr, base, dev, stream, ws_bytes, fl, world, dist):
    """Same metric through the public API with host buffers: each step copies
    Q, K, V, dO from pinned host memory, runs fwd + bwd, and reads O, LSE, dQ,
    dK, dV back into pinned host memory.  Steps are pipelined the way a training
    loop would run them: step i+1's inputs go up and step i-1's outputs come
    back (one copy stream each way) while step i computes, on two alternating
    buffer sets ordered by events.  The timed region runs from the first upload
    to the last download, so every step's copies are inside it."""
    import torch

    import attention_core_gb300 as ac
    hq_in = {n: getattr(base, n).pin_memory() for n in ("q", "k", "v", "dout")}
    sets = []
    for _ in range(2):
        dv_in = {n: torch.empty_like(x, device=dev) for n, x in hq_in.items()}
        outs = {"o": torch.empty_like(dv_in["q"]), "dq": torch.empty_like(dv_in["q"]),
                "dk": torch.empty_like(dv_in["k"]), "dv": torch.empty_like(dv_in["v"]),
                "lse": torch.empty((w["b"], w["h_q"], w["s"]), dtype=torch.float32, device=dev)}
        host_out = {n: torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for n, x in outs.items()}
        ev = {k: torch.cuda.Event() for k in ("h2d", "comp", "d2h")}
        sets.append({"in": dv_in, "out": outs, "host": host_out, "ev": ev, "used": False})
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    h2d = sum(x.numel() * x.element_size() for x in hq_in.values())
    d2h = sum(x.numel() * x.element_size() for x in sets[0]["out"].values())
    pr.timing_events = 0
    s_up = torch.cuda.Stream(dev)
    s_down = torch.cuda.Stream(dev)
    sh = stream.cuda_stream

    def step(i):
        bs = sets[i % 2]
        dv_in, outs, ev = bs["in"], bs["out"], bs["ev"]
        with torch.cuda.stream(s_up):
            if bs["used"]:
                s_up.wait_event(ev["comp"])          # step i-2 has read these inputs
            for n in hq_in:
                dv_in[n].copy_(hq_in[n], non_blocking=True)
            ev["h2d"].record(s_up)
        stream.wait_event(ev["h2d"])
        if bs["used"]:
            stream.wait_event(ev["d2h"])             # step i-2's outputs are home
        rc = ac.attn_core_fwd(pr, dv_in["q"].data_ptr(), dv_in["k"].data_ptr(), dv_in["v"].data_ptr(),
                              outs["o"].data_ptr(), outs["lse"].data_ptr(), sh)
        if rc:
            raise ac.AttnCoreError(rc, "attn_core_fwd")
        rc = ac.attn_core_bwd_recompute(
            pr, dv_in["q"].data_ptr(), dv_in["k"].data_ptr(), dv_in["v"].data_ptr(),
            outs["o"].data_ptr(), outs["lse"].data_ptr(), dv_in["dout"].data_ptr(),
            outs["dq"].data_ptr(), outs["dk"].data_ptr(), outs["dv"].data_ptr(), ws.data_ptr(),
            ws_bytes, sh)
        if rc:
            raise ac.AttnCoreError(rc, "attn_core_bwd_recompute")
        ev["comp"].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev["comp"])
            for n in outs:
                bs["host"][n].copy_(outs[n], non_blocking=True)
            ev["d2h"].record(s_down)
        bs["used"] = True

    for i in range(max(3, args.warmup // 4)):
        step(i)
    torch.cuda.synchronize(dev)
    k2 = max(5, min(args.steps, 50))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    e0.record(stream)
    s_up.wait_stream(stream)
    for i in range(k2):
        step(i)
    stream.wait_stream(s_down)
    stream.wait_stream(s_up)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = job_ms(e0.elapsed_time(e1), dist, dev)
    return {"value": job_tflops(fl["total"], k2, world, ms), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k2,
            "ms_per_step": ms / k2, "pipelined": "uploads, compute and downloads of adjacent steps overlap"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gpt175b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay figure")
    ap.add_argument("--no-dal", action="store_true",
                    help="skip the dropout + residual add + layer norm measurement")
    ap.add_argument("--no-layer", action="store_true",
                    help="skip the layer-level recompute-overhead measurement")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other workload configurations")
    ap.add_argument("--no-varlen", action="store_true",
                    help="skip the packed mixed-length batch")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="time budget of the CPU-oracle baseline sample")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    w = _workload(args.workload)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
