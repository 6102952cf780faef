#!/usr/bin/env python
"""Benchmark of one residual-attention decode step.

Workload: one Llama-3-8B-shaped layer, 8 LoRA agents sharing a 32,768-token
bf16 base cache in 16-token pages (H_q=32, H_kv=8, d=128, rank 16), one
decode query per agent.  A step is one ``fk_residual_attention`` call: the
attention kernel plus the split-K combine.  Prints one JSON line.

The line also carries ``prefill``: the low-rank prefill a forked agent runs
over that shared prefix before its first decode step (``Lk = X A_k``,
``Lv = X A_v`` over the 32,768 prefix tokens, d_model 4096, rank 16, one
``fk_residual_prefill`` call), timed on its own with its own roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

N > 1 runs one independent replica per GPU (the path has no data exchange);
launch it with torch.distributed.run.  ``--impl reference`` times the CPU
oracle on the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "agent decode tokens/sec and achieved HBM GB/s, 8 agents × 32K shared ctx"
UNIT = "agent-tokens/s"
WORKLOAD = "llama8b_32k"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL_SOURCES = ("shared_base_kv_gb300/csrc/fk_decode.cu",
                  "shared_base_kv_gb300/csrc/fk_kernels.cu",
                  "shared_base_kv_gb300/csrc/fk_device.cuh",
                  "shared_base_kv_gb300/csrc/fk_internal.h")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_kernel_llama8b_32k.txt")
KERNEL8_SOURCES = ("shared_base_kv_gb300/csrc/fk_decode8.cu",
                   "shared_base_kv_gb300/csrc/fk_kernels.cu",
                   "shared_base_kv_gb300/csrc/fk_device.cuh",
                   "shared_base_kv_gb300/csrc/fk_internal.h")
TRAFFIC8_FILE = os.path.join(ROOT, "profiles", "decode8_kernel_llama8b_32k.txt")
PREFILL_SOURCES = ("shared_base_kv_gb300/csrc/fk_prefill.cu",
                   "shared_base_kv_gb300/csrc/fk_device.cuh",
                   "shared_base_kv_gb300/csrc/fk_internal.h")
PREFILL_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "prefill_kernel_llama8b_32k.txt")
PREFILL_SHAPE = {"n": 32768, "d_model": 4096, "rank": 16}


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def workload_desc(w) -> str:
    return (f"{w.name}: {w.n_layers} layer, {w.A} agents x {w.prefix} shared tokens "
            f"(+private 0), H_q={w.H_q}, H_kv={w.H_kv}, d={w.d}, r={int(w.ranks[0])}, "
            f"C={w.C}, page 16, bf16 pages and rCache")


def algorithmic_bytes(w) -> dict:
    """Bytes the step must move at least once: every live base page token
    (K and V) read once, all residual rows, q read and out written."""
    import numpy as np
    base = int(np.sum(w.slot_fill)) * w.H_kv * w.d * 2 * 2
    rc = int(np.sum(w.seq_lens.astype(np.int64) * w.ranks)) * 2 * 2
    qo = w.A * w.C * w.H_q * w.d * 2
    return {"bcache": base, "rcache": rc, "q": qo, "out": qo,
            "kernel": base + rc + qo, "step": base + rc + 2 * qo}


def measured_peak_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_peak_bf16():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def traffic_per_launch(path=TRAFFIC_FILE, sources=KERNEL_SOURCES):
    """dram read+write bytes per launch from the committed ncu summary, if it
    was taken on the current kernel sources."""
    try:
        vals = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    vals[k.strip()] = v.strip()
        if vals.get("kernel_source_sha256") != kernel_source_hash(sources):
            return None
        return int(float(vals["dram_bytes_per_launch"]))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle --

def oracle_rate(w, budget_s: float, n_pairs_max: int = 10 ** 9, keys: int = 0,
                first_pair: int = 0, pair_stride: int = 1):
    """Time the CPU oracle on (agent, kv-head) pairs of the workload.

    Each pair is 1/H_kv of an agent's decode token.  With ``keys`` > 0 the
    agents' contexts are cut to their first ``keys`` tokens and the units
    scaled by keys / T (cost is linear in the keys).  A worker of a pool
    takes pairs first_pair, first_pair + pair_stride, ...  Returns
    (agent-tokens per second, pairs done, seconds)."""
    import numpy as np
    import oracle
    ld = w.layer(0)
    pk = ld.pages_k.to(dtype=__import__("torch").float64).numpy()
    pv = ld.pages_v.to(dtype=__import__("torch").float64).numpy()
    seq = w.seq_lens.copy()
    lk, lv = ld.lk, ld.lv
    scale = 1.0
    if keys:
        seq = np.minimum(seq, keys).astype(np.int32)
        lk = [x[:keys] for x in lk]
        lv = [x[:keys] for x in lv]
        scale = float(keys) / float(w.seq_lens.max())
    pairs = [(a, h) for a in range(w.A) for h in range(w.H_kv)][first_pair::pair_stride]
    done, t0 = 0, time.perf_counter()
    while done < n_pairs_max and (time.perf_counter() - t0) < budget_s:
        a, h = pairs[done % len(pairs)]
        oracle.residual_attention(pk, pv, w.block_table, seq, lk, lv, ld.bk, ld.bv, ld.q,
                                  w.s, w.rope_base, w.causal, w.P, pairs=[(a, h)])
        done += 1
    dt = time.perf_counter() - t0
    return done * scale / w.H_kv / dt, done, dt


def _oracle_worker(job):
    """One process of the CPU baseline's pool: its own copy of the workload,
    every n-th (agent, kv-head) pair."""
    budget_s, first, stride = job
    import workloads
    w = workloads.make_workload(WORKLOAD)
    return oracle_rate(w, budget_s, first_pair=first, pair_stride=stride)


def cpu_baseline_child(budget_s: float, workers: int):
    """The oracle as it stands on the host's cores: one single-threaded
    process per core, each over its share of the (agent, kv-head) pairs;
    the job's rate is the sum of theirs."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        res = pool.map(_oracle_worker, [(budget_s, k, workers) for k in range(workers)])
    print(json.dumps({"value": sum(r[0] for r in res), "pairs": sum(r[1] for r in res),
                      "seconds": max(r[2] for r in res), "workers": workers}))


def run_cpu_baseline(budget_s: float = 15.0) -> dict:
    workers = max(1, min(os.cpu_count() or 1, 32))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child",
                        str(budget_s), "--cpu-workers", str(workers)], capture_output=True,
                       text=True, env=env, timeout=900)
    try:
        d = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return {"value": None, "unit": UNIT, "cores": workers, "kind": "oracle",
                "sample": f"failed: {r.stderr[-300:]}"}
    return {"value": d["value"], "unit": UNIT, "cores": d["workers"], "kind": "oracle",
            "sample": f"{d['pairs']} (agent, kv-head) pairs of the full workload at 32,768 keys "
                      f"in {d['seconds']:.1f} s, fp64 NumPy, {d['workers']} single-threaded "
                      f"processes (one per host core, BLAS pinned to 1 thread); a pair is 1/8 "
                      f"agent-token"}


# -------------------------------------------------------------- GPU arm --

def reduce_over_ranks(total_ms: float, e2e_ms: float, units: int, e2e_units: int, world: int,
                      device) -> tuple:
    """Whole-job throughput of N independent replicas: the units every rank
    processed divided by the slowest rank's time (max over ranks)."""
    import torch
    t = torch.tensor([total_ms, e2e_ms], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total_ms, e2e_ms = float(t[0]), float(t[1])
    return (units * world / (total_ms / 1e3), total_ms,
            e2e_units * world / (e2e_ms / 1e3), e2e_ms)


class L2Flush:
    """Between timed launches: write a buffer of twice the L2 size, then read
    another one, so that L2 holds none of the next launch's inputs and the
    write's dirty lines are written back before the launch's events start
    (left dirty, their write-back would be charged to the next kernel)."""

    def __init__(self, dev, l2_bytes: int):
        import torch
        self.w = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        self.r = torch.ones(2 * l2_bytes // 4, dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.r.sum()


def run_gb300(args, rank: int, world: int, local_rank: int):
    import numpy as np
    import torch
    import torch.distributed as dist
    import workloads
    from shared_base_kv_gb300 import (fk_last_launch_count, fk_pool_set_profile_event,
                                      fk_residual_attention, harness)
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workloads.make_workload(WORKLOAD)
    dw = harness.DeviceWorkload(w, device=f"cuda:{local_rank}")
    w.drop()
    q = dw.queries(0)
    out = torch.empty_like(q)
    agents = np.arange(w.A, dtype=np.int32)
    bt = np.ascontiguousarray(dw.block_table, dtype=np.int32)
    seq = np.ascontiguousarray(w.seq_lens, dtype=np.int32)
    stream = torch.cuda.current_stream(dev)
    h = dw.pool.h
    props = torch.cuda.get_device_properties(dev)
    flush = L2Flush(dev, int(getattr(props, "L2_cache_size", 128 << 20)))

    def step():
        fk_residual_attention(h, 0, q, agents, bt, seq, False, False, out, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches = 0
    for k in range(K):
        flush.zero_()                       # L2 flush between steps, outside the events
        ev_s[k].record(stream)
        step()
        ev_e[k].record(stream)
        launches += fk_last_launch_count(h)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [ev_s[k].elapsed_time(ev_e[k]) for k in range(K)]
    total_ms = sum(step_ms)
    # the attention kernel's own duration, for the roofline, from further
    # steps with an event recorded between it and the combine.  That event
    # makes the combine wait for the attention grid's end before it is even
    # launched (no programmatic overlap), so these steps are kept out of the
    # timed ones above.
    KM = max(1, min(K, 500))
    km_s = [torch.cuda.Event(enable_timing=True) for _ in range(KM)]
    km_m = [torch.cuda.Event(enable_timing=True) for _ in range(KM)]
    for e in km_m:
        e.record(stream)     # creates the event; the library re-records it after the main kernel
    torch.cuda.synchronize(dev)
    for k in range(KM):
        flush.zero_()
        fk_pool_set_profile_event(h, km_m[k])
        km_s[k].record(stream)
        step()
    torch.cuda.synchronize(dev)
    fk_pool_set_profile_event(h, None)
    main_ms = [km_s[k].elapsed_time(km_m[k]) for k in range(KM)]
    graph = graph_step_ms(dev, stream, flush, h, q, agents, bt, seq, out, min(K, 500))
    # end to end through the public call, host buffers: H2D q, call, D2H out
    q_host = q.cpu().pin_memory()
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_dev = torch.empty_like(q)
    KE = max(1, min(K, args.e2e_steps))
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(KE)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(KE)]
    for k in range(KE):
        flush.zero_()
        e_s[k].record(stream)
        q_dev.copy_(q_host, non_blocking=True)
        fk_residual_attention(h, 0, q_dev, agents, bt, seq, False, False, out, stream)
        out_host.copy_(out, non_blocking=True)
        e_e[k].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = sum(e_s[k].elapsed_time(e_e[k]) for k in range(KE))
    ok = bool(torch.isfinite(out.float()).all().item())
    dw.check()
    prefill = measure_prefill(dev, stream, flush, args.prefill_steps) if args.prefill_steps else None
    configs = measure_configs(dev, stream, flush) if (world == 1 and not args.no_configs) else None
    value, total_ms, e2e_value, e2e_ms = reduce_over_ranks(
        total_ms, e2e_ms, w.A * K, w.A * KE, world, dev)
    ab = algorithmic_bytes(w)
    slots8 = os.environ.get("FORKKV_DECODE_SLOTS") == "8"
    main_avg_s = statistics.mean(main_ms) / 1e3
    peak, peak_kind = measured_peak_hbm()
    achieved = ab["kernel"] / main_avg_s / 1e9
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w),
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed between steps, outside the step's events: a memset of 2x L2, "
                         "then a read of another 2x L2 buffer (writes back the dirty lines)",
                   "kernel_timing": "roofline.kernel_ms from separate steps with an event "
                                    "between the attention kernel and the combine",
                   "step_ms_p10_p50_p90": percentiles(step_ms),
                   "cuda_graph": graph,
                   "step_hbm_gbs": ab["step"] / (total_ms / K / 1e3) / 1e9,
                   "step_bytes": ab["step"]},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": (traffic_per_launch(TRAFFIC8_FILE, KERNEL8_SOURCES) if slots8
                                 else traffic_per_launch()),
                     "kernel": ("decode8_kernel" if slots8
                                else "mbuild_kernel<128> + decode_kernel<128,false>"),
                     "kernel_ms": statistics.mean(main_ms),
                     "bytes_per_launch": ab["kernel"],
                     "peak_kind": f"{peak_kind} hbm_gbs"},
        "e2e": {"value": e2e_value, "unit": UNIT,
                "h2d_bytes_per_step": int(q.numel() * q.element_size()),
                "d2h_bytes_per_step": int(out.numel() * out.element_size())},
        "gpu_launches": launches,
        "clocks": clk,
        "outputs_finite": ok,
        "prefill": prefill,
    }
    if configs is not None:
        res["configs"] = configs
    return res


def percentiles(ms) -> list:
    import numpy as np
    return [float(np.percentile(ms, p)) for p in (10, 50, 90)]


def graph_step_ms(dev, stream, flush, h, q, agents, bt, seq, out, steps: int) -> dict:
    """The same step captured once into a CUDA graph and replayed (the call's
    work list is cached, so the capture holds only its kernel launches)."""
    import torch
    from shared_base_kv_gb300 import fk_residual_attention
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fk_residual_attention(h, 0, q, agents, bt, seq, False, False, out, side)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g, stream=side):
            fk_residual_attention(h, 0, q, agents, bt, seq, False, False, out, side)
        torch.cuda.synchronize(dev)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = [e0.elapsed_time(e1) for e0, e1 in ev]
        return {"ms_per_step": statistics.mean(ms), "ms_p10_p50_p90": percentiles(ms),
                "steps": steps}
    except Exception as e:                      # a capture the runtime refuses
        return {"error": f"{type(e).__name__}: {str(e)[:200]}"}


def measure_configs(dev, stream, flush) -> list:
    """Absolute numbers for every workload (one fk_residual_attention call per
    layer; the 32-layer workload's step is its 32 calls).  Median and
    p10/p90 over L2-flushed iterations."""
    import numpy as np
    import torch
    import workloads
    from shared_base_kv_gb300 import fk_residual_attention, harness
    res = []
    # the last line is the headline workload with Shared-A agents (LRAgent
    # summary, "BaseLRShared"): all eight read agent 0's low-rank rows, so
    # the rCache bytes count once
    for name, comp, iters, shared in (("tiny", None, 200, False), ("llama8b_32k", None, 200, False),
                                      ("agents32_layers32", None, 30, False),
                                      ("qwen72b_chunk", None, 50, False),
                                      ("compressed", "gpu", 200, False),
                                      ("llama8b_32k", None, 200, True)):
        w = workloads.make_workload(name)
        if shared:
            for l in range(w.n_layers):
                ld = w.layer(l)
                for a in range(1, w.A):
                    ld.lk[a], ld.lv[a] = ld.lk[0], ld.lv[0]
        dw = harness.DeviceWorkload(w, device=str(dev), compressed=comp, shared_a=shared)
        qs = [dw.queries(l) for l in range(w.n_layers)]
        w.drop()
        out = torch.empty_like(qs[0])
        agents = np.arange(w.A, dtype=np.int32)
        bt = np.ascontiguousarray(dw.block_table, dtype=np.int32)
        seq = np.ascontiguousarray(w.seq_lens, dtype=np.int32)
        h = dw.pool.h

        def step():
            for l in range(w.n_layers):
                fk_residual_attention(h, l, qs[l], agents, bt, seq, w.causal, comp is not None,
                                      out, stream)

        for _ in range(3):
            step()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(iters)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        dw.check()
        ms = [e0.elapsed_time(e1) for e0, e1 in ev]
        p10, p50, p90 = percentiles(ms)
        ab = algorithmic_bytes(w)
        per_layer = ab["step"]
        if shared:                 # one low-rank cache for all agents
            per_layer -= ab["rcache"] - int(w.seq_lens[0]) * int(w.ranks[0]) * 2 * 2
        if comp is not None:     # int8 K (d B) + 3-bit V (3d/8 B) + fp32 norm per (token, head)
            per_layer = (int(np.sum(w.slot_fill)) * w.H_kv * (w.d + 3 * w.d // 8 + 4)
                         + ab["rcache"] + ab["q"] + ab["out"])
        G = w.H_q // w.H_kv
        flops = 0
        for a in range(w.A):     # per (agent, key, kv head): recon + scores + P Vb + P Lv; up-projection per row
            r = int(w.ranks[a])
            flops += w.H_kv * (int(w.seq_lens[a]) * (2 * r * w.d + G * w.C * (4 * w.d + 2 * r))
                               + G * w.C * 2 * r * w.d)
        flops *= w.n_layers
        gbs = per_layer * w.n_layers / (p50 / 1e3) / 1e9
        tflops = flops / (p50 / 1e3) / 1e12
        G = w.H_q // w.H_kv
        if G * w.C >= 128 and w.d == 128 and comp is None:
            kernel, bound = "chunk_kernel", "tensor"
        elif G * w.C == 4:
            eight = os.environ.get("FORKKV_DECODE_SLOTS") == "8" and w.d == 128 and comp is None
            kernel = "decode8_kernel" if eight else f"mbuild_kernel<{w.d}> + decode_kernel<{w.d},{int(comp is not None)}>"
            bound = "hbm"
        else:
            kernel, bound = f"attention_kernel<{w.d},{int(comp is not None)}>", "hbm"
        if bound == "tensor":
            pk, pkind = measured_peak_bf16()
            roof = {"bound": "tensor", "achieved": tflops, "peak": pk, "unit": "TFLOP/s",
                    "frac": tflops / pk, "peak_kind": f"{pkind} bf16_tflops (burst)"}
        else:
            pk, pkind = measured_peak_hbm()
            roof = {"bound": "hbm", "achieved": gbs, "peak": pk, "unit": "GB/s",
                    "frac": gbs / pk, "peak_kind": f"{pkind} hbm_gbs"}
        roof["kernel"] = kernel + " + combine_kernel"
        roof["timed"] = "whole step (every launch of the call), median"
        res.append({"workload": name + (" shared_a" if shared else ""), "layers": w.n_layers,
                    "agents": w.A, "C": w.C,
                    "ms_p50": p50, "ms_p10": p10, "ms_p90": p90,
                    "agent_tokens_per_s": w.A * w.C / (p50 / 1e3),
                    "algorithmic_bytes": per_layer * w.n_layers,
                    "gbs": gbs,
                    "algorithmic_tflop": flops / 1e12,
                    "tflops": tflops,
                    "compressed": comp is not None,
                    "roofline": roof})
        dw.pool.close()
        del dw, qs, out
        torch.cuda.empty_cache()
    return res


def measure_prefill(dev, stream, flush, steps: int) -> dict:
    """One forked agent's low-rank prefill over the shared prefix, timed
    with CUDA events on the launching stream (L2 flushed between launches,
    outside the events)."""
    import torch
    from shared_base_kv_gb300 import Pool, fk_agent_register, fk_check, fk_residual_prefill
    n, dm, r = PREFILL_SHAPE["n"], PREFILL_SHAPE["d_model"], PREFILL_SHAPE["rank"]
    pool = Pool(n_layers=1, n_q_heads=32, n_kv_heads=8, head_dim=128, num_pages=4,
                max_agents=1, max_rank=r, max_tokens=n)
    g = torch.Generator(device=dev).manual_seed(1234)
    B = torch.zeros(1, r, 8 * 128, dtype=torch.bfloat16, device=dev)
    fk_agent_register(pool.h, 0, r, 1.0, B, B)
    X = torch.randn(n, dm, generator=g, device=dev).to(torch.bfloat16)
    Ak = (torch.randn(dm, r, generator=g, device=dev) / dm ** 0.5).to(torch.bfloat16)
    Av = (torch.randn(dm, r, generator=g, device=dev) / dm ** 0.5).to(torch.bfloat16)
    for _ in range(3):
        fk_residual_prefill(pool.h, 0, 0, 0, X, Ak, Av, stream)
    torch.cuda.synchronize(dev)
    # all launches are enqueued before one synchronize, so the host's own
    # call overhead overlaps the flush and never sits inside the events
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        fk_residual_prefill(pool.h, 0, 0, 0, X, Ak, Av, stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    fk_check(pool.h, stream)
    pool.close()
    avg = statistics.mean(ms)
    algo = n * dm * 2 + 2 * dm * r * 2 + 2 * n * r * 2
    peak, peak_kind = measured_peak_hbm()
    achieved = algo / (avg / 1e3) / 1e9
    return {
        "workload": f"one agent's low-rank prefill over {n} shared prefix tokens, "
                    f"d_model {dm}, rank {r}: X [{n}, {dm}] bf16 times A_k, A_v [{dm}, {r}]",
        "ms": avg, "launches": steps,
        "tokens_per_s": n / (avg / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": traffic_per_launch(PREFILL_TRAFFIC_FILE, PREFILL_SOURCES),
                     "kernel": f"lr_prefill_kernel<{r}>", "bytes_per_launch": algo,
                     "peak_kind": f"{peak_kind} hbm_gbs"},
    }


def run_chunk_small(args) -> dict:
    """The chunk kernel's call on a reduced Qwen-72B-shaped causal chunk (16
    agents, 16,384 shared prefix tokens + 32 private, C = 32): a case small
    enough to profile whole (its launches hold about 1 GB)."""
    import numpy as np
    import torch
    import workloads
    from shared_base_kv_gb300 import fk_residual_attention, harness
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev, int(torch.cuda.get_device_properties(dev).L2_cache_size))
    w = workloads.make_workload("qwen72b_chunk", prefix=16384, A=16)
    dw = harness.DeviceWorkload(w, device="cuda:0")
    q = dw.queries(0)
    w.drop()
    out = torch.empty_like(q)
    agents = np.arange(w.A, dtype=np.int32)
    bt = np.ascontiguousarray(dw.block_table, dtype=np.int32)
    seq = np.ascontiguousarray(w.seq_lens, dtype=np.int32)

    def step():
        fk_residual_attention(dw.pool.h, 0, q, agents, bt, seq, True, False, out, stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    dw.check()
    ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    return {"workload": "qwen72b_chunk reduced: 16 agents x (16384 + 32) tokens, C = 32 causal",
            "ms_p10_p50_p90": percentiles(ms), "steps": args.steps}


_REF = {}


def _ref_init(keys: int):
    """A worker of the reference arm's pool: the workload's first layer in
    float64, contexts cut to their first ``keys`` keys."""
    import numpy as np
    import torch
    import workloads
    w = workloads.make_workload(WORKLOAD)
    ld = w.layer(0)
    _REF.update(w=w, ld=ld, pk=ld.pages_k.to(torch.float64).numpy(),
                pv=ld.pages_v.to(torch.float64).numpy(),
                seq=np.minimum(w.seq_lens, keys).astype(np.int32),
                lk=[x[:keys] for x in ld.lk], lv=[x[:keys] for x in ld.lv])


def _ref_pair(pair):
    import oracle
    r = _REF
    w, ld = r["w"], r["ld"]
    oracle.residual_attention(r["pk"], r["pv"], w.block_table, r["seq"], r["lk"], r["lv"], ld.bk,
                              ld.bv, ld.q, w.s, w.rope_base, w.causal, w.P, pairs=[pair])
    return 1


def run_reference(args):
    """The oracle as it stands on the host's cores: a pool of single-threaded
    processes, one per core; each step runs one (agent, kv-head) pair per
    process, over contexts cut to a prefix sized so that the whole run ends
    within a few minutes, scaled to full-context agent-tokens."""
    import multiprocessing as mp
    import workloads
    w = workloads.make_workload(WORKLOAD)
    workers = max(1, min(os.cpu_count() or 1, 32))
    _, _, per_pair_1k = oracle_rate(w, 1e9, n_pairs_max=1, keys=1024)
    budget = 100.0    # seconds, sized on one process; concurrent processes share memory bandwidth
    n = args.steps + args.warmup
    T = int(w.seq_lens.max())
    keys = int(max(16, min(T, T * budget / max(1e-9, n * per_pair_1k * T / 1024.0))))
    keys = (keys // 16) * 16 or 16
    pairs = [(a, h) for a in range(w.A) for h in range(w.H_kv)]
    step_pairs = lambda k: [pairs[(k * workers + j) % len(pairs)] for j in range(workers)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers, initializer=_ref_init, initargs=(keys,)) as pool:
        for k in range(args.warmup):
            pool.map(_ref_pair, step_pairs(k), chunksize=1)
        t0 = time.perf_counter()
        for k in range(args.steps):
            pool.map(_ref_pair, step_pairs(args.warmup + k), chunksize=1)
        dt = time.perf_counter() - t0
    rate = args.steps * workers * (keys / T) / w.H_kv / dt
    res = {
        "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": workload_desc(w),
                   # the job being compared (the GPU arm's config); where it ran
                   # is in cpu_baseline
                   "parallelism": f"replicas x{int(os.environ.get('WORLD_SIZE', '1'))}"},
        "cpu_baseline": {"value": rate, "unit": UNIT, "kind": "oracle", "cores": workers,
                         "sample": f"each step: the fp64 oracle on {workers} (agent, kv-head) "
                                   f"pairs in parallel, one per process, over the first {keys} "
                                   f"of {T} keys, scaled to full-context agent-tokens ({keys}/{T} "
                                   f"x 1/{w.H_kv} per pair)"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--prefill-steps", type=int, default=100)
    ap.add_argument("--chunk-small", action="store_true",
                    help="only time the chunk kernel's call on a reduced Qwen-72B-shaped chunk")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing every workload (tiny, llama8b_32k, agents32_layers32, "
                         "qwen72b_chunk, compressed), whose numbers the default run adds "
                         "as 'configs' (at N=1)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-child", type=float, default=None)
    ap.add_argument("--cpu-workers", type=int, default=1)
    args = ap.parse_args()
    if args.cpu_baseline_child is not None:
        cpu_baseline_child(args.cpu_baseline_child, args.cpu_workers)
        return
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        os.environ["OMP_NUM_THREADS"] = os.environ.get("OMP_NUM_THREADS", "1")
        print(json.dumps(run_reference(args)), flush=True)
        return
    if args.chunk_small:
        import __graft_entry__
        __graft_entry__.build()
        print(json.dumps(run_chunk_small(args)), flush=True)
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline()          # before the first GPU call, in a fresh process
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    res = run_gb300(args, rank, world, local_rank)
    if cpu is not None:
        res["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
