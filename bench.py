#!/usr/bin/env python3
"""Benchmark of the fused per-token KV-cache write on GB300.

Default workload: MLA ragged prefill (16 requests, new lengths U[512,8192],
70,820 tokens with the benchmark seed, 128 q heads, 512 latent + 64 rope,
page 128, FP8 E4M3 cache out with scale 1.0), the largest configuration of
the MLA write.  A step is one call of ``kvw_mla_rope_rmsnorm_quant`` over that
batch: RoPE on q_rope and on the rope part, RMSNorm of the latent part, FP8
quantisation and the paged scatter.  The same run then measures, under the
line's ``also`` key, the MLA decode step (256 requests x 1 token, with its
end-to-end figure), the bf16-cache prefill, the GQA Q/K RoPE (bf16 and E4M3
K cache), the K-cache RMSNorm and the latent gather with dynamic FP8
launches the same way.  ``--workload`` picks another main workload.

Timing: W warm-up steps, then K timed steps between a barrier and a device
synchronize on both sides.  Each step's launch is bracketed by CUDA events on
the stream it is launched on; before every step the L2 is flushed (512 MiB
written, then 512 MiB read, so no input line is resident and no dirty line
is left to write back) unless the inputs are larger than L2.  Values are
whole-job throughput (tokens/s over all ranks, slowest rank's time).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead, on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gqa_kv_cache_mla_gb300 import workloads as W  # noqa: E402

METRIC = "MLA fused RoPE/RMSNorm/FP8 KV-write tokens/s; achieved HBM GB/s vs peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = W.REGISTRY
DEFAULT_SEED = 2
DEFAULT_WORKLOAD = "mla_prefill_fp8"
# measured after the main workload, in the same run, under the line's "also" key
DEFAULT_ALSO = ("mla_decode", "mla_prefill_bf16", "gqa_interleaved", "gqa_fp8k", "knorm128",
                "knorm64", "mla_gather_prefill_dynamic")
HEADLINE = ("mla_prefill_fp8", "mla_prefill_bf16", "mla_decode", "mla_decode_bf16")


def kind_of(w):
    """mla | gqa | kno | gather | codec, from the workload's type."""
    return {W.MLAWorkload: "mla", W.GQAWorkload: "gqa", W.KNormWorkload: "kno",
            W.GatherWorkload: "gather", W.ConvertWorkload: "codec"}[type(w)]


def combine_ranks(ms, tokens, world, device=None):
    """Replicas: the job's time is the slowest rank's, its work the sum of the
    ranks' tokens.  Only timing crosses ranks; there is no data collective."""
    if world == 1:
        return ms, tokens
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


def source_hash(kernel_file):
    """Hash of a kernel's source and of every shared device header."""
    csrc = os.path.join(ROOT, "gqa_kv_cache_mla_gb300", "csrc")
    h = hashlib.sha256()
    for f in [kernel_file] + sorted(x for x in os.listdir(csrc) if x.endswith(".cuh")):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel_file):
    """DRAM bytes per launch from the committed ncu summary, if it still
    describes the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "%s.md" % workload)
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    hs = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not hs or hs.group(1) != source_hash(kernel_file):
        return None
    return float(m.group(1))


def algorithmic_bytes(w, name=None):
    """Bytes one launch must move: every distinct byte read or written once."""
    k = kind_of(w)
    if k == "mla":
        c = w.cache
        pos = np.concatenate([c.cache_lengths[b] + np.arange(w.offsets[b + 1] - w.offsets[b])
                              for b in range(w.B)]) if w.T else np.zeros(0)
        q_out = 2 if w.q_out_dtype == W.DTYPE_BF16 else 1
        row_in = c.elem_bytes if w.inplace else 2  # in place: the row comes from the cache
        return (w.T * (w.H * W.MLA_ROPE_DIM * (2 + q_out) + W.MLA_ROW * (row_in + c.elem_bytes))
                + len(np.unique(pos)) * W.MLA_ROPE_DIM * 4)
    if k == "gqa":
        c = w.cache
        kb = c.elem_bytes
        if w.position_ids is None:
            rows = len(np.unique(np.concatenate(
                [c.cache_lengths[b] + np.arange(w.offsets[b + 1] - w.offsets[b])
                 for b in range(w.B)])))
            return W.algorithmic_bytes_gqa(w.T, w.q_proj.shape[1], c.num_heads, c.head_size, rows,
                                           kb)
        base = W.algorithmic_bytes_gqa(w.T, w.q_proj.shape[1], c.num_heads, c.head_size, 0, kb)
        if w.mrope_section is not None:  # each position row supplies only its section's pairs
            return base + sum(len(np.unique(w.position_ids[r])) * int(sec) * 8
                              for r, sec in enumerate(w.mrope_section))
        return base + len(np.unique(w.position_ids)) * c.head_size * 4
    if k == "kno":
        c = w.cache
        if not w.per_head_norm:  # one row of Hk*S values per token
            return W.algorithmic_bytes_knorm(w.T, 1, w.gamma.size)
        return W.algorithmic_bytes_knorm(w.T, c.num_heads, w.gamma.size)
    if k == "gather":
        out_b = 2 if w.out_dtype == W.DTYPE_BF16 else 1
        return w.rows * (W.MLA_ROW * (w.cache.elem_bytes + out_b) + (4 if w.dynamic else 0))
    if w.per_row:
        return w.x.size * 3 + w.x.shape[0] * 4
    return w.x.size * 3


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(w, name, budget_s, single_thread=True):
    """The oracle, as it is, on the host cores, over whole batches of the
    same workload until ``budget_s`` seconds of CPU time have elapsed."""
    import oracle

    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    if not oracle.has_openmp():
        threads = 1
    k = kind_of(w)
    if k == "mla":
        cache = w.cache.data.copy()  # written in place by every call (allocated once)
        q_out = np.zeros(w.q_rope.shape, np.uint16 if w.q_out_dtype == 0 else np.uint8)
        if w.inplace:
            fn = lambda: oracle.mla_rope_rmsnorm_inplace(w, q_rope_out=q_out, cache_data=cache,
                                                         nthreads=threads, out_dtype=w.q_out_dtype)
        else:
            fn = lambda: oracle.mla_rope_rmsnorm_quant(w, q_rope_out=q_out, cache_data=cache,
                                                       nthreads=threads, out_dtype=w.q_out_dtype)
    elif k == "gqa":
        cache = w.cache.data.copy()
        out = np.zeros_like(w.q_proj)
        fn = lambda: oracle.qk_rope_paged_ragged(w, output=out, cache_data=cache,
                                                 nthreads=threads)
    elif k == "kno":
        cache = w.cache.data.copy()
        fn = lambda: oracle.rms_norm_kv_cache_paged(w, cache_data=cache, nthreads=threads)
    elif k == "gather":
        threads = 1
        if w.dynamic:
            fn = lambda: oracle.mla_gather_latent_dynamic(w.cache, w.layer_idx, w.ctx_offsets)
        else:
            fn = lambda: oracle.mla_gather_latent(w.cache, w.layer_idx, w.ctx_offsets,
                                                  w.out_dtype, w.out_scale)
    else:
        threads = 1
        fn = ((lambda: oracle.quantize_rows_e4m3(w.x)) if w.per_row
              else (lambda: oracle.convert_bf16_to_e4m3(w.x, w.scale)))
    fn()  # warm: page in buffers

    def timed(f, budget):
        n, t0 = 0, time.perf_counter()
        while True:
            f()
            n += 1
            el = time.perf_counter() - t0
            if el >= budget:
                return n, el

    n, el = timed(fn, budget_s)
    tps = n * w.T / el
    res = {"value": tps, "unit": "tokens/s" if k not in ("gather", "codec") else "rows/s",
           "cores": threads, "kind": "oracle",
           "sample": "%d whole batches of %d units (%s), %.1f s wall" % (n, w.T, name, el),
           "gbs": algorithmic_bytes(w, name) * n / el / 1e9}
    if single_thread and threads > 1 and k in ("mla", "gqa", "kno"):
        # the same oracle on one thread, over a shorter bounded sample
        kw = {"out_dtype": w.q_out_dtype} if k == "mla" else {}
        one = {"mla": lambda: (oracle.mla_rope_rmsnorm_inplace if w.inplace
                               else oracle.mla_rope_rmsnorm_quant)(w, q_rope_out=q_out,
                                                                   cache_data=cache, nthreads=1,
                                                                   **kw),
               "gqa": lambda: oracle.qk_rope_paged_ragged(w, output=out, cache_data=cache,
                                                          nthreads=1),
               "kno": lambda: oracle.rms_norm_kv_cache_paged(w, cache_data=cache, nthreads=1)}[k]
        n1, el1 = timed(one, budget_s / 3)
        res["single_thread"] = {"value": n1 * w.T / el1, "cores": 1,
                                "sample": "%d whole batches, %.1f s wall" % (n1, el1)}
    return res


def unit_of(w):
    return "tokens/s" if kind_of(w) in ("mla", "gqa", "kno") else "rows/s"


def metric_of(name, unit):
    return METRIC if name in HEADLINE else "%s %s; achieved HBM GB/s vs peak" % (name, unit)


def config_of(name, w, world):
    """The workload description both arms print (identical keys and values)."""
    abytes = algorithmic_bytes(w, name)
    k = kind_of(w)
    fp8_out = (getattr(getattr(w, "cache", None), "dtype", 0) == W.DTYPE_FP8_E4M3
               or k == "codec" or (k == "gather" and w.out_dtype == W.DTYPE_FP8_E4M3))
    return {"workload": name + ": " + WORKLOADS[name][2], "tokens_per_gpu": int(w.T),
            "l2": ("flushed before every GPU step (512 MiB written, 512 MiB read)"
                   if abytes < 2 * L2_BYTES else
                   "inputs larger than L2 (%.2f GB per step)" % (abytes / 1e9)),
            "io": "bf16 in, fp32 arithmetic, %s out" % ("e4m3" if fp8_out else "bf16"),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    name = args.workload
    w = WORKLOADS[name][0](DEFAULT_SEED)
    import oracle

    oracle.build()
    times = []
    threads = None
    # keep the whole run within about two minutes whatever K and W are
    step_s = min(args.ref_step_s, 120.0 / (args.warmup + args.steps))
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(w, name, budget_s=step_s, single_thread=False)
        threads = cb["cores"]
        if i >= args.warmup:
            times.append(w.T / cb["value"])
    ms = 1000.0 * statistics.mean(times)
    value = w.T / (ms / 1000.0)
    unit = unit_of(w)
    line = {"impl": "reference",
            "metric": metric_of(name, unit),
            "value": value, "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; shapes and distributions of the benchmark configs)",
            "config": config_of(name, w, world),
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads,
                             "kind": "oracle",
                             "sample": "each step: whole %d-token batches for %.2f s" %
                                       (w.T, step_s)},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


class Flusher:
    """Evicts the L2 between timed steps: 512 MiB written, then 512 MiB read."""

    def __init__(self, dev):
        import torch

        self.fw = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.fr = torch.ones(128 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.fw.fill_(1)
        self.fr.sum()


def measure(name, steps, warmup, dev, rank, world, flusher, e2e=True, cpu_s=None,
            host_timing=True):
    """Device-timed throughput of one workload (and optionally its end-to-end
    figure and the oracle beside it).  Returns the fields of a bench line."""
    import torch
    import torch.distributed as dist

    from gqa_kv_cache_mla_gb300 import device as D

    builder, kfile, _ = WORKLOADS[name]
    # replicas: each rank writes its own independent batch (weak scaling)
    w = builder(DEFAULT_SEED + 100 * rank)
    k = kind_of(w)
    cls = {"mla": D.DeviceMLA, "gqa": D.DeviceGQA, "kno": D.DeviceKNorm,
           "gather": D.DeviceGather, "codec": D.DeviceConvert}[k]
    d = cls(w, device=dev, guard=False)
    stream = torch.cuda.current_stream(dev)
    run = lambda: d.run(stream=stream)
    abytes = algorithmic_bytes(w, name)
    flush = abytes < 2 * L2_BYTES

    for _ in range(warmup):
        if flush:
            flusher()
        run()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(steps):
        if flush:
            flusher()
        ev[i][0].record(stream)
        run()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    per = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(per)
    ms_max, tokens_all = combine_ranks(ms, w.T, world, dev)
    unit = unit_of(w)
    assert d.flags() == 0, "kernel reported data errors on the benchmark inputs"
    if k == "mla" and w.inplace:  # restore the rows the in-place steps rewrote
        d.cache.reset(w.cache.data)

    # end to end through the public API: pinned host inputs -> device, launch,
    # q/output and the error word back to the host, every step
    e2e_line = None
    if e2e and k in ("mla", "gqa", "kno") and not getattr(w, "inplace", False):
        r = measure_e2e(d, w, k, stream, dev, max(3, min(steps, 200)), warmup)
        r["ms"], _ = combine_ranks(r["ms"], w.T, world, dev)
        floor = copy_floor(r["h2d"], r["d2h"], dev, reps=max(8, min(steps, 64)))
        e2e_line = {"value": tokens_all / (r["ms"] / 1000.0), "unit": unit,
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                    "ms_per_step": r["ms"],
                    "copy_floor_ms": floor["both_ms"], "e2e_over_copy_floor":
                        r["ms"] / floor["both_ms"] if floor["both_ms"] else None,
                    "copy_floor": floor, "replay_ms_per_step": r["replay_ms_per_step"],
                    "how": "every step: one copy of its packed inputs (and a zeroed error "
                           "word) from pinned host memory, the kvw call, one copy of the "
                           "error word and the outputs back to pinned host memory; steps "
                           "pipelined %d deep on copy-in / compute / copy-out streams, %d "
                           "steps per CUDA graph replay, mean over %d replays" % (
                               r["depth"], r["per_graph"], len(r["replay_ms_per_step"]))}

    peak, peak_src = measured_peak()
    achieved = abytes / (ms / 1000.0) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": ncu_traffic(name, kfile),
            "algorithmic_bytes": abytes, "peak_source": peak_src,
            "kernel": kfile.replace(".cu", "")}
    host_us = (host_call_us(run, stream) if name in ("mla_decode",) and host_timing
               else None)
    if k == "mla" and w.inplace:
        d.cache.reset(w.cache.data)
    cpu = None
    if cpu_s and rank == 0 and world == 1:
        cpu = cpu_baseline(w, name, budget_s=cpu_s)
    out = {"name": name, "value": tokens_all / (ms_max / 1000.0), "unit": unit,
           "ms_per_step": ms_max, "steps": steps, "config": config_of(name, w, world),
           "roofline": roof, "e2e": e2e_line, "cpu_baseline": cpu, "clocks": clk,
           "timing": {"ms_median": statistics.median(per), "ms_min": min(per),
                      "wall_s_timed_region": wall,
                      "kernel_source_sha256_16": source_hash(kfile)},
           "host_us_per_call": host_us}
    del d
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from gqa_kv_cache_mla_gb300 import kvw  # noqa: F401  (fails loudly without the library)

    flusher = Flusher(dev)
    main_r = measure(args.workload, args.steps, args.warmup, dev, rank, world, flusher,
                     e2e=not args.no_e2e, cpu_s=None if args.no_cpu_baseline else args.cpu_s,
                     host_timing=not args.no_host_timing)
    also = []
    for name in args.also:
        if name == args.workload:
            continue
        steps = args.also_steps or default_steps(name)
        r = measure(name, steps, args.warmup, dev, rank, world, flusher,
                    e2e=not args.no_e2e and name in ("mla_decode",), cpu_s=None,
                    host_timing=not args.no_host_timing)
        also.append({"workload": r["config"]["workload"], "value": r["value"],
                     "unit": r["unit"], "ms_per_step": r["ms_per_step"], "steps": steps,
                     "roofline": {x: r["roofline"][x] for x in
                                  ("achieved", "frac", "algorithmic_bytes", "traffic",
                                   "kernel")},
                     "e2e": r["e2e"], "clocks": r["clocks"],
                     "host_us_per_call": r["host_us_per_call"],
                     "ms_median": r["timing"]["ms_median"], "ms_min": r["timing"]["ms_min"]})
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0
    line = {
        "metric": metric_of(args.workload, main_r["unit"]),
        "value": main_r["value"], "unit": main_r["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": main_r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; shapes and distributions of the benchmark configs)",
        "config": main_r["config"],
        "roofline": main_r["roofline"], "cpu_baseline": main_r["cpu_baseline"],
        "e2e": main_r["e2e"], "gpu_launches": args.steps, "clocks": main_r["clocks"],
        "timing": main_r["timing"],
        "also": also,
    }
    print(json.dumps(line), flush=True)
    return 0


def copy_floor(h2d, d2h, dev, reps=32):
    """Plain pinned copies of one e2e step's byte counts (one cudaMemcpyAsync
    each way per step): host->device alone, device->host alone, and both at
    once on two streams (the floor for a step whose copies overlap)."""
    import torch

    h_src = torch.empty(max(h2d, 16), dtype=torch.uint8, pin_memory=True)
    d_dst = torch.empty(max(h2d, 16), dtype=torch.uint8, device=dev)
    d_src = torch.zeros(max(d2h, 16), dtype=torch.uint8, device=dev)
    h_dst = torch.empty(max(d2h, 16), dtype=torch.uint8, pin_memory=True)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    launch = torch.cuda.current_stream(dev)

    def timed(do_in, do_out):
        for n in range(reps + 2):  # 2 untimed, then reps timed
            if n == 2:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(launch)
                s_in.wait_stream(launch)
                s_out.wait_stream(launch)
            if do_in:
                with torch.cuda.stream(s_in):
                    d_dst[:h2d].copy_(h_src[:h2d], non_blocking=True)
            if do_out:
                with torch.cuda.stream(s_out):
                    h_dst[:d2h].copy_(d_src[:d2h], non_blocking=True)
        launch.wait_stream(s_in)
        launch.wait_stream(s_out)
        b.record(launch)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    r = {"h2d_ms": timed(True, False) if h2d else 0.0,
         "d2h_ms": timed(False, True) if d2h else 0.0}
    r["both_ms"] = timed(h2d > 0, d2h > 0) if (h2d or d2h) else 0.0
    r["h2d_gbs"] = h2d / (r["h2d_ms"] / 1e3) / 1e9 if r["h2d_ms"] else None
    r["d2h_gbs"] = d2h / (r["d2h_ms"] / 1e3) / 1e9 if r["d2h_ms"] else None
    r["numa"] = numa_info(dev)
    return r


def numa_info(dev):
    """NUMA node of the GPU's PCI device and the nodes of this process's CPUs
    (pinned buffers are placed on the allocating CPU's node)."""
    out = {"gpu_node": None, "cpu_nodes": None}
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(dev.index), "--query-gpu=pci.bus_id",
                              "--format=csv,noheader"], capture_output=True, text=True,
                             timeout=20).stdout.strip().lower()
        dom, rest = bus.split(":", 1)
        path = "/sys/bus/pci/devices/%s:%s/numa_node" % (dom[-4:], rest)
        out["gpu_node"] = int(open(path).read().strip())
    except Exception:
        pass
    try:
        cpus = os.sched_getaffinity(0)
        nodes = set()
        base = "/sys/devices/system/node"
        for nd in os.listdir(base):
            if not re.fullmatch(r"node\d+", nd):
                continue
            spec = open(os.path.join(base, nd, "cpulist")).read().strip()
            ids = set()
            for part in filter(None, spec.split(",")):
                lo, _, hi = part.partition("-")
                ids.update(range(int(lo), int(hi or lo) + 1))
            if ids & cpus:
                nodes.add(int(nd[4:]))
        out["cpu_nodes"] = sorted(nodes)
    except Exception:
        pass
    return out


def host_call_us(run, stream, calls=1000):
    """Host time of one entry-point call (argument checks, device queries,
    launch), measured while the stream is held busy by a bounded sleep
    kernel so the calls only queue: wall time of ``calls`` calls / calls."""
    import torch

    run()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(200_000_000)  # about 0.1 s at 2 GHz
    t0 = time.perf_counter()
    for _ in range(calls):
        run()
    el = time.perf_counter() - t0
    torch.cuda.synchronize()
    return el / calls * 1e6


def default_steps(name):
    return {"mla_decode": 4000, "mla_decode_bf16": 4000}.get(name, 300)


def measure_e2e(d, w, k, stream, dev, steps, warmup, depth=3, per_graph=32, chunks=1):
    """Throughput through the public API with host buffers: every step copies
    its inputs from pinned host memory, launches the entry point and copies
    its results back.  Each step's I/O lives in one device buffer laid out as
    [inputs | error word | outputs] (16-byte aligned pieces), mirrored by
    pinned host buffers, so a step is one host->device copy of the inputs and
    a zeroed error word, the kvw call, and one device->host copy of the error
    word and the outputs.  Steps are pipelined ``depth`` deep over separate
    copy-in, compute and copy-out streams (a serving loop overlaps step i's
    compute with step i+1's inputs and step i-1's results), each buffer set
    reused only after the step that last used it is done; ``per_graph`` steps
    are captured in one CUDA graph.  Each copy is split into ``chunks`` pieces
    on as many streams, so that several copy engines share it."""
    import ctypes

    import torch

    from gqa_kv_cache_mla_gb300 import kvw

    if k == "mla":
        ins = [("q", d.q.tensor), ("kv", d.kv.tensor), ("off", d.offsets.tensor),
               ("clen", d.cache_lengths.tensor), ("pt", d.page_table.tensor)]
        outs = [("q_out", d.q_out.tensor)]
    elif k == "gqa":
        ins = [("q", d.q.tensor), ("off", d.offsets.tensor), ("clen", d.cache_lengths.tensor),
               ("pt", d.page_table.tensor)]
        if d.pos is not None:
            ins.append(("pos", d.pos.tensor))
        outs = [("out", d.out.tensor)]
    else:
        ins = [("off", d.offsets.tensor), ("clen", d.cache_lengths.tensor),
               ("pt", d.page_table.tensor)]
        outs = []

    def up16(x):
        return (x + 15) // 16 * 16

    layout, pos = {}, 0
    for name, t in ins:
        layout[name] = (pos, t)
        pos = up16(pos + t.numel() * t.element_size())
    err_at = pos
    pos += 16
    for name, t in outs:
        layout[name] = (pos, t)
        pos = up16(pos + t.numel() * t.element_size())
    total = pos
    h2d, d2h = err_at + 16, total - err_at  # [inputs | err] in, [err | outputs] out

    def view(buf, name):
        o, t = layout[name]
        n = t.numel() * t.element_size()
        return buf[o:o + n].view(t.dtype).view(t.shape)

    sets = []
    for _ in range(depth):
        dbuf = torch.empty(total, dtype=torch.uint8, device=dev)
        h_in = torch.zeros(h2d, dtype=torch.uint8, pin_memory=True)  # error word stays 0
        for name, t in ins:
            o, _ = layout[name]
            n = t.numel() * t.element_size()
            h_in[o:o + n].copy_(t.reshape(-1).view(torch.uint8).cpu())
        h_out = torch.empty(d2h, dtype=torch.uint8, pin_memory=True)
        v = {name: view(dbuf, name) for name in layout}
        v["err"] = dbuf[err_at:err_at + 4].view(torch.int32)
        desc = kvw.PagedCacheT()
        ctypes.memmove(ctypes.byref(desc), ctypes.byref(d.desc), ctypes.sizeof(desc))
        desc.page_table = v["pt"].data_ptr()
        desc.cache_lengths = v["clen"].data_ptr()
        sets.append(dict(dbuf=dbuf, v=v, desc=desc, h_in=h_in, h_out=h_out,
                         computed=torch.cuda.Event(), copied_out=[]))
    s_ins = [torch.cuda.Stream(dev) for _ in range(chunks)]
    s_outs = [torch.cuda.Stream(dev) for _ in range(chunks)]

    def pieces(n):  # [lo, hi) byte ranges, 16-byte aligned
        step_ = up16((n + chunks - 1) // chunks)
        return [(lo, min(n, lo + step_)) for lo in range(0, n, step_)]

    def call(S, stream):
        v = S["v"]
        if k == "mla":
            kvw.kvw_mla_rope_rmsnorm_quant(v["q_out"], v["q"], v["off"], d.freqs.tensor,
                                           d.gamma.tensor, v["kv"], S["desc"], w.layer_idx,
                                           w.epsilon, v["err"], stream,
                                           kv_row_stride=w.kv_in.shape[-1],
                                           out_dtype=w.q_out_dtype)
        elif k == "gqa":
            kvw.kvw_qk_rope_paged_ragged(
                v["q"], v["off"], S["desc"], d.freqs.tensor, v.get("pos"), w.interleaved,
                None if w.mrope_section is None else [int(x) for x in w.mrope_section],
                w.layer_idx, v["out"], v["err"], stream)
        else:
            kvw.kvw_rms_norm_kv_cache_paged(S["desc"], d.gamma.tensor, w.epsilon,
                                            w.weight_offset, w.layer_idx, w.T, v["off"],
                                            w.multiply_before_cast, w.per_head_norm, v["err"],
                                            stream)

    def step(S, comp, first):
        for j, (lo, hi) in enumerate(pieces(h2d)):
            s_in = s_ins[j]
            s_in.wait_stream(comp) if first else s_in.wait_event(S["computed"])
            if not first:
                for e in S["copied_out"]:
                    s_in.wait_event(e)  # its previous results were read back
            in_ready = torch.cuda.Event()
            with torch.cuda.stream(s_in):
                S["dbuf"][lo:hi].copy_(S["h_in"][lo:hi], non_blocking=True)
                in_ready.record(s_in)
            comp.wait_event(in_ready)
        with torch.cuda.stream(comp):
            call(S, comp)
            S["computed"].record(comp)
        S["copied_out"] = []
        for j, (lo, hi) in enumerate(pieces(d2h)):
            s_out = s_outs[j]
            s_out.wait_event(S["computed"])
            with torch.cuda.stream(s_out):
                S["h_out"][lo:hi].copy_(S["dbuf"][err_at + lo:err_at + hi], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_out)
                S["copied_out"].append(e)

    K = max(depth, per_graph // depth * depth)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    with torch.cuda.graph(graph, stream=cap, capture_error_mode="thread_local"):
        for n in range(K):
            step(sets[n % depth], cap, first=n < depth)
        for st in s_ins + s_outs:  # join every side stream back into the capture
            done = torch.cuda.Event()
            done.record(st)
            cap.wait_event(done)
    # at least three replays, each timed on its own (the host link is shared
    # with other work on the node: one replay alone can catch a slow moment)
    reps = max(3, (steps + K - 1) // K)
    for _ in range(max(1, warmup // K)):
        graph.replay()
    torch.cuda.synchronize()
    launch = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record(launch)
    for i in range(reps):
        graph.replay()
        ev[i + 1].record(launch)
    torch.cuda.synchronize()
    replay_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]
    for S in sets:
        assert int(S["h_out"][:4].view(torch.int32)[0]) == 0, "data errors in the e2e run"
    if outs:  # the results read back equal the device path's results
        name, t = outs[0]
        o = layout[name][0] - err_at
        n = t.numel() * t.element_size()
        assert torch.equal(sets[0]["h_out"][o:o + n], t.reshape(-1).view(torch.uint8).cpu()), \
            "e2e results differ from the device run"
    return {"ms": sum(replay_ms) / (reps * K), "h2d": h2d, "d2h": d2h, "depth": depth,
            "per_graph": K, "chunks": chunks,
            "replay_ms_per_step": [round(t / K, 4) for t in replay_ms]}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of the job: 1, or the torchrun world size (one rank per GPU)")
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--also", default=None,
                    help="comma-separated workloads measured after the main one ('' for none; "
                         "default: %s with the default workload, none otherwise)" %
                         ",".join(DEFAULT_ALSO))
    ap.add_argument("--also-steps", type=int, default=None,
                    help="timed steps of each 'also' workload (default: its own count)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-host-timing", action="store_true",
                    help="skip the host-time-per-call measurement of the decode call")
    ap.add_argument("--cpu-s", type=float, default=10.0,
                    help="seconds of oracle time for the cpu_baseline sample")
    ap.add_argument("--ref-step-s", type=float, default=2.0,
                    help="seconds of oracle time per step of --impl reference")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = dist_env()[2]
    if args.gpus != world:
        ap.error("--gpus %d but WORLD_SIZE is %d: launch N > 1 GPUs with torchrun "
                 "(--nproc-per-node N), one rank per GPU" % (args.gpus, world))
    if args.also is None:
        args.also = list(DEFAULT_ALSO) if args.workload == DEFAULT_WORKLOAD else []
    else:
        args.also = [x for x in args.also.split(",") if x]
        bad = [x for x in args.also if x not in WORKLOADS]
        if bad:
            ap.error("unknown workloads: %s" % ",".join(bad))
    if args.steps is None:
        args.steps = default_steps(args.workload)
        if args.impl == "reference":
            args.steps = 5
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
