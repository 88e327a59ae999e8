#!/usr/bin/env python3
"""Benchmark of the GQA AV decode reduction on GB300.

One step = one call of gqa_av_decode on one batch of the large-batch decode
workload (B=32, Cmax=131072, Hq=64, Hkv=8, G=8, D=128, bf16 V, lengths uniform
in [32768, 131072]: 8.6 GB of V, about 6.0 GB read per call) unless
--workload names another. Metric: achieved HBM GB/s over the compulsory bytes
(every in-range V row once, every in-range attn weight once, out once,
seq_lens), with µs/call as ms_per_step.

Device timing: the K calls are captured in CUDA graphs (one call per node,
cycling through rotating input sets whose total exceeds 3x the L2 size when
one set is smaller than that, so every call reads cold inputs) and replayed
between CUDA events on the launching stream; an untimed replay is queued just
before the start event, so the GPU is busy when the timed region opens and no
host launch latency falls inside it. e2e: the same calls through the public
API with the inputs copied from pinned host memory and out copied back,
inside the timed region.

`per_config` (default on): the four smaller decode workloads, each in both
modes (GQA reuse and the per-head baseline), their graph replays interleaved
and repeated until the standard error of each mean is below 0.5 %.

`--impl reference` times the fp64 CPU oracle (the only reference this method
has) on the host cores, on a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gqa_attention_weighted_gb300 import workloads as W  # noqa: E402

METRIC = "GQA AV decode achieved HBM GB/s over compulsory bytes (V read once), µs/call"
UNIT = "GB/s"
METRIC_QK = ("GQA QK-softmax decode achieved HBM GB/s over compulsory bytes (K read once), "
             "µs/call")
QK_SOURCES = ["gqa_attention_weighted_gb300/csrc/gqa_qk_kernel.cuh",
              "gqa_attention_weighted_gb300/csrc/gqa_qk_mma.cuh",
              "gqa_attention_weighted_gb300/csrc/gqa_qk_stream.cuh",
              "gqa_attention_weighted_gb300/csrc/gqa_qk_api.cu",
              "gqa_attention_weighted_gb300/csrc/gqa_av_kernel.cuh"]
METRIC_ATTN = ("GQA fused decode attention achieved HBM GB/s over compulsory bytes (K and V "
               "read once), µs/call")
ATTN_SOURCES = ["gqa_attention_weighted_gb300/csrc/gqa_attn_kernel.cuh",
                "gqa_attention_weighted_gb300/csrc/gqa_attn_api.cu",
                "gqa_attention_weighted_gb300/csrc/gqa_av_kernel.cuh"]
DEFAULT_WORKLOAD = "large"
# The decode workloads reported beside the headline, each in both modes.
PER_CONFIG = ("small", "llama", "phi", "mqa")
# L2 size the config line states (GB300: 126.5 MiB); the GPU arm sizes its
# rotating input sets from the device's own figure.
L2_NOMINAL = 132644864
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["gqa_attention_weighted_gb300/csrc/gqa_av_kernel.cuh",
                  "gqa_attention_weighted_gb300/csrc/gqa_av_mma.cuh",
                  "gqa_attention_weighted_gb300/csrc/gqa_av_stream.cuh",
                  "gqa_attention_weighted_gb300/csrc/gqa_av_instances.cuh",
                  "gqa_attention_weighted_gb300/csrc/gqa_av_api.cu"]
ENGINES = {"auto": 0, "fma": 1, "tensor": 2, "stream": 3}
SPLIT_MODES = {"auto": 0, "fixed": 1, "balanced": 2, "streamed": 3}
KERNEL_NAMES = {1: "gqa_av_kernel", 2: "gqa_av_mma_kernel", 3: "gqa_av_generic_kernel"}
STREAM_KERNEL = "gqa_av_stream_kernel"  # the tensor engine's streamed split rule (split_mode 3)


def kernel_name(plan) -> str:
    """The AV main kernel a plan runs."""
    return STREAM_KERNEL if plan["split_mode"] == 3 else KERNEL_NAMES[plan["engine"]]


def kernel_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def committed_entry(workload: str, mode: int, engine: int, split_mode: int):
    """The committed ncu summary of the main kernel for this workload, mode,
    engine and split rule, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    for e in entries:
        if (e.get("kernel_hash") == kernel_hash() and e.get("workload") == workload
                and e.get("mode") == mode and e.get("engine") == engine
                and e.get("split_mode") == split_mode and e.get("op", "av") == "av"):
            return e
    return None


def committed_traffic(workload: str, mode: int, engine: int, split_mode: int):
    """DRAM bytes per launch from the committed ncu summary (see committed_entry)."""
    e = committed_entry(workload, mode, engine, split_mode)
    return None if e is None else e.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        if shutil.which("nvidia-smi"):
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(",") for r in f if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl != "reference" else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ GPU arm
def bench_config(w, args, cbytes, flops, world):
    """The `config` object of both arms' lines: what the workload is and how it
    is run, computable without the GPU library."""
    set_bytes = cbytes_input_set(w)
    l2 = (f"inputs larger than L2: {set_bytes / 1e9:.2f} GB per input set vs "
          f"{L2_NOMINAL / 2**20:.1f} MiB of L2, one set" if set_bytes >= 3 * L2_NOMINAL else
          "rotating input sets totalling more than 3x the L2")
    return {**w.describe(), "mode": args.mode, "engine": args.engine,
            "split_mode": args.split_mode, "paged_block_size": args.paged or None,
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "compulsory_bytes_per_call": cbytes, "flops_per_call": flops, "l2": l2}


def cbytes_input_set(w):
    """Device bytes of one set of inputs and output (attn, V, out)."""
    return w.B * w.Cmax * (w.Hkv * w.D * 2 + w.Hq * 4) + w.B * w.Hq * w.D * 4


def dtype_of(engine: int, v_dtype: str) -> str:
    """The arithmetic the resolved kernel computes in."""
    if engine == 2:
        return (f"{v_dtype} V x fp32 weights split into {v_dtype} hi + lo (tcgen05), "
                f"fp32 accumulate")
    return f"{v_dtype} V widened to fp32, fp32 weights, fp32 FMA"


def rotating_sets(x, w, dev):
    """x plus clones, so that the sets total more than 3x the device's L2."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = cbytes_input_set(w)
    n_sets = max(1, math.ceil(3 * l2 / set_bytes)) if set_bytes < 3 * l2 else 1
    sets = [x] + [{k: t.clone() for k, t in x.items()} for _ in range(n_sets - 1)]
    outs = [torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
            for _ in range(n_sets)]
    return sets, outs, n_sets, set_bytes, l2


def capture(stream, n, call, sets, outs):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            call(sets[i % len(sets)], outs[i % len(outs)])
    return g


def timing_event():
    """A CUDA timing event that can be recorded inside a graph capture (as an
    event-record node), or None where this torch cannot make one."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None


def capture_timed(stream, warm, n, call, sets, outs):
    """One graph: `warm` untimed calls, the start event, `n` calls, the end
    event. The timed calls start on a GPU already busy with the same work,
    with no graph boundary or host launch inside the timed region. Returns
    (graph, start, end), or None where events cannot be captured."""
    start, end = timing_event(), timing_event()
    if start is None:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(warm):
            call(sets[i % len(sets)], outs[i % len(outs)])
        start.record(stream)
        for i in range(warm, warm + n):
            call(sets[i % len(sets)], outs[i % len(outs)])
        end.record(stream)
    return g, start, end


def time_interleaved(stream, arms, min_reps=5, max_reps=200, se_target=0.005, budget_s=6.0):
    """Replays each arm's graph in turn, round after round, until every arm's
    mean µs/call has a standard error below `se_target` of itself (at least
    `min_reps` rounds, at most `max_reps` or about `budget_s` seconds).
    arms: {name: (graph, calls timed per replay, start, end)}: the events are
    recorded inside the graph around its timed calls (capture_timed), or, with
    start None, on the stream around the whole replay. Returns {name: stats}."""
    samples = {k: [] for k in arms}
    names = list(arms)
    t0 = time.perf_counter()

    def stats(k):
        xs = samples[k]
        m = statistics.fmean(xs)
        se = statistics.stdev(xs) / math.sqrt(len(xs)) / m if len(xs) > 1 else float("inf")
        return m, se

    for r in range(max_reps):
        evs = []
        for k in names:
            g, n, e0, e1 = arms[k]
            if e0 is None:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
            else:
                g.replay()
            evs.append((k, n, e0, e1))
        stream.synchronize()
        for k, n, e0, e1 in evs:
            samples[k].append(e0.elapsed_time(e1) * 1e3 / n)
        if r + 1 >= min_reps and (all(stats(k)[1] < se_target for k in names)
                                  or time.perf_counter() - t0 > budget_s):
            break
    out = {}
    for k in names:
        m, se = stats(k)
        out[k] = {"us_per_call": round(m, 4), "se_pct": round(100 * se, 3),
                  "replays": len(samples[k]), "calls_per_replay": arms[k][1]}
    return out


def per_config(gq, dev, stream, peak):
    """The four smaller decode workloads, each in the GQA-reuse mode and the
    per-head baseline mode (the page's override knob), timed interleaved."""
    res = {}
    for name in PER_CONFIG:
        w = W.get(name)
        x = W.generate(w, dev, pad="zero")
        lens = x["seq_lens"].cpu().tolist()
        cbytes = W.compulsory_bytes(w, lens)
        sets, outs, n_sets, set_bytes, l2 = rotating_sets(x, w, dev)
        arms, plans = {}, {}
        with torch.cuda.stream(stream):
            for arm, mode in (("gqa", gq.MODE_GQA), ("per_head", gq.MODE_PER_HEAD)):
                def call(s, o, mode=mode):
                    gq.gqa_av_decode(s["attn"], s["v"], s["seq_lens"], o, mode=mode)
                for i in range(3):
                    call(sets[i % n_sets], outs[i % n_sets])
                # Calls per replay: about 3 ms of work, 20 to 2000 calls.
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for i in range(10):
                    call(sets[i % n_sets], outs[i % n_sets])
                e1.record(stream)
                e1.synchronize()
                est_us = e0.elapsed_time(e1) * 1e3 / 10
                n = int(min(2000, max(20, 3000.0 / max(est_us, 1e-3))))
                warm = int(min(n, max(3, 30.0 / max(est_us, 1e-3))))
                timed = capture_timed(stream, warm, n, call, sets, outs)
                arms[arm] = ((timed[0], n, timed[1], timed[2]) if timed else
                             (capture(stream, n, call, sets, outs), n, None, None))
                plans[arm] = gq.gqa_av_plan(w.B, w.Cmax, w.Hq, w.Hkv, w.D,
                                            gq.native.v_dtype_code(x["v"].dtype), mode)
            gq.gqa_av_device_status(stream)
            t = time_interleaved(stream, arms)
            gq.gqa_av_device_status(stream)
        entry = {"workload": w.name, "compulsory_bytes_per_call": cbytes,
                 "l2": f"rotating {n_sets} input sets, {n_sets * set_bytes / 1e6:.0f} MB "
                       f"(L2 {l2 / 1e6:.0f} MB)"}
        for arm in arms:
            st = t[arm]
            gbs = cbytes / (st["us_per_call"] * 1e-6) / 1e9
            pl = plans[arm]
            entry[arm] = {**st, "GBps": round(gbs, 2), "frac": round(gbs / peak, 4),
                          "kernel": kernel_name(pl), "engine": pl["engine"],
                          "split_mode": pl["split_mode"], "nsplit": pl["nsplit"],
                          "ctas": pl["ctas"],
                          "launches_per_call": 2 if pl["combine_ctas"] else 1}
        entry["per_head_over_gqa_time"] = round(
            t["per_head"]["us_per_call"] / t["gqa"]["us_per_call"], 3)
        res[name] = entry
        del sets, outs, x, arms
        torch.cuda.empty_cache()
    return res


def traffic_for(w, lens, plan):
    """roofline.traffic: DRAM bytes of the main kernel per launch, from the
    committed ncu summary when it was taken on the current source with this
    workload's plan. The large batch is too big for a multi-pass capture, so
    it takes its 1/8-context twin's figure (same tiles, split rule and grid),
    scaled by the ratio of context rows. Returns (bytes or None, source)."""
    t = committed_traffic(w.name, plan["mode"], plan["engine"], plan["split_mode"])
    if t is not None:
        return t, "ncu capture of this workload"
    if w.name != W.get("large").name:
        return None, None
    twin = W.get("ragged")
    entry = committed_entry(twin.name, plan["mode"], plan["engine"], plan["split_mode"])
    if entry is None or not entry.get("context_rows"):
        return None, None
    rows = sum(int(v) for v in lens)
    scaled = entry["traffic_bytes_per_launch"] * rows / entry["context_rows"]
    return int(round(scaled)), (f"ncu capture of {twin.name} ({entry['context_rows']} context "
                                f"rows) scaled to {rows} context rows")


def run_gpu(args, rank, world, local):
    import gqa_attention_weighted_gb300 as gq

    w = W.get(args.workload)
    dev = torch.device("cuda", torch.cuda.current_device())
    mode = {"auto": gq.MODE_AUTO, "gqa": gq.MODE_GQA, "per_head": gq.MODE_PER_HEAD}[args.mode]
    tuning = {}
    if args.engine == "stream":  # the tensor engine's streamed split rule
        tuning["engine"], tuning["split_mode"] = 2, 3
    elif args.engine != "auto":
        tuning["engine"] = ENGINES[args.engine]
    if args.split_mode != "auto":
        tuning["split_mode"] = SPLIT_MODES[args.split_mode]
    tuning = tuning or None

    def call(s, out):
        if "table" in s:
            gq.gqa_av_decode_paged(s["attn"], s["v"], s["table"], s["seq_lens"], out, mode=mode,
                                   tuning=tuning)
        elif tuning is None:
            gq.gqa_av_decode(s["attn"], s["v"], s["seq_lens"], out, mode=mode)
        else:
            gq.gqa_av_decode_tuned(s["attn"], s["v"], s["seq_lens"], out, mode=mode,
                                   tuning=tuning)

    x = W.generate(w, dev, pad="zero")
    x_contig = x
    if args.paged:
        x = paged_inputs(x, args.paged, w.seed)
    lens = x["seq_lens"].cpu().tolist()
    cbytes = W.compulsory_bytes(w, lens)
    flops = W.flops(w, lens)
    sets, outs, n_sets, set_bytes, l2 = rotating_sets(x, w, dev)
    plan = gq.gqa_av_plan(w.B, w.Cmax, w.Hq, w.Hkv, w.D, gq.native.v_dtype_code(x["v"].dtype), mode,
                          tuning)

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            call(sets[i % n_sets], outs[i % n_sets])
        stream.synchronize()
        gq.gqa_av_device_status(stream)

        # One graph of warm-up calls, the start event, the K timed calls and
        # the end event when K fits one graph (events recorded inside it);
        # else graphs of graph_len calls replayed after an untimed replay.
        warm = max(3, min(args.warmup, args.graph_len))
        timed = capture_timed(stream, warm, args.steps, call, sets, outs) \
            if args.steps <= args.graph_len else None
        if timed is not None:
            g_main, start, end = timed
            reps, rem, chunk = 1, 0, args.steps
            g_rem = None
            g_main.replay()  # untimed: the graph's own first run
            stream.synchronize()
        else:
            chunk = min(args.steps, args.graph_len)
            reps, rem = divmod(args.steps, chunk)
            g_main = capture(stream, chunk, call, sets, outs)
            g_rem = capture(stream, rem, call, sets, outs) if rem else None
            g_main.replay()  # graph warm-up (untimed)
            stream.synchronize()
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            if timed is not None:
                g_main.replay()
            else:
                # An untimed replay goes first, so the GPU is already busy when
                # the start event fires and the host's graph launch overlaps GPU work.
                g_main.replay()
                start.record(stream)
                for _ in range(reps):
                    g_main.replay()
                if g_rem is not None:
                    g_rem.replay()
                end.record(stream)
            end.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        elapsed_ms = start.elapsed_time(end)
        gq.gqa_av_device_status(stream)
        timing_desc = (f"one CUDA graph of {warm} untimed calls, the start event, the {args.steps} "
                       "timed calls and the end event (events recorded inside the graph)"
                       if timed is not None else
                       f"CUDA graphs of {chunk} calls x {reps}" + (f" + {rem}" if rem else "")
                       + ", events on the launch stream after an untimed replay")
        del g_main, g_rem

    elapsed_ms = max_over_ranks(elapsed_ms, world)
    ms_per_step = elapsed_ms / args.steps
    value = cbytes * args.steps * world / (elapsed_ms * 1e-3) / 1e9
    per_launch_s = ms_per_step * 1e-3
    achieved = cbytes / per_launch_s / 1e9
    peak, peak_kind = measured_peak()
    del sets, outs
    torch.cuda.empty_cache()

    e2e = run_e2e(gq, w, x, call, dev, args, world)
    traffic, traffic_src = (None, None) if args.paged else traffic_for(w, lens, plan)

    pc = None
    if rank == 0 and not args.no_per_config and not args.paged and args.workload == DEFAULT_WORKLOAD:
        pc = per_config(gq, dev, stream, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(w, x_contig, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "us_per_call": ms_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype_of(plan["engine"], w.v_dtype), "data": "synthetic",
        "config": bench_config(w, args, cbytes, flops, world),
        "plan": {**plan, "resolved_mode": plan["mode"], "resolved_engine": plan["engine"],
                 "resolved_split_mode": plan["split_mode"]},
        "timing": (f"{timing_desc}; {n_sets} input set(s), {n_sets * set_bytes / 1e6:.0f} MB "
                   f"(device L2 {l2 / 1e6:.0f} MB)"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                     "frac_of_8tbs_nominal": round(achieved / 8000.0, 4),
                     "traffic": traffic, "traffic_source": traffic_src,
                     "kernel": kernel_name(plan), "kernel_hash": kernel_hash(),
                     "duration": "average time of one whole call (main kernel and, when the "
                                 "context is split, the split-combine kernel) over the timed "
                                 "region; the main kernel alone is shorter"},
        "e2e": e2e,
        "gpu_launches": args.steps * (2 if plan["combine_ctas"] else 1),
        "clocks": clk.summary(),
    }
    if pc is not None:
        line["per_config"] = pc
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def paged_inputs(x, bs, seed):
    """The workload's V as a paged cache: blocks of `bs` rows in a pool in a
    seeded random order, and the block table that maps each sequence onto it."""
    v = x["v"]
    B, C, Hkv, D = v.shape
    maxb = (C + bs - 1) // bs
    g = torch.Generator(device="cpu").manual_seed(seed + 2)
    perm = torch.randperm(B * maxb, generator=g).to(v.device)
    pool = torch.zeros((B * maxb, bs, Hkv, D), dtype=v.dtype, device=v.device)
    padded = torch.zeros((B, maxb * bs, Hkv, D), dtype=v.dtype, device=v.device)
    padded[:, :C] = v
    pool[perm] = padded.view(B * maxb, bs, Hkv, D)
    table = perm.view(B, maxb).to(torch.int32).contiguous()
    return {"attn": x["attn"], "v": pool, "table": table, "seq_lens": x["seq_lens"]}


def run_gpu_qk(args, rank, world, local):
    """The decode score step (include/gqa_qk.h) on the workload's shape: q drawn
    N(0, 1), K drawn like the workload's V, attn [B, Cmax, Hq] written."""
    import gqa_attention_weighted_gb300 as gq

    w = W.get(args.workload)
    dev = torch.device("cuda", torch.cuda.current_device())
    mode = {"auto": gq.MODE_AUTO, "gqa": gq.MODE_GQA, "per_head": gq.MODE_PER_HEAD}[args.mode]
    x = W.generate(w, dev, pad="zero")
    g = torch.Generator(device=dev).manual_seed(w.seed + 1)
    x = {"q": torch.randn((w.B, w.Hq, w.D), generator=g, device=dev, dtype=torch.float32),
         "k": x["v"], "seq_lens": x["seq_lens"]}
    lens = x["seq_lens"].cpu().tolist()
    cbytes = W.compulsory_bytes(w, lens)  # K once, attn written once, q, seq_lens
    flops = W.flops(w, lens)
    scale = w.D ** -0.5

    engine = ENGINES[args.engine]
    # The kernel the library picks (include/gqa_qk.h): streamed on shapes with
    # at least as many tiles as SMs, else the fixed-split tensor-core kernel.
    qk_heads = w.G if (mode == gq.MODE_GQA or (mode == gq.MODE_AUTO and w.G > 1)) else 1
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    qk_tiles = w.B * (w.Hq // qk_heads)
    short_few = qk_tiles < sms and w.D <= 128 and qk_tiles * w.Cmax <= 2048 * 2 * sms
    resolved_engine = engine or (3 if w.B <= 2048 and not short_few else 2)

    def call(st, attn):
        gq.gqa_qk_softmax_decode(st["q"], st["k"], st["seq_lens"], attn, mode=mode, scale=scale,
                                 engine=engine)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = x["k"].numel() * 2 + w.B * w.Cmax * w.Hq * 4 + x["q"].numel() * 4
    n_sets = max(1, math.ceil(3 * l2 / set_bytes)) if set_bytes < 3 * l2 else 1
    sets = [x] + [{k: t.clone() for k, t in x.items()} for _ in range(n_sets - 1)]
    outs = [torch.zeros((w.B, w.Cmax, w.Hq), dtype=torch.float32, device=dev)
            for _ in range(n_sets)]
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            call(sets[i % n_sets], outs[i % n_sets])
        gq.gqa_qk_device_status(stream)
        chunk = min(args.steps, args.graph_len)
        reps, rem = divmod(args.steps, chunk)

        def capture(n):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for i in range(n):
                    call(sets[i % n_sets], outs[i % n_sets])
            return gr

        g_main = capture(chunk)
        g_rem = capture(rem) if rem else None
        g_main.replay()
        stream.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            g_main.replay()  # untimed: the GPU is busy when the start event fires
            start.record(stream)
            for _ in range(reps):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            end.record(stream)
            end.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        elapsed_ms = start.elapsed_time(end)
        gq.gqa_qk_device_status(stream)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    ms_per_step = elapsed_ms / args.steps
    value = cbytes * args.steps * world / (elapsed_ms * 1e-3) / 1e9
    achieved = cbytes / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = measured_peak()

    # End to end: pinned H2D of q, K rows c < L_b and seq_lens, the call, D2H
    # of the attn rows it wrote (rows c < L_b).
    host = {k: t.cpu().pin_memory() for k, t in x.items()}
    dbuf = {k: torch.empty_like(t) for k, t in x.items()}
    attn_d = torch.zeros((w.B, w.Cmax, w.Hq), dtype=torch.float32, device=dev)
    attn_h = torch.empty_like(attn_d, device="cpu").pin_memory()
    e_steps = max(1, min(args.e2e_steps, args.steps))
    e_lens = [max(0, min(int(v), w.Cmax)) for v in lens]
    ins = in_range_copies([(dbuf[k], host[k]) for k in host], w, e_lens)
    outs_back = in_range_copies([(attn_h, attn_d)], w, e_lens)
    with torch.cuda.stream(stream):
        def step():
            for d, h in ins:
                d.copy_(h, non_blocking=True)
            call(dbuf, attn_d)
            for h, d in outs_back:
                h.copy_(d, non_blocking=True)
        for _ in range(3):
            step()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(stream)
        for _ in range(e_steps):
            step()
        e1.record(stream)
        e1.synchronize()
        barrier(world)
    e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e_steps
    e2e = {"value": round(cbytes * world / (e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
           "ms_per_step": e_ms, "steps": e_steps,
           "h2d_bytes_per_step": sum(h.numel() * h.element_size() for _, h in ins),
           "d2h_bytes_per_step": sum(d.numel() * d.element_size() for _, d in outs_back)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline_qk(w, x, scale, args.cpu_seconds)
    resolved = 1 if (mode == gq.MODE_GQA or (mode == gq.MODE_AUTO and w.G > 1)) else 0
    line = {
        "metric": METRIC_QK, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "us_per_call": ms_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": (f"{w.v_dtype} K x fp32 q split into {w.v_dtype} hi + lo (tcgen05), fp32 "
                  "accumulate, fp32 softmax" if resolved_engine >= 2 else
                  f"{w.v_dtype} K widened to fp32, fp32 FMA, fp32 softmax"), "data": "synthetic",
        "config": {**w.describe(), "op": "qk", "mode": args.mode, "resolved_mode": resolved,
                   "engine": args.engine, "resolved_engine": resolved_engine,
                   "scale": scale, "parallelism": f"replicas{world}" if world > 1 else "single",
                   "compulsory_bytes_per_call": cbytes, "flops_per_call": flops,
                   "l2": f"rotating {n_sets} input sets, {n_sets * set_bytes / 1e6:.0f} MB "
                         f"(L2 {l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA graphs of {chunk} calls x {reps}"
                             + (f" + {rem}" if rem else "") + ", events on the launch stream"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                     "traffic": committed_traffic_qk(w.name, resolved, resolved_engine),
                     "kernel": {1: "gqa_qk_kernel", 2: "gqa_qk_mma_kernel"}.get(
                         resolved_engine, "gqa_qk_stream_kernel"),
                     "kernel_hash": kernel_hash(QK_SOURCES),
                     "duration": "average time of one whole call (score kernel and the "
                                 "normalise kernel) over the timed region"},
        "e2e": e2e,
        "gpu_launches": args.steps * 2,
        "clocks": clk.summary(),
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_gpu_attn(args, rank, world, local):
    """Fused decode attention (include/gqa_attn.h) on the workload's shape: V and
    seq_lens as for the AV call, K drawn the same way, q ~ N(0, logit_sigma^2)."""
    import gqa_attention_weighted_gb300 as gq

    w = W.get(args.workload)
    dev = torch.device("cuda", torch.cuda.current_device())
    mode = {"auto": gq.MODE_AUTO, "gqa": gq.MODE_GQA, "per_head": gq.MODE_PER_HEAD}[args.mode]
    x = W.generate_qkv(w, dev, pad="zero")
    lens = x["seq_lens"].cpu().tolist()
    cbytes = W.attention_compulsory_bytes(w, lens)
    flops = W.attention_flops(w, lens)
    scale = w.D ** -0.5
    smode = SPLIT_MODES[args.split_mode]
    plan = gq.gqa_attn_plan(w.B, w.Cmax, w.Hq, w.Hkv, w.D, gq.native.v_dtype_code(x["k"].dtype),
                            mode, args.attn_warps, args.attn_splits, smode, True,
                            args.attn_column_blocks)

    def call(st, out):
        gq.gqa_attn_decode(st["q"], st["k"], st["v"], st["seq_lens"], out, mode=mode, scale=scale,
                           consumer_warps=args.attn_warps, nsplit=args.attn_splits,
                           split_mode=smode, column_blocks=args.attn_column_blocks)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = sum(t.numel() * t.element_size() for t in x.values()) + w.B * w.Hq * w.D * 4
    n_sets = max(1, math.ceil(3 * l2 / set_bytes)) if set_bytes < 3 * l2 else 1
    sets = [x] + [{k: t.clone() for k, t in x.items()} for _ in range(n_sets - 1)]
    outs = [torch.zeros((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
            for _ in range(n_sets)]
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            call(sets[i % n_sets], outs[i % n_sets])
        gq.gqa_attn_device_status(stream)
        chunk = min(args.steps, args.graph_len)
        reps, rem = divmod(args.steps, chunk)

        def capture(n):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for i in range(n):
                    call(sets[i % n_sets], outs[i % n_sets])
            return gr

        g_main = capture(chunk)
        g_rem = capture(rem) if rem else None
        g_main.replay()
        stream.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            g_main.replay()  # untimed: the GPU is busy when the start event fires
            start.record(stream)
            for _ in range(reps):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            end.record(stream)
            end.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        elapsed_ms = start.elapsed_time(end)
        gq.gqa_attn_device_status(stream)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    ms_per_step = elapsed_ms / args.steps
    value = cbytes * args.steps * world / (elapsed_ms * 1e-3) / 1e9
    achieved = cbytes / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = measured_peak()

    # End to end: pinned H2D of q, K, V and seq_lens, the call, D2H of out.
    host = {k: t.cpu().pin_memory() for k, t in x.items()}
    dbuf = {k: torch.empty_like(t) for k, t in x.items()}
    out_d = torch.zeros((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    out_h = torch.empty_like(out_d, device="cpu").pin_memory()
    e_steps = max(1, min(args.e2e_steps, args.steps))
    # Only the K and V rows each sequence reads (c < L_b) go to the device.
    ins = in_range_copies([(dbuf[k], host[k]) for k in host], w,
                          [max(0, min(int(v), w.Cmax)) for v in lens])
    with torch.cuda.stream(stream):
        def step():
            for d, h in ins:
                d.copy_(h, non_blocking=True)
            call(dbuf, out_d)
            out_h.copy_(out_d, non_blocking=True)
        for _ in range(3):
            step()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(stream)
        for _ in range(e_steps):
            step()
        e1.record(stream)
        e1.synchronize()
        barrier(world)
    e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e_steps
    e2e = {"value": round(cbytes * world / (e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
           "ms_per_step": e_ms, "steps": e_steps,
           "h2d_bytes_per_step": sum(h.numel() * h.element_size() for _, h in ins),
           "d2h_bytes_per_step": out_h.numel() * 4}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline_attn(w, x, scale, args.cpu_seconds)
    launches = 1 if (plan["nsplit"] == 1 and plan["split_mode"] == 1) else 2
    line = {
        "metric": METRIC_ATTN, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "us_per_call": ms_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": (f"{w.v_dtype} K and V x fp32 scaled q and softmax weights split into "
                  f"{w.v_dtype} hi + lo (mma.sync), fp32 accumulate, fp32 softmax"), "data": "synthetic",
        "config": {**w.describe(), "op": "attn", "mode": args.mode, "plan": plan,
                   "scale": scale, "q": f"N(0, {w.logit_sigma}^2)",
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "compulsory_bytes_per_call": cbytes, "flops_per_call": flops,
                   "l2": f"rotating {n_sets} input sets, {n_sets * set_bytes / 1e6:.0f} MB "
                         f"(L2 {l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA graphs of {chunk} calls x {reps}"
                             + (f" + {rem}" if rem else "") + ", events on the launch stream"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                     "traffic": committed_traffic_attn(w.name, plan["mode"]),
                     "kernel": "gqa_attn_kernel",
                     "kernel_hash": kernel_hash(ATTN_SOURCES),
                     "duration": "average time of one whole call (attention kernel and, with "
                                 "several splits, the combine kernel) over the timed region"},
        "e2e": e2e,
        "gpu_launches": args.steps * launches,
        "clocks": clk.summary(),
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


def committed_traffic_attn(workload: str, mode: int):
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    for e in entries:
        if (e.get("op") == "attn" and e.get("kernel_hash") == kernel_hash(ATTN_SOURCES)
                and e.get("workload") == workload and e.get("mode") == mode):
            return e.get("traffic_bytes_per_launch")
    return None


def oracle_baseline_attn(w, x, scale, seconds):
    """The fused-attention oracle, as it stands (numpy fp64), on a context prefix."""
    import numpy as np
    from oracle import gqa_attn
    rows = w.Cmax
    q = x["q"].cpu().numpy()

    def inputs(n):
        kb = x["k"][:, :n].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        vb = x["v"][:, :n].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        return kb, vb, x["seq_lens"].cpu().clamp(max=n).numpy().astype(np.int32)

    kb, vb, lens = inputs(rows)
    t0 = time.perf_counter()
    gqa_attn.gqa_attention(q, kb, vb, w.v_dtype, lens, scale)
    t1 = time.perf_counter() - t0
    if t1 > seconds:
        rows = max(1, int(rows * seconds / t1 / 2))
        kb, vb, lens = inputs(rows)
    sample_bytes = W.attention_compulsory_bytes(w, lens.tolist())
    n, t_total = 0, 0.0
    while t_total < seconds or n < 1:
        t0 = time.perf_counter()
        gqa_attn.gqa_attention(q, kb, vb, w.v_dtype, lens, scale)
        t_total += time.perf_counter() - t0
        n += 1
    import oracle
    return {"value": round(sample_bytes * n / t_total / 1e9, 4), "unit": UNIT,
            "cores": oracle.host_cores(), "kind": "oracle",
            "sample": f"{n} passes over context positions [0, {rows}) of {w.name} "
                      f"({sample_bytes} compulsory bytes per pass), numpy fp64 (its BLAS "
                      f"threads over the affinity mask), {t_total:.1f} s"}


def committed_traffic_qk(workload: str, mode: int, engine: int):
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    for e in entries:
        if (e.get("op") == "qk" and e.get("kernel_hash") == kernel_hash(QK_SOURCES)
                and e.get("workload") == workload and e.get("mode") == mode
                and e.get("engine") == engine):
            return e.get("traffic_bytes_per_launch")
    return None


def oracle_baseline_qk(w, x, scale, seconds):
    """The score-step oracle, as it stands (numpy fp64), on a context prefix."""
    import numpy as np
    from oracle import gqa_qk
    rows = w.Cmax
    q = x["q"].cpu().numpy()

    def inputs(n):
        kb = x["k"][:, :n].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        return kb, x["seq_lens"].cpu().clamp(max=n).numpy().astype(np.int32)

    kb, lens = inputs(rows)
    t0 = time.perf_counter()
    gqa_qk.gqa_qk_softmax(q, kb, w.v_dtype, lens, scale)
    t1 = time.perf_counter() - t0
    if t1 > seconds:
        rows = max(1, int(rows * seconds / t1 / 2))
        kb, lens = inputs(rows)
    sample_bytes = W.compulsory_bytes(w, lens.tolist())
    n, t_total = 0, 0.0
    while t_total < seconds or n < 1:
        t0 = time.perf_counter()
        gqa_qk.gqa_qk_softmax(q, kb, w.v_dtype, lens, scale)
        t_total += time.perf_counter() - t0
        n += 1
    import oracle
    return {"value": round(sample_bytes * n / t_total / 1e9, 4), "unit": UNIT,
            "cores": oracle.host_cores(), "kind": "oracle",
            "sample": f"{n} passes over context positions [0, {rows}) of {w.name} "
                      f"({sample_bytes} compulsory bytes per pass), numpy fp64 (its BLAS "
                      f"threads over the affinity mask), {t_total:.1f} s"}


def in_range_copies(pairs, w, lens):
    """(dst, src) flat copies of at most 1 GiB for each (dst, src) tensor pair:
    for the [B, Cmax, ...] tensors, rows c < L_b of each sequence (contiguous
    per sequence; rows past a length are never read or written), the rest
    whole (everything whole when `lens` is None)."""
    out = []
    for d, h in pairs:
        if lens is not None and h.dim() >= 2 and h.shape[0] == w.B and h.shape[1] == w.Cmax:
            pieces = [(d[b, :L].reshape(-1), h[b, :L].reshape(-1)) for b, L in enumerate(lens) if L > 0]
        else:
            pieces = [(d.view(-1), h.view(-1))]
        for df, hf in pieces:
            per = max(1, (1 << 30) // hf.element_size())
            for i in range(0, hf.numel(), per):
                out.append((df[i:i + per], hf[i:i + per]))
    return out


def run_e2e(gq, w, x, call, dev, args, world):
    """Same call with host inputs, through the public API: every step copies
    from pinned host memory what the call reads -- rows c < L_b of attn and V
    (contiguous for each sequence; rows past a length are never read, as for
    a serving engine's cache) and the lengths -- split over `args.e2e_streams`
    copy streams, makes the call once they have landed, and copies out back to
    pinned host memory. The result is checked bitwise against the same call on
    the device-resident inputs."""
    host = {}
    for k, t in x.items():
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        host[k] = h
    out_host = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, pin_memory=True)
    dbuf = {k: torch.empty_like(t) for k, t in x.items()}
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    copiers = [torch.cuda.Stream(device=dev) for _ in range(max(1, args.e2e_streams))]
    d2h = out_host.numel() * 4
    steps = max(1, min(args.e2e_steps, args.steps))
    lens = [max(0, min(int(v), w.Cmax)) for v in x["seq_lens"].cpu().tolist()]
    # Copies of at most 1 GiB, dealt to the copy streams in turn: the rows
    # each sequence reads of the [B, Cmax, ...] tensors, the rest whole.
    # A paged cache's blocks are copied whole.
    chunks = in_range_copies([(dbuf[k], host[k]) for k in host], w, None if args.paged else lens)
    h2d = sum(src.numel() * src.element_size() for _, src in chunks)

    def step():
        ready = torch.cuda.Event()
        ready.record(stream)  # the previous step's call has been issued before this
        for j, (dst, src) in enumerate(chunks):
            cs = copiers[j % len(copiers)]
            if j < len(copiers):
                cs.wait_event(ready)
            with torch.cuda.stream(cs):
                dst.copy_(src, non_blocking=True)
        for cs in copiers:
            stream.wait_stream(cs)
        with torch.cuda.stream(stream):
            call(dbuf, out)
            out_host.copy_(out, non_blocking=True)

    for _ in range(2):
        step()
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    start.record(stream)
    for _ in range(steps):
        step()
    end.record(stream)
    end.synchronize()
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(end), world) / steps
    ref = torch.empty_like(out)
    with torch.cuda.stream(stream):
        call(x, ref)
    stream.synchronize()
    if not torch.equal(out_host, ref.cpu()):
        raise RuntimeError("e2e: the call on the copied inputs differs from the device-resident call")
    cbytes = W.compulsory_bytes(w, x["seq_lens"].cpu().tolist())
    return {"value": round(cbytes * world / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "ms_per_step": ms, "steps": steps, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "copy_streams": len(copiers),
            "copies_per_step": len(chunks), "h2d_GBps": round(h2d / (ms * 1e-3) / 1e9, 2),
            "checked": "bitwise against the device-resident call"}


# --------------------------------------------------------- oracle timings
def oracle_inputs(w, x, rows):
    """The workload cut to its first `rows` context positions (a bounded sample)."""
    import numpy as np
    attn = x["attn"][:, :rows].contiguous().cpu().numpy()
    vb = x["v"][:, :rows].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    lens = x["seq_lens"].cpu().clamp(max=rows).numpy().astype(np.int32)
    return attn, vb, lens


def oracle_rate(w, x, seconds, threads, rows):
    """Passes of the fp64 oracle, as it stands, over context positions
    [0, rows) of the workload with `threads` threads, for about `seconds`
    seconds (the prefix shrinks first if one pass would take longer).
    Returns (GB/s over the sample's compulsory bytes, rows, passes, seconds)."""
    import oracle
    attn, vb, lens = oracle_inputs(w, x, rows)
    t0 = time.perf_counter()
    oracle.gqa_av(attn, vb, w.v_dtype, lens, nthreads=threads)
    t1 = time.perf_counter() - t0
    if t1 > seconds / 2:  # shrink the sample so a pass fits the budget twice over
        rows = max(1, int(rows * seconds / t1 / 4))
        attn, vb, lens = oracle_inputs(w, x, rows)
    sample_bytes = W.compulsory_bytes(w, lens.tolist())
    n, t_total = 0, 0.0
    while t_total < seconds or n < 1:
        t0 = time.perf_counter()
        oracle.gqa_av(attn, vb, w.v_dtype, lens, nthreads=threads)
        t_total += time.perf_counter() - t0
        n += 1
    return sample_bytes * n / t_total / 1e9, rows, n, t_total, sample_bytes


def oracle_baseline(w, x, seconds):
    """The fp64 oracle, as it stands, on every host core in the affinity mask,
    and on one core, each on a bounded context prefix of the workload."""
    import oracle
    cores = oracle.host_cores()
    rows0 = min(w.Cmax, max(1, int(w.Cmax * min(1.0, 2e9 / max(1, W.compulsory_bytes(
        w, x["seq_lens"].cpu().tolist()))))))
    v, rows, n, t, sb = oracle_rate(w, x, seconds, cores, rows0)
    v1, rows1, n1, t1, sb1 = oracle_rate(w, x, seconds / 3, 1, min(rows, max(1, rows // cores)))
    return {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} passes over context positions [0, {rows}) of {w.name} "
                      f"({sb} compulsory bytes per pass), fp64, {t:.1f} s",
            "one_core": {"value": round(v1, 4), "unit": UNIT, "cores": 1,
                         "sample": f"{n1} passes over context positions [0, {rows1}) "
                                   f"({sb1} compulsory bytes per pass), fp64, {t1:.1f} s"}}


def run_reference(args, rank, world):
    """Reference arm: the oracle timed per step on a bounded sample of the
    workload. The inputs are drawn on the GPU when there is one (the GPU arm's
    draws, so the same lengths and bytes), else on the host."""
    if rank != 0:
        return
    import oracle
    w = W.get(args.workload)
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = W.generate(w, gen_dev, pad="zero")
    lens_all = x["seq_lens"].cpu().tolist()
    cbytes, flops = W.compulsory_bytes(w, lens_all), W.flops(w, lens_all)
    cores = oracle.host_cores()
    budget = 90.0  # seconds for warm-up plus timed steps together
    # First pass on at most ~2 GB of the workload, then sized to the budget.
    rows = min(w.Cmax, max(1, int(w.Cmax * min(1.0, 2e9 / max(1, cbytes)))))
    attn, vb, lens = oracle_inputs(w, x, rows)
    t0 = time.perf_counter()
    oracle.gqa_av(attn, vb, w.v_dtype, lens, nthreads=cores)
    t1 = max(time.perf_counter() - t0, 1e-6)
    per_step = budget / max(1, args.steps + args.warmup)
    if t1 > per_step:
        rows = max(1, int(rows * per_step / t1))
        attn, vb, lens = oracle_inputs(w, x, rows)
    del x
    sample_bytes = W.compulsory_bytes(w, lens.tolist())
    for _ in range(args.warmup):
        oracle.gqa_av(attn, vb, w.v_dtype, lens, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gqa_av(attn, vb, w.v_dtype, lens, nthreads=cores)
    elapsed = time.perf_counter() - t0
    value = sample_bytes * args.steps / elapsed / 1e9
    sample = (f"context positions [0, {rows}) of {w.name} per step "
              f"({sample_bytes} compulsory bytes), fp64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, args, cbytes, flops, world),
        "sample_rows": rows,
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="one of: " + ", ".join(W.ALIASES))
    ap.add_argument("--mode", choices=["auto", "gqa", "per_head"], default="auto")
    ap.add_argument("--engine", choices=list(ENGINES), default="auto",
                    help="kernel: the library's choice, the CUDA-core FMA kernel, the "
                         "tcgen05 tensor-core kernel, or the streamed tcgen05 kernel")
    ap.add_argument("--split-mode", choices=list(SPLIT_MODES), default="auto",
                    help="context splits: the library's choice, fixed splits of each "
                         "sequence, splits balanced over the batch's lengths, or the streamed "
                         "schedule (tensor-core engine)")
    ap.add_argument("--op", choices=["av", "qk", "attn"], default="av",
                    help="av: the AV reduction (the benchmark); qk: the decode score step "
                         "before it; attn: both fused in one pass over K and V")
    ap.add_argument("--attn-warps", type=int, default=0,
                    help="attn: consumer warps per CTA (0: the library's choice)")
    ap.add_argument("--attn-splits", type=int, default=0,
                    help="attn: context splits per tile (0: the library's choice)")
    ap.add_argument("--attn-column-blocks", type=int, default=0,
                    help="attn: output column blocks per head group (0: the library's choice)")
    ap.add_argument("--paged", type=int, default=0, metavar="BLOCK_SIZE",
                    help="run the AV call on a paged copy of V (blocks of this many rows in a "
                         "shuffled pool, gqa_av_decode_paged)")
    ap.add_argument("--graph-len", type=int, default=4000,
                    help="calls per CUDA graph (the timed calls form one graph up to this many)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--e2e-streams", type=int, default=1,
                    help="copy streams the e2e leg splits each step's host-to-device copies over")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload, per-mode timings beside the headline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be >= 1 and --warmup >= 0")

    rank, world, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            if not torch.cuda.is_available():
                raise SystemExit("bench.py: the GB300 arm needs a CUDA GPU")
            {"qk": run_gpu_qk, "attn": run_gpu_attn}.get(args.op, run_gpu)(args, rank, world,
                                                                            local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
