"""Benchmark: the five HLO hero fusions on one GB300, one JSON line.

A step is one pass of the whole hot path: the five fusions, each launched once through the C ABI on
its seeded synthetic full-size inputs (already resident in HBM). They share no buffer, so the timed step
runs each on a stream of its own (runner.ConcurrentFusions), launched in this order:
  row_reduce_exp     f32[256,512]                       exp, reduce-add over dim 1
  transpose_log      f32[8192,8192]                     log(p) + transpose(log(p))
  col_reduce_max     bf16[8192,16384]                   reduce-max over dim 0 (f32 accumulation)
  bcast_exp_reduce   bf16[8,1,1280,16384]{3,2,0,1}      exp, + broadcast b, reduce-add over dim 3
  quant_relayout     s8[4096,4096]                      dequant (per-axis) -> {0,1} -> quant (per-tensor)
value = algorithmic bytes of the step / step time (GB/s). The same step is then timed again with the
fusions one after another on one stream ("sequential"), an event between each: per-fusion GB/s, fraction
of the measured HBM copy peak and elements/s, and the roofline of the dominant kernel, come from that pass.
L2 is flushed (a 256 MiB write) before every timed step, outside the timed interval, and the host waits
for each timed step before it queues the next.

Multi-GPU (torchrun): every rank runs its own replica of the step (weak scaling, no collective); value
= bytes processed by all ranks / max over ranks of the timed region.

--impl reference times the CPU oracle (the plain C++ reference of the same fusions) on the host cores.
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

import numpy as np  # noqa: E402

from transpose_heroes_gb300 import inputs as inp  # noqa: E402

METRIC = "achieved HBM GB/s per fusion and fraction of GB300 peak; elements/s"
ORDER = ["row_reduce_exp", "transpose_log", "col_reduce_max", "bcast_exp_reduce", "quant_relayout"]
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("HLO hero fusions, one launch each per step: row_reduce_exp f32[256,512]{1,0}; "
            "transpose_selfadd_log f32[8192,8192]{1,0}; col_reduce_max bf16[8192,16384]{1,0}; "
            "bcast_exp_row_reduce bf16[8,1,1280,16384]{3,2,0,1}+bf16[16384]; "
            "quant_relayout s8[4096,4096]{1,0}->{0,1}")
L2_NOTE = ("L2 flushed by a 256 MiB device write before every timed step (outside the timed interval), then a "
           "device-side spin (8M cycles) so that the host has queued the whole step before it starts: host issue time "
           "is outside the device timing (it is inside e2e)")
HOST_LEAD_CYCLES = 8_000_000  # device clock cycles the stream spins after the flush
# fusions beyond the five workloads, measured beside the step: the loop fusion of "XLA:GPU Emitters"
# (section "Loop emitter"), the max/argmax variadic reduce of "XLA Operation Semantics" and a
# quantized add (dequantize_op_quantize)
NEXT_ROWS = {"gelu_bf16": lambda seed: inp.gelu_bf16(seed=seed), "argmax_f32": lambda seed: inp.argmax_f32(seed=seed),
             "quant_add_s8": lambda seed: inp.quant_add_s8(seed=seed),
             "transpose3_exp_abs_f32": lambda seed: inp.transpose3_exp_abs(seed=seed)}
# kernel each fusion launches (for the launch list / roofline)
KERNELS = {"row_reduce_exp": "row_warp_kernel", "transpose_log": "selfadd_tma_kernel",
           "col_reduce_max": "col_reduce_kernel", "bcast_exp_reduce": "row_stream_kernel",
           "quant_relayout": "quant_tma_kernel"}
CLEAN_L2_NOTE = ("alone_clean_l2_us / clean_l2_us (not part of value): the fusion timed alone after the same "
                 "256 MiB write followed by a 256 MiB read, so that the write's dirty lines leave L2 before the "
                 "launch instead of during it (what ncu's cache flush leaves)")
STEP_SYNC_NOTE = ("the host waits for each timed step to finish before it queues the next (flush, device-side "
                  "spin, step): with all steps queued ahead the concurrent step took ~241 us instead of ~222 us")
SCHEDULE_NOTE = ("the five fusions of a step are independent (no buffer shared): each runs on a stream of "
                 "its own, forked from and joined back into the timing stream; the events bracket the whole "
                 "step")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record():
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if it was taken on
    the kernel's current source: the record lists the source files the kernel is built from (its
    translation unit and the headers under csrc/) with their SHA-256, and every one must still match."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    files = d.get("source_files") or []
    if not files or d.get("source_sha256") != source_hash(files):
        return None
    return d


def kernel_sources(tu):
    """The files a kernel's translation unit is built from: the .cu file and every header in csrc/."""
    csrc = os.path.join(ROOT, "transpose_heroes_gb300", "csrc")
    hs = sorted(n for n in os.listdir(csrc) if n.endswith((".cuh", ".h", ".inc")))
    return [tu] + hs


def source_hash(files):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "transpose_heroes_gb300", "csrc")
    for name in files:
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
        except OSError:
            return None
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU works (reads only)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = f"/tmp/hlofusion_clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(values, reduce_fn):
    """Combines one float per rank (max for times, sum for bytes) through torch.distributed when
    initialised, else returns the local value."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return values
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(values)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if reduce_fn == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------------------------------
# CPU baseline (the oracle as it stands)
# ------------------------------------------------------------------------------------------------------
def cpu_sample_fusions(fraction: float):
    """A bounded sample of the same workload: each fusion on a leading fraction of its rows (whole rows,
    so every output is complete), the row-reduce in full."""
    fr = max(min(fraction, 1.0), 1e-4)
    out = [inp.row_reduce_exp(seed=1)]
    n = max(64, int(8192 * fr ** 0.5) // 64 * 64)
    out.append(inp.transpose_log(seed=1, n=n))
    out.append(inp.col_reduce_max(seed=1, rows=max(8, int(8192 * fr)), cols=16384))
    out.append(inp.bcast_exp_reduce(seed=1, d0=1, d2=max(1, int(10240 * fr)), d3=16384))
    out.append(inp.quant_relayout(seed=1, n0=max(16, int(4096 * fr) // 16 * 16), n1=4096))
    return out


def run_oracle_once(fusions):
    import oracle

    t0 = time.perf_counter()
    nbytes = 0
    for f in fusions:
        if f.kind == "reduce":
            oracle.reduce(f.data, f.dims, f.dtype, f.dimensions, f.reduce_kind, f.init, f.out_dtype, m2m=f.m2m,
                          out_m2m=f.out_m2m, prologue=f.prologue)
        elif f.kind == "transpose":
            oracle.transpose(f.data, f.dims, f.dtype, f.permutation, m2m=f.m2m, out_m2m=f.out_m2m,
                             self_add=f.self_add, prologue=f.prologue, epilogue=f.epilogue)
        else:
            oracle.quant_fusion(f.data, f.dims, f.dtype, f.in_q, f.out_m2m, f.out_dtype, out_q=f.out_q, m2m=f.m2m)
        nbytes += f.algorithmic_bytes
    return nbytes, time.perf_counter() - t0


def _timed_passes(fusions, min_seconds):
    run_oracle_once(fusions)  # warm-up, not counted
    total_bytes, total_t, passes = 0, 0.0, 0
    while total_t < min_seconds:
        b, dt = run_oracle_once(fusions)
        total_bytes += b
        total_t += dt
        passes += 1
    return total_bytes, total_t, passes


def cpu_baseline(min_seconds=10.0):
    """The oracle, as it stands, on the host cores: whole passes of the full workload on all cores until
    at least min_seconds have run (the first pass is a warm-up and not counted); then the same on one
    thread, on a 1/32 row sample of the workload."""
    import oracle

    oracle.build()
    cores = len(os.sched_getaffinity(0))
    oracle.set_num_threads(cores)
    fusions = cpu_sample_fusions(1.0)
    total_bytes, total_t, passes = _timed_passes(fusions, min_seconds)
    sample = (f"{passes} timed passes (after one warm-up pass) of the five fusions at full size: " +
              "; ".join(f"{f.name}" for f in fusions))
    oracle.set_num_threads(1)
    small = cpu_sample_fusions(1.0 / 32)
    b1, t1, p1 = _timed_passes(small, min_seconds)
    oracle.set_num_threads(cores)
    one = {"value": b1 / t1 / 1e9, "unit": "GB/s", "cores": 1, "seconds": t1,
           "sample": f"{p1} timed passes (after one warm-up pass) of the leading 1/32 of each fusion's rows "
                     "(row_reduce_exp in full): " + "; ".join(f.name for f in small)}
    return {"value": total_bytes / total_t / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
            "seconds": total_t, "one_thread": one}


def reference_arm(args):
    rank, world, local = dist_env()
    if world > 1 and rank != 0:
        return 0
    import oracle

    oracle.build()
    cores = len(os.sched_getaffinity(0))
    oracle.set_num_threads(cores)
    # size the per-step sample so that warmup + steps take about a minute on these cores
    probe = cpu_sample_fusions(1.0 / 256)
    pbytes, pdt = run_oracle_once(probe)
    per_step_budget = 60.0 / max(1, args.steps + args.warmup)
    fraction = min(1.0, (1.0 / 256) * per_step_budget / max(pdt, 1e-3))
    fusions = cpu_sample_fusions(fraction)
    for _ in range(args.warmup):
        run_oracle_once(fusions)
    total_bytes, total_t = 0, 0.0
    for _ in range(args.steps):
        b, dt = run_oracle_once(fusions)
        total_bytes += b
        total_t += dt
    value = total_bytes / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_fraction_of_rows": fraction, "seed": 1},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"leading {fraction:.4g} of each fusion's rows (row_reduce_exp in full), "
                                   "the plain C++ oracle, OpenMP over independent outputs"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------------
def ours(args):
    import torch
    import torch.distributed as dist

    from transpose_heroes_gb300 import build as libbuild
    from transpose_heroes_gb300.runner import ConcurrentFusions, DeviceFusion

    rank, world, local = dist_env()
    if args.gpus != world:
        # one process per GPU: N > 1 is launched by torchrun, which sets WORLD_SIZE = N
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch N > 1 with "
              f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus}",
              file=sys.stderr)
        return 2
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    libbuild.build()
    dev = f"cuda:{local}"
    fusions = [inp.full(n, seed=args.seed) for n in ORDER]
    devs = [DeviceFusion(f, device=dev, pin_host=True) for f in fusions]
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    step_bytes = sum(f.algorithmic_bytes for f in fusions)
    step_elems = sum(f.elements for f in fusions)

    # the step: the five fusions (independent, no shared buffers) each on a stream of its own, forked
    # from and joined back into `stream`
    concurrent = ConcurrentFusions(devs, device=dev)

    def sequential_step(evs=None):
        """The same five fusions one after another on `stream`, an event between each: their own times."""
        for i, d in enumerate(devs):
            if evs is not None:
                evs[i].record(stream)
            d.run(stream=stream)
        if evs is not None:
            evs[len(devs)].record(stream)

    def sync_all():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        flush.fill_(1)
        concurrent.run(stream)
        flush.fill_(2)
        sequential_step()
    sync_all()
    ev_c = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        ev_c[k][0].record(stream)
        concurrent.run(stream)
        ev_c[k][1].record(stream)
        torch.cuda.synchronize()  # each step starts from an idle device (see STEP_SYNC_NOTE)
    sync_all()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(devs) + 1)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        sequential_step(ev[k])
        torch.cuda.synchronize()
    sync_all()
    clocks = sampler.stop()
    per_fusion_ms = [[ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps)] for i in range(len(devs))]
    step_ms = [a.elapsed_time(b) for a, b in ev_c]
    local_total_s = sum(step_ms) / 1e3
    total_s = aggregate(local_total_s, "max")
    all_bytes = aggregate(float(step_bytes * args.steps), "sum")
    value = all_bytes / total_s / 1e9
    seq_total_s = aggregate(sum(ev[k][0].elapsed_time(ev[k][len(devs)]) for k in range(args.steps)) / 1e3, "max")
    sequential = {"value": all_bytes / seq_total_s / 1e9, "unit": "GB/s",
                  "ms_per_step": 1e3 * seq_total_s / args.steps,
                  "note": "the five fusions one after another on one stream (per_fusion comes from this pass)"}

    hbm, peak_src = peaks()
    reps = max(3, min(args.steps, 200))

    clean_src = torch.ones(64 << 20, dtype=torch.float32, device=dev)  # 256 MiB read after the flush
    clean_acc = torch.empty((), dtype=torch.float32, device=dev)

    def time_alone(fn, clean=False):
        """Mean CUDA-event interval of fn over `reps` launches, L2 flushed before each (the 256 MiB write;
        with clean=True then a 256 MiB read, so that the write's dirty lines are written back before the
        launch instead of during it)."""
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in evs:
            flush.fill_(3)
            if clean:
                torch.sum(clean_src, dim=0, out=clean_acc)
            torch.cuda._sleep(HOST_LEAD_CYCLES // 8)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
        return 1e3 * statistics.mean(a.elapsed_time(b) for a, b in evs)

    def copy_same_bytes_us(nbytes):
        """A plain device-to-device copy moving nbytes (half read, half written: torch's copy_ of a
        contiguous byte tensor, a cudaMemcpyAsync), timed alone the same way: what a copy of these bytes
        reaches in this timing loop."""
        src = torch.empty(nbytes // 2, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        us = time_alone(lambda: dst.copy_(src))
        del src, dst
        return us

    per = {}
    for i, f in enumerate(fusions):
        ms = statistics.mean(per_fusion_ms[i])
        gbs = f.algorithmic_bytes / (ms / 1e3) / 1e9
        per[ORDER[i]] = {"kernel": KERNELS[ORDER[i]], "us": 1e3 * ms, "us_min": 1e3 * min(per_fusion_ms[i]),
                         "algorithmic_bytes": f.algorithmic_bytes, "gbs": gbs, "frac_of_" + peak_src: gbs / hbm,
                         "elements_per_s": f.elements / (ms / 1e3)}
        copy_us = copy_same_bytes_us(f.algorithmic_bytes)
        per[ORDER[i]].update({"copy_same_bytes_us": copy_us, "speed_vs_copy": copy_us / (1e3 * ms),
                              "alone_clean_l2_us": time_alone(lambda d=devs[i]: d.run(stream=stream), clean=True)})
    dom = max(per, key=lambda k: per[k]["us"])
    dom_gbs = per[dom]["gbs"]
    tr = traffic_record()
    roofline = {"bound": "hbm", "kernel": per[dom]["kernel"], "fusion": dom, "achieved": dom_gbs, "peak": hbm,
                "peak_source": peak_src, "unit": "GB/s", "frac": dom_gbs / hbm,
                "traffic": (tr["dram_bytes_per_launch"] if tr and tr.get("fusion") == dom else None),
                "algorithmic_bytes_per_launch": per[dom]["algorithmic_bytes"]}

    # end to end through the same C-ABI calls: pinned host inputs -> device, fusions, outputs -> host
    e2e_steps = max(1, min(args.steps, 20))
    h2d = sum(d.h2d_bytes for d in devs)
    d2h = sum(d.d2h_bytes for d in devs)
    for d in devs:
        d.h2d()
        d.run(stream=stream)
        d.d2h()
    torch.cuda.synchronize()
    # three streams so that copies in, fusions and copies out overlap (the copy engines run both
    # directions at once); per-fusion events keep each buffer's reads and writes in order across steps
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in devs]
    ev_ran = [torch.cuda.Event() for _ in devs]
    ev_out = [torch.cuda.Event() for _ in devs]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for k in range(e2e_steps):
        for i, d in enumerate(devs):
            with torch.cuda.stream(s_in):
                if k:
                    s_in.wait_event(ev_ran[i])  # the previous step's fusion has read d's input
                d.h2d()
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if k:
                stream.wait_event(ev_out[i])  # the previous step's output has been copied out
            d.run(stream=stream)
            ev_ran[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_ran[i])
                d.d2h()
                ev_out[i].record(s_out)
    for ev in ev_out:
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = aggregate(e0.elapsed_time(e1) / 1e3, "max")
    e2e_bytes = aggregate(float(step_bytes * e2e_steps), "sum")
    e2e = {"value": e2e_bytes / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": e2e_steps}

    # fusions beyond the five workloads (the loop fusions and the rest of the path's next steps), each
    # timed alone the same way (L2 flushed before every launch, CUDA events), not part of `value`
    next_rows = {}
    for name, make in NEXT_ROWS.items():
        f = make(args.seed)
        d = DeviceFusion(f, device=dev, pin_host=False)
        us = time_alone(lambda: d.run(stream=stream))
        gbs = f.algorithmic_bytes / (us / 1e6) / 1e9
        copy_us = copy_same_bytes_us(f.algorithmic_bytes)
        next_rows[name] = {"workload": f.description, "us": us, "algorithmic_bytes": f.algorithmic_bytes,
                           "gbs": gbs, "frac_of_" + peak_src: gbs / hbm, "elements_per_s": f.elements / (us / 1e6),
                           "launches": reps, "copy_same_bytes_us": copy_us, "speed_vs_copy": copy_us / us,
                           "clean_l2_us": time_alone(lambda: d.run(stream=stream), clean=True)}
        del d

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": world, "l2": L2_NOTE, "seed": args.seed,
                       "parallelism": f"replicas{world}", "schedule": SCHEDULE_NOTE, "host": STEP_SYNC_NOTE,
                       "clean_l2": CLEAN_L2_NOTE},
            "elements_per_s": aggregate(float(step_elems * args.steps), "sum") / total_s,
            "sequential": sequential, "per_fusion": per, "roofline": roofline, "clocks": clocks, "e2e": e2e,
            "gpu_launches": len(devs) * args.steps, "next_rows": next_rows,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def parse_kw(text):
    """'n=6144,dims=(3,512,2048)' -> {'n': 6144, 'dims': (3, 512, 2048)} (literals only)."""
    import ast

    out, depth, cur = {}, 0, ""
    parts = []
    for ch in text:
        depth += ch in "([{"
        depth -= ch in ")]}"
        if ch == "," and depth == 0:
            parts.append(cur)
            cur = ""
        else:
            cur += ch
    if cur.strip():
        parts.append(cur)
    for part in parts:
        k, v = part.split("=", 1)
        out[k.strip()] = ast.literal_eval(v.strip())
    return out


def one_fusion(args):
    """Times one fusion alone (a maker of transpose_heroes_gb300.inputs, e.g. transpose_log, gelu_bf16,
    sum_exp_f32, with --fusion-kw for its sizes): --warmup launches, then --steps launches each after an
    L2 flush, CUDA events on the launching stream; prints one JSON line. Used for per-kernel profiles."""
    import torch

    from transpose_heroes_gb300 import build as libbuild
    from transpose_heroes_gb300.runner import DeviceFusion

    libbuild.build()
    f = getattr(inp, args.fusion)(seed=args.seed, **parse_kw(args.fusion_kw))
    d = DeviceFusion(f)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        flush.fill_(1)
        d.run(stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in evs:
        flush.fill_(2)
        torch.cuda._sleep(HOST_LEAD_CYCLES // 8)
        a.record(stream)
        d.run(stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
    us = 1e3 * statistics.mean(a.elapsed_time(b) for a, b in evs) if evs else 0.0
    hbm, src = peaks()
    gbs = f.algorithmic_bytes / (us / 1e6) / 1e9 if us else 0.0
    print(json.dumps({"fusion": f.name, "workload": f.description, "us": us, "algorithmic_bytes": f.algorithmic_bytes,
                      "gbs": gbs, "frac_of_" + src: gbs / hbm, "launches": args.steps}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--fusion", help="time one fusion alone (a maker in transpose_heroes_gb300.inputs)")
    ap.add_argument("--fusion-kw", default="", help="the maker's sizes, e.g. n=6144 or dims=(3,512,2048)")
    args = ap.parse_args()
    if args.fusion:
        return one_fusion(args)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)
    return ours(args)


if __name__ == "__main__":
    sys.exit(main())
