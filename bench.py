"""Benchmark of the per-token adapter routing hot path on one GB300 (or N, one rank per GPU).

Workload: the 4-modality kernel benchmark of "MoLoRA: Composable Specialization via
Per-Token Adapter Routing" (Table 3: K = 4 modalities, 2048 tokens, d = 4096), with rank 16,
bf16 x / A / B, fp32 y updated in place, tokens in runs of geometric length (mean 64) with one
uniformly drawn modality (vocabulary range) per run; synthetic, seeded.

One step = the whole path over one batch: vocabulary routing and dispatch (histogram, scan,
permutation; one kernel) -> grouped LoRA apply.  The timed steps are captured back to back as one CUDA
graph (consecutive kernels overlap their prologues through programmatic dependent launch)
between one pair of CUDA events.  The steps cycle through six resident batches of about
50 MB each, so a batch's x and y have been evicted from the 129 MB L2 by the time the batch
comes round again (inputs larger than L2 instead of a flush).  ``value`` = tokens / mean step time;
``apply_only`` gives the same for the apply kernel alone (the same batches, back to back),
and ``roofline`` relates that
kernel's algorithmic bytes per launch (x read once, y read and written once, the adapters
it touches read once) to its measured duration.  ``e2e`` runs the same path through the
public calls with every step's inputs copied from pinned host memory and its y copied back
inside the timed region, pipelined as a serving loop would (copy-in, compute and copy-out
of consecutive steps overlap on three streams).  ``cpu_baseline`` times the CPU oracle (single thread) on the same
inputs.

Multi-GPU: tokens are independent, so each rank runs its own batch (weak scaling, no
collective on the data path); the step time is the max over ranks.

``--impl reference`` times the CPU oracle itself as the reference arm.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "per-token LoRA apply tokens/s (2048 tok, d=4096, K=4); % of HBM roofline"
UNIT = "tokens/s"
WORKLOAD = "modality4"
FLUSH_BYTES = 256 << 20
N_BATCHES = 6


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--path", choices=["auto", "grouped", "scalar"], default="grouped")
    p.add_argument("--soak-s", type=float, default=1.0, help="untimed seconds of steps while clocks settle")
    p.add_argument("--cpu-budget-s", type=float, default=10.0, help="CPU seconds for the oracle baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--mode", choices=["step", "crossover", "crossover_topk", "crossover_stacked", "decode_step", "topk",
                                      "router", "perseq", "skew",
                                      "bf16y", "indirect", "split", "kernels", "tiling", "cv"],
                   default="step",
                   help="step: the contract line; the others print extra measurement lines (see run_mode)")
    p.add_argument("--replays", type=int, default=1000, help="graph replays per point in --mode topk")
    p.add_argument("--topk-k", default="1,2,3,4", help="--mode topk: comma-separated k values")
    p.add_argument("--ranks", default="16",
                   help="--mode crossover / perseq / tiling: comma-separated adapter ranks (8, 16, 32, 64)")
    p.add_argument("--topk-arms", default="fused_stacked,grouped,router",
                   help="--mode topk: which of fused_stacked, grouped, router to time")
    return p.parse_args(argv)


# --------------------------------------------------------------------------- distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, world: int, step_seconds_max: float, steps: int) -> dict:
    """Whole-job throughput: every rank processes its own batch each step; the job's step
    time is the slowest rank's."""
    ms = step_seconds_max / steps * 1e3
    return {"value": tokens_per_rank * world * steps / step_seconds_max, "ms_per_step": ms}


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix=f"molora_clocks_gpu{self.gpu_index}_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            if self.path:
                self.fh.close()
                os.remove(self.path)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        lines = open(self.path).read().splitlines()
        try:
            os.remove(self.path)
        except OSError:
            pass
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- the GPU arm

def algorithmic_bytes(wl, n_active_adapters: int) -> int:
    """Bytes the apply must move at least once: x read, y read + written, the active
    adapters' A and B read, ids + permutation read."""
    x = wl.N * wl.d_in * wl.x.element_size()
    y = 2 * wl.N * wl.d_out * 4
    ab = n_active_adapters * (wl.d_in * wl.r + wl.r * wl.d_out) * wl.A.element_size()
    idx = 2 * wl.N * wl.k * 4 + (wl.K + 1) * 4
    return x + y + ab + idx


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def run_ours(args, rank, world, local):
    import token_adapter_routing_gb300 as m
    from token_adapter_routing_gb300 import build as lib_build

    lib_build.build()
    m.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")

    # N_BATCHES distinct batches share the resident hot set (A, B) and the vocabulary ranges;
    # the timed steps cycle through them, so each step's x and y were last touched
    # N_BATCHES - 1 steps (about 250 MB of traffic) earlier and are no longer in L2.
    wls = [workloads.make(WORKLOAD, seed=1234 + 1 + rank * 1000 + b) for b in range(N_BATCHES)]
    wl = wls[0]
    starts, A, B = wl.starts.to(dev), wl.A.to(dev), wl.B.to(dev)
    batches = []
    for w_ in wls:
        batches.append({
            "tok": w_.tok.to(dev), "x": w_.x.to(dev), "y": w_.y0.to(dev),
            "adapter": torch.empty(w_.N, dtype=torch.int32, device=dev),
            "counts": torch.empty(w_.K, dtype=torch.int32, device=dev),
            "offsets": torch.empty(w_.K + 1, dtype=torch.int32, device=dev),
            "perm": torch.empty(w_.N, dtype=torch.int32, device=dev)})
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def route(i):
        # the token ids are resident before the timed region and no kernel writes them, so the
        # routing of step i+1 may read them while step i's apply runs (its stores still wait)
        b = batches[i % N_BATCHES]
        m.molora_route_vocab_dispatch_ex(b["tok"], starts, m.INPUTS_READY, adapter=b["adapter"], counts=b["counts"],
                                         offsets=b["offsets"], perm=b["perm"], err_word=err)

    def step(i):
        route(i)
        apply(i)

    def apply(i):
        b = batches[i % N_BATCHES]
        m.molora_lora_apply(b["x"], A, B, b["adapter"], b["y"], wl.scale, counts=b["counts"], offsets=b["offsets"],
                            perm=b["perm"], err_word=err, path=args.path)

    def capture(fn, count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                fn(i)
        return g

    warm = max(3, args.warmup)
    with torch.cuda.stream(stream):
        for i in range(N_BATCHES):
            step(i)  # eager first (loads the module, sets kernel attributes, routes every batch)
        stream.synchronize()
        g_warm, g_steps, g_applies = capture(step, warm), capture(step, args.steps), capture(apply, args.steps)
        g_one = capture(step, 1)
        g_route = capture(route, args.steps)
        g_warm_apply = capture(lambda i: apply(0), args.steps)
    n_active = [int((torch.bincount(b["adapter"].cpu().long(), minlength=wl.K) > 0).sum().item()) for b in batches]
    launches_per_step = 2  # route_vocab + dispatch (one kernel), apply

    def timed_block(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / 1e3

    def timed_flushed(g, steps):
        """One batch, a 256 MiB write before each replay, events around each replay."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            evs[i][0].record(stream)
            g.replay()
            evs[i][1].record(stream)
        stream.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3 / steps

    with torch.cuda.stream(stream):
        g_warm.replay()
        stream.synchronize()
        clocks = ClockSampler(local)
        clocks.start()
        t_end = time.time() + args.soak_s
        while time.time() < t_end:
            g_steps.replay()
            stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        step_s = timed_block(g_steps)    # exactly args.steps steps, back to back
        torch.cuda.synchronize()
        barrier(world)
        apply_s = timed_block(g_applies)  # the apply kernel alone, same batches, back to back
        torch.cuda.synchronize()
        barrier(world)
        clk = clocks.stop()
        flushed_s = timed_flushed(g_one, min(args.steps, 100))
        rd_s = timed_block(g_route)  # routing + dispatch alone, the same batches, back to back
        g_warm_apply.replay()
        stream.synchronize()
        warm_s = timed_block(g_warm_apply)  # one batch over and over: x and y stay in L2
    total_s = max_over_ranks(step_s, world, dev)
    apply_s = max_over_ranks(apply_s, world, dev)
    flushed_s = max_over_ranks(flushed_s, world, dev)
    agg = aggregate(wl.N, world, total_s, args.steps)

    assert int(err.item()) == 0, f"device error word {int(err.item()):#x}"

    peaks, peak_kind = measured_peaks()
    algo = sum(algorithmic_bytes(w_, n) for w_, n in zip(wls, n_active)) // N_BATCHES
    batch_mb = sum(t.numel() * t.element_size() for t in batches[0].values()) / 1e6
    apply_mean_s = apply_s / args.steps
    achieved_gbs = algo / apply_mean_s / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved_gbs / peaks["hbm_gbs"], 4), "traffic": None, "peak_kind": peak_kind,
            "kernel": "lora_grouped_kernel" if args.path != "scalar" else "lora_scalar_kernel",
            "algorithmic_bytes_per_launch": algo, "launch_us_mean": round(apply_mean_s * 1e6, 3),
            "frac_of_8TBs": round(achieved_gbs / 8000.0, 4)}
    traffic = load_profiled_traffic(args.path)
    if traffic is not None:
        roof["traffic"] = traffic
        roof["traffic_source"] = ("ncu, profiles/lora_grouped_kernel_modality4.md: dram__bytes_read.sum + "
                                  "dram__bytes_write.sum per launch, steady state (--cache-control none, "
                                  "back-to-back launches of this command), mean of three launches")

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(m, wl, dev, args, world)

    result = {
        "metric": METRIC, "value": round(agg["value"], 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(agg["ms_per_step"], 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "4-modality kernel benchmark: N=2048 tokens, d_in=d_out=4096, K=4, r=16, "
                               "bf16 x/A/B, fp32 y, vocabulary routing, geometric runs (mean 64)",
                   "global_batch": wl.N * world, "tokens_per_rank": wl.N, "path": args.path,
                   "step": "route_vocab_dispatch_ex (vocabulary routing, histogram, scan, permutation in one "
                           "kernel; INPUTS_READY: it reads the token ids while the previous step's apply runs "
                           "and stores after it) -> lora_apply",
                   "l2": (f"inputs larger than L2: the steps cycle through {N_BATCHES} resident batches "
                          f"(x, y, indices: {batch_mb:.0f} MB each), so a batch's data is evicted before it "
                          "comes round again"),
                   "timing": "one pair of CUDA events around all timed steps, captured back to back as one "
                             "CUDA graph (programmatic dependent launch between consecutive kernels)",
                   "parallelism": f"dp{world}" if world > 1 else "single-gpu"},
        "ms_per_step_flushed": round(flushed_s * 1e3, 6),
        "route_dispatch_us": round(max_over_ranks(rd_s, world, dev) / args.steps * 1e6, 3),
        "apply_warm_us": round(max_over_ranks(warm_s, world, dev) / args.steps * 1e6, 3),
        "apply_only": {"value": round(wl.N * world / apply_mean_s, 1), "unit": UNIT,
                       "us_per_launch": round(apply_mean_s * 1e6, 3)},
        "roofline": roof,
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
        "apply_timing": "the apply kernel alone over the same batches, back to back in one CUDA graph, "
                        "timed in a second block of the same run",
        "flushed_timing": "ms_per_step_flushed: one batch, a 256 MiB write before each step, CUDA events around "
                          "each graph replay (includes the graph launch)",
        "extra_timing": "route_dispatch_us: the fused routing + dispatch kernel alone over the same batches, back "
                        "to back (with INPUTS_READY, so each call reads while the previous one runs); "
                        "apply_warm_us: the apply on one batch over and over (x and y stay in L2)",
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget_s)
        result["cpu_baseline_all_cores"] = cpu_baseline_all_cores(wl, args.cpu_budget_s / 2)
    return result


def run_e2e(m, wl, dev, args, world):
    """Public calls with host buffers, run as a serving loop would: step i's inputs (token ids,
    x, y0) go host -> device on a copy-in stream while step i-1 computes and step i-2's y goes
    device -> host on a copy-out stream (two device buffer sets, event-ordered).  Timed from
    the first copy in to the last copy out; every step moves its own inputs and result."""
    tok_h = wl.tok.pin_memory()
    x_h = wl.x.pin_memory()
    y0_h = wl.y0.pin_memory()
    y_h = [torch.empty_like(y0_h).pin_memory() for _ in range(2)]
    starts = wl.starts.to(dev)
    A, B = wl.A.to(dev), wl.B.to(dev)  # the hot set stays resident
    bufs = [{"tok": torch.empty_like(wl.tok, device=dev), "x": torch.empty_like(wl.x, device=dev),
             "y": torch.empty_like(wl.y0, device=dev),
             "adapter": torch.empty(wl.N, dtype=torch.int32, device=dev),
             "counts": torch.empty(wl.K, dtype=torch.int32, device=dev),
             "offsets": torch.empty(wl.K + 1, dtype=torch.int32, device=dev),
             "perm": torch.empty(wl.N, dtype=torch.int32, device=dev)} for _ in range(2)]
    s_in, s_comp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

    def run(steps):
        ev_in = [torch.cuda.Event() for _ in range(steps)]
        ev_comp = [torch.cuda.Event() for _ in range(steps)]
        ev_out = [torch.cuda.Event() for _ in range(steps)]
        for i in range(steps):
            b = bufs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_out[i - 2])  # this buffer set's last result has left
                b["tok"].copy_(tok_h, non_blocking=True)
                b["x"].copy_(x_h, non_blocking=True)
                b["y"].copy_(y0_h, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[i])
                # tok comes from a host copy this stream waits for, not from the kernel before
                m.molora_route_vocab_dispatch_ex(b["tok"], starts, m.INPUTS_READY, adapter=b["adapter"],
                                                 counts=b["counts"], offsets=b["offsets"], perm=b["perm"])
                m.molora_lora_apply(b["x"], A, B, b["adapter"], b["y"], wl.scale, counts=b["counts"],
                                    offsets=b["offsets"], perm=b["perm"], path=args.path)
                ev_comp[i].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                y_h[i % 2].copy_(b["y"], non_blocking=True)
                ev_out[i].record(s_out)

    steps = max(5, min(args.steps, 50))
    run(3)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    run(steps)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    e1.record(s_out)
    torch.cuda.synchronize()
    sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    h2d = tok_h.numel() * 4 + x_h.numel() * x_h.element_size() + y0_h.numel() * 4
    d2h = y_h[0].numel() * 4
    return {"value": round(wl.N * world * steps / sec, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(sec / steps * 1e3, 4),
            "pipeline": "copy-in, compute and copy-out on three streams, two device buffer sets"}


def load_profiled_traffic(path):
    """DRAM bytes per apply launch from the committed ncu summary of the grouped kernel on
    this workload (a line `dram_bytes_per_launch: <int>`): read + write, measured in steady
    state over back-to-back launches with the caches left alone (so the y write-back the
    launch causes is counted).  None for the scalar path."""
    fn = os.path.join(ROOT, "profiles", "lora_grouped_kernel_modality4.md")
    if path == "scalar" or not os.path.exists(fn):
        return None
    try:
        for line in open(fn):
            if line.strip().startswith("dram_bytes_per_launch:"):
                return int(line.split(":", 1)[1].strip().split()[0])
    except (OSError, ValueError):
        return None
    return None


# --------------------------------------------------------------------------- CPU oracle

def oracle_step(wl):
    import oracle
    adapter, _ = oracle.route_vocab(wl.tok, wl.starts)
    counts, offsets, perm, _ = oracle.dispatch(adapter, wl.K)
    y, _ = oracle.lora_apply(wl.x, wl.A, wl.B, adapter, wl.y0, wl.scale)
    return y


def cpu_baseline(wl, budget_s):
    """The oracle as it stands, single-threaded, on the full batch, repeated for ~budget_s."""
    import oracle
    oracle.build()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_step(wl)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    return {"value": round(wl.N * reps / el, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"full batch ({wl.N} tokens: route_vocab + dispatch + lora_apply in double) x {reps} reps, "
                      f"{el:.1f} s"}


def cpu_baseline_all_cores(wl, budget_s):
    """The same oracle step with the apply split over the host's cores: route and dispatch once
    on the whole batch, then one oracle apply call per token block on a thread pool (the C
    oracle runs without the interpreter lock)."""
    import concurrent.futures
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    bounds = [wl.N * i // cores for i in range(cores + 1)]

    def step(pool):
        adapter, _ = oracle.route_vocab(wl.tok, wl.starts)
        oracle.dispatch(adapter, wl.K)
        futs = [pool.submit(oracle.lora_apply, wl.x[a:b], wl.A, wl.B, adapter[a:b], wl.y0[a:b], wl.scale)
                for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        return [f.result()[0] for f in futs]

    with concurrent.futures.ThreadPoolExecutor(max_workers=cores) as pool:
        reps, t0 = 0, time.perf_counter()
        while True:
            step(pool)
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s or reps >= 1000:
                break
    return {"value": round(wl.N * reps / el, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"full batch ({wl.N} tokens), apply split into {cores} token blocks on {cores} threads, "
                      f"x {reps} reps, {el:.1f} s"}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, as it stands, on this arm's workload and metric."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    wl = workloads.make(WORKLOAD, seed=1234 + 1)
    for _ in range(max(0, args.warmup)):
        oracle_step(wl)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(wl)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = wl.N * args.steps / total
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "4-modality kernel benchmark: N=2048 tokens, d_in=d_out=4096, K=4, r=16, "
                                   "bf16 x/A/B, fp32 y, vocabulary routing, geometric runs (mean 64)",
                       "global_batch": wl.N, "implementation": "CPU oracle (plain C, double, one thread)"},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"full batch of {wl.N} tokens per step, {args.steps} steps"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------------- extra modes

def _graph(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def _replay_ms(g, stream, reps, flush=None):
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            if flush is not None:
                flush.zero_()
            g.replay()
        for e0, e1 in evs:
            if flush is not None:
                flush.zero_()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
    return sorted(e0.elapsed_time(e1) for e0, e1 in evs)


def _loop_us(fn, stream, n=50, reps=5):
    """Per-call time of fn run n times back to back in one CUDA graph (one event pair around
    the replay: no per-call event quantum; the small inputs and the hot set stay in L2)."""
    with torch.cuda.stream(stream):
        fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                fn()
        g.replay()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            stream.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / n)
    return statistics.median(ts)


def _router_loop(m, wl, k, stream, dev, n=30):
    """The router alone, n calls back to back in one CUDA graph (one event pair around the
    replay, as in the main line), over enough x batches that their total exceeds twice the
    129 MB L2 (at most 8), so x streams from DRAM.  Returns (us per call, x batches)."""
    nb = max(1, min(8, -(-2 * (129 << 20) // (wl.x.numel() * wl.x.element_size()))))
    g = torch.Generator().manual_seed(4321)
    xs = [wl.x.to(dev)] + [torch.randn(wl.x.shape, generator=g).to(wl.x.dtype).to(dev) for _ in range(nb - 1)]
    W1, W2 = wl.W1.to(dev), wl.W2.to(dev)
    ids = torch.empty(wl.N, k, dtype=torch.int32, device=dev)
    w = torch.empty(wl.N, k, dtype=torch.float32, device=dev)
    state = {"i": 0}

    def call():
        m.molora_router_topk(xs[state["i"] % nb], W1, W2, k, ids=ids, w=w, want_logits=False)
        state["i"] += 1
    return _loop_us(call, stream, n=n, reps=7), nb


def _pct(v, q):
    return v[min(len(v) - 1, int(q * len(v)))]


def run_mode(args):
    """Extra measurements, one JSON line per point:
    crossover  decode sweep (Figures 5 and 9): batch 1..2048 x K 4..64 hot-set adapters, d=4096,
               rank r in --ranks (16 by default; the figures use 64), top-1, uniform and Zipf(1.1)
               adapter draws: route_vocab -> scalar apply,
               and route_vocab_dispatch -> grouped apply; each point timed cold (a CUDA graph
               per call, L2 flushed before each replay, p50 -- the GPU's event clock ticks in
               about 2 us here) and warm (50 calls back to back in one graph, the decode
               steady state with the hot set in L2), which decides the faster path.
    crossover_topk  top-2 with router-like weights, r = 16: d = 4096 at K = 4 and 8 over batch
               1..2048, and 2048 -> 6144 at K = 4 over 512..8192 tokens; scalar, grouped (with
               dispatch) and dense (without) applies, L2 flushed.
    decode_step  the decode step on the scalar path (vocabulary routing, then the scalar apply) at
               batch 1, 32, 160 and 512 (d = 4096, r = 16, K = 16), with and without
               INPUTS_READY on the routing call; warm, 50 steps back to back in one graph over
               four batches of inputs sharing one adapter buffer.
    crossover_stacked  the stacked pair against dispatch + grouped apply (ids and weights given)
               at d = 4096: K*r of 256, 512 and 1024 with r = 16 and 64, k = 1, 2, 4, N = 1024..8192;
               warm, 50 calls back to back in one graph.
    topk       top-k scaling (Table 16): N=8192, d=4096, K=8, r=64, k=1..4, router -> dispatch
               -> apply as one CUDA graph replayed --replays times back to back; p50 / p99.
    router     the learned-router workload at a Qwen3-1.7B MLP shape (N=4096, 2048 -> 6144,
               K=4, r=16, top-2): router alone; router -> dispatch -> grouped apply; router ->
               dense apply; router and dense apply fused in one kernel
               (molora_router_lora_apply); and each apply alone.
    perseq     the per-sequence baseline on the 4-modality workload (Tables 3 and 4): K masked
               passes over all tokens against one per-token pass, at each rank in --ranks
               (Table 3 uses 64).
    cv         step latency spread (Table 11): the decode step (route_vocab -> apply on the AUTO
               path, d = 4096, r = 16, K = 16 hot-set adapters drawn uniformly or Zipf(1.1) -- the
               access patterns of Figure 8) at batch 32..256, issued eagerly
               (two library calls) or as one CUDA graph replay, 1000 steps each, every step timed
               on the host clock around launch + synchronize (the GPU event clock ticks in about
               2 us here): mean, p50, p99 and the coefficient of variation.
    skew       the 4-modality workload with the group-size distributions of Table 9 (uniform,
               80/10/5/5, 95/2/2/1 modality shares per run): the apply alone and the whole step,
               back to back over six batches as in the main line.
    bf16y      the 4-modality workload with y held in bf16 (molora_lora_apply_bf16y), the apply
               alone back to back over six batches, grouped and scalar paths.
    indirect   Table 2: the hot set as two slabs (direct) against K separately allocated
               adapters (indirect, molora_lora_apply_indirect), N=2048, d=4096, r=16, top-1,
               uniform adapters, K = 4, 16, 64; the apply alone back to back over six batches.
    split      Table 6: per-token routing against per-sequence routing that must split the batch
               into its single-modality runs (one masked pass per run), on the 4-modality shape
               with interleaved text-heavy (70/10/10/10) and balanced runs, and separated (one
               contiguous block per modality); one CUDA graph each, L2 flushed between replays.
    tiling     Table 9's fixed vs adaptive tiles for the grouped apply: the plan the library
               chooses (adaptive: tile rows and cluster size from the slot and adapter counts)
               against fixed 64-row and fixed 128-row tiles in clusters of 8, and the scalar
               path, on the 4-modality workload under the three skews and on the decode sweep
               (K = 8..64, 256..2048 tokens, uniform and Zipf draws); the whole step (routing +
               dispatch + apply), 50 steps back to back in one graph, median of 5.  Runs the
               tuning build (build(tuning=True)), whose plan can be forced by environment."""
    import token_adapter_routing_gb300 as m
    from token_adapter_routing_gb300 import build as lib_build
    if args.mode == "tiling":
        m.load_library(lib_build.build(tuning=True))
    else:
        lib_build.build()
        m.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def emit(d):
        print(json.dumps(d), flush=True)

    if args.mode == "split":
        for label, dist, separated in (("interleaved, text-heavy", "70-10-10-10", False),
                                       ("interleaved, balanced", "uniform", False),
                                       ("separated", "uniform", True)):
            wl = workloads.make(WORKLOAD, dist=dist)
            tok = wl.tok.sort().values if separated else wl.tok  # ranges are contiguous in the vocabulary
            starts = wl.starts
            a_host = (torch.bucketize(tok.long(), starts.long(), right=True) - 1).to(torch.int32)
            runs, s0 = [], 0
            for t in range(1, wl.N + 1):
                if t == wl.N or a_host[t] != a_host[s0]:
                    runs.append((s0, t, int(a_host[s0])))
                    s0 = t
            tok_d, starts_d = tok.to(dev), starts.to(dev)
            x, A, B, y = wl.x.to(dev), wl.A.to(dev), wl.B.to(dev), wl.y0.to(dev)
            adapter = torch.empty(wl.N, dtype=torch.int32, device=dev)
            counts = torch.empty(wl.K, dtype=torch.int32, device=dev)
            offsets = torch.empty(wl.K + 1, dtype=torch.int32, device=dev)
            perm = torch.empty(wl.N, dtype=torch.int32, device=dev)

            def per_token():
                m.molora_route_vocab_dispatch(tok_d, starts_d, adapter=adapter, counts=counts, offsets=offsets,
                                              perm=perm)
                m.molora_lora_apply(x, A, B, adapter, y, wl.scale, counts=counts, offsets=offsets, perm=perm)

            def per_sequence_split():
                m.molora_route_vocab(tok_d, starts_d, adapter=adapter)
                for s0_, e0_, a_ in runs:
                    m.molora_lora_apply_masked_pass(x[s0_:e0_], A, B, adapter[s0_:e0_], a_, y[s0_:e0_], wl.scale)

            t_ms = _replay_ms(_graph(per_token, stream), stream, 50, flush)
            s_ms = _replay_ms(_graph(per_sequence_split, stream), stream, 50, flush)
            emit({"mode": "split", "distribution": label, "workload": "N=2048, d=4096, K=4, r=16",
                  "runs": len(runs), "per_token_us_p50": round(_pct(t_ms, 0.5) * 1e3, 2),
                  "per_sequence_split_us_p50": round(_pct(s_ms, 0.5) * 1e3, 2),
                  "speedup": round(_pct(s_ms, 0.5) / _pct(t_ms, 0.5), 2), "l2": "flushed between replays"})
    elif args.mode == "indirect":
        for K in (4, 16, 64):
            wls = [workloads.make("decode_sweep", seed=4000 + b, N=2048, K=K) for b in range(N_BATCHES)]
            starts, A, B = wls[0].starts.to(dev), wls[0].A.to(dev), wls[0].B.to(dev)
            A_list = [A[i].clone() for i in range(K)]
            B_list = [B[i].clone() for i in range(K)]
            bs = []
            for w_ in wls:
                adapter, counts, offsets, perm = m.molora_route_vocab_dispatch(w_.tok.to(dev), starts)
                bs.append({"x": w_.x.to(dev), "y": w_.y0.to(dev), "adapter": adapter, "counts": counts,
                           "offsets": offsets, "perm": perm})
            row = {"mode": "indirect", "workload": f"N=2048, d=4096, K={K}, r=16, top-1 uniform",
                   "path": m.molora_select_path(torch.bfloat16, 2048, 4096, 4096, K, 16, 1)}
            for layout, (AA, BB) in (("direct", (A, B)), ("indirect", (A_list, B_list))):
                def apply(i, AA=AA, BB=BB):
                    b = bs[i % N_BATCHES]
                    m.molora_lora_apply(b["x"], AA, BB, b["adapter"], b["y"], wls[0].scale, counts=b["counts"],
                                        offsets=b["offsets"], perm=b["perm"])
                n = 120
                with torch.cuda.stream(stream):
                    for i in range(N_BATCHES):
                        apply(i)
                    stream.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for i in range(n):
                            apply(i)
                    g.replay()
                    ts = []
                    for _ in range(5):
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        g.replay()
                        e1.record(stream)
                        stream.synchronize()
                        ts.append(e0.elapsed_time(e1) * 1e3 / n)
                row[f"{layout}_us"] = round(statistics.median(ts), 3)
            row["indirect_over_direct"] = round(row["indirect_us"] / row["direct_us"], 3)
            emit(row)
    elif args.mode == "bf16y":
        peaks, _ = measured_peaks()
        wls = [workloads.make(WORKLOAD, seed=1234 + 1 + b) for b in range(N_BATCHES)]
        starts, A, B = wls[0].starts.to(dev), wls[0].A.to(dev), wls[0].B.to(dev)
        bs = []
        for w_ in wls:
            adapter, counts, offsets, perm = m.molora_route_vocab_dispatch(w_.tok.to(dev), starts)
            bs.append({"x": w_.x.to(dev), "y": w_.y0.to(torch.bfloat16).to(dev), "adapter": adapter,
                       "counts": counts, "offsets": offsets, "perm": perm})
        n = 120
        for path in ("grouped", "scalar"):
            def apply(i, path=path):
                b = bs[i % N_BATCHES]
                m.molora_lora_apply(b["x"], A, B, b["adapter"], b["y"], wls[0].scale, counts=b["counts"],
                                    offsets=b["offsets"], perm=b["perm"], path=path)
            with torch.cuda.stream(stream):
                for i in range(N_BATCHES):
                    apply(i)
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(n):
                        apply(i)
                g.replay()
                ts = []
                for _ in range(5):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                    stream.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1e3 / n)
            us = statistics.median(ts)
            w0 = wls[0]
            n_active = int((torch.bincount(bs[0]["adapter"].cpu().long(), minlength=w0.K) > 0).sum().item())
            algo = (w0.N * w0.d_in * 2 + 2 * w0.N * w0.d_out * 2
                    + n_active * (w0.d_in * w0.r + w0.r * w0.d_out) * 2 + 2 * w0.N * 4 + (w0.K + 1) * 4)
            emit({"mode": "bf16y", "path": path, "workload": "N=2048, d=4096, K=4, r=16, y bf16",
                  "apply_us": round(us, 3), "tokens_per_s": round(w0.N / (us * 1e-6), 1),
                  "algorithmic_bytes": algo, "apply_GBps": round(algo / (us * 1e-6) / 1e9, 1),
                  "frac_of_measured": round(algo / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                  "l2": f"inputs larger than L2 ({N_BATCHES} resident batches, back to back)"})
    elif args.mode == "tiling":
        def loop_us(fn, n=50, reps=5):
            with torch.cuda.stream(stream):
                fn()
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(n):
                        fn()
                g.replay()
                stream.synchronize()
                ts = []
                for _ in range(reps):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                    stream.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1e3 / n)
            return statistics.median(ts)

        def force(C=None, TM=None):
            for key in ("MOLORA_CLUSTER", "MOLORA_TILE_ROWS", "MOLORA_ONE_PER_SM"):
                os.environ.pop(key, None)
            if C:
                os.environ["MOLORA_CLUSTER"] = str(C)
            if TM:
                os.environ["MOLORA_TILE_ROWS"] = str(TM)

        ranks = [int(v) for v in args.ranks.split(",")]
        cases = []
        if 16 in ranks:
            cases += [(WORKLOAD, {"dist": d}) for d in ("uniform", "80-10-5-5", "95-2-2-1")]
            cases += [("decode_sweep", {"N": b, "K": K}) for K in (8, 16, 32, 64) for b in (256, 512, 1024, 2048)]
            cases += [("decode_sweep", {"N": b, "K": K, "dist": "zipf"}) for K in (32, 64) for b in (512, 2048)]
        # other ranks: a grid over the batch (at rank 64 and d = 4096 the plans run one CTA per SM)
        cases += [("decode_sweep", {"N": b, "K": K, "r": r}) for r in ranks if r != 16 for K in (4, 8, 16, 32)
                  for b in (512, 768, 1024, 1280, 1536, 1792, 2048, 3072, 4096)]
        for name, kw in cases:
            wl = workloads.make(name, **kw)
            tok, starts = wl.tok.to(dev), wl.starts.to(dev)
            x, A, B, y = wl.x.to(dev), wl.A.to(dev), wl.B.to(dev), wl.y0.to(dev)
            adapter = torch.empty(wl.N, dtype=torch.int32, device=dev)
            counts = torch.empty(wl.K, dtype=torch.int32, device=dev)
            offsets = torch.empty(wl.K + 1, dtype=torch.int32, device=dev)
            perm = torch.empty(wl.N, dtype=torch.int32, device=dev)

            def step():
                m.molora_route_vocab_dispatch(tok, starts, adapter=adapter, counts=counts, offsets=offsets, perm=perm)
                m.molora_lora_apply(x, A, B, adapter, y, wl.scale, counts=counts, offsets=offsets, perm=perm,
                                    path="grouped")

            def scalar_step():
                m.molora_route_vocab(tok, starts, adapter=adapter)
                m.molora_lora_apply(x, A, B, adapter, y, wl.scale, path="scalar")

            res = {"mode": "tiling", "workload": name, "N": wl.N, "K": wl.K, "r": wl.r, "dist": kw.get("dist", "uniform"),
                   "unit": "us per step"}
            force()
            res["scalar"] = round(loop_us(scalar_step), 2)
            res["adaptive"] = round(loop_us(step), 2)
            force(8, 64)
            res["fixed_64"] = round(loop_us(step), 2)
            force(8, 128)
            res["fixed_128"] = round(loop_us(step), 2)
            force()
            emit(res)
    elif args.mode == "skew":
        peaks, _ = measured_peaks()
        for dist in ("uniform", "80-10-5-5", "95-2-2-1"):
            wls = [workloads.make(WORKLOAD, seed=1234 + 1 + b, dist=dist) for b in range(N_BATCHES)]
            starts, A, B = wls[0].starts.to(dev), wls[0].A.to(dev), wls[0].B.to(dev)
            bs = [{"tok": w_.tok.to(dev), "x": w_.x.to(dev), "y": w_.y0.to(dev),
                   "adapter": torch.empty(w_.N, dtype=torch.int32, device=dev),
                   "counts": torch.empty(w_.K, dtype=torch.int32, device=dev),
                   "offsets": torch.empty(w_.K + 1, dtype=torch.int32, device=dev),
                   "perm": torch.empty(w_.N, dtype=torch.int32, device=dev)} for w_ in wls]

            def route(i):
                b = bs[i % N_BATCHES]
                m.molora_route_vocab_dispatch(b["tok"], starts, adapter=b["adapter"], counts=b["counts"],
                                              offsets=b["offsets"], perm=b["perm"])

            def apply(i):
                b = bs[i % N_BATCHES]
                m.molora_lora_apply(b["x"], A, B, b["adapter"], b["y"], wls[0].scale, counts=b["counts"],
                                    offsets=b["offsets"], perm=b["perm"], path="grouped")

            n = 120
            with torch.cuda.stream(stream):
                for i in range(N_BATCHES):
                    route(i)
                    apply(i)
                stream.synchronize()
                gs, ga = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs, stream=stream):
                    for i in range(n):
                        route(i)
                        apply(i)
                with torch.cuda.graph(ga, stream=stream):
                    for i in range(n):
                        apply(i)
                res = {}
                for name, g in (("step", gs), ("apply", ga)):
                    g.replay()
                    ts = []
                    for _ in range(5):
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        g.replay()
                        e1.record(stream)
                        stream.synchronize()
                        ts.append(e0.elapsed_time(e1) * 1e3 / n)
                    res[name] = statistics.median(ts)
            groups = [torch.bincount(b["adapter"].cpu().long(), minlength=wls[0].K).tolist() for b in bs]
            n_active = [sum(1 for c in gr if c > 0) for gr in groups]
            algo = sum(algorithmic_bytes(w_, na) for w_, na in zip(wls, n_active)) / N_BATCHES
            emit({"mode": "skew", "dist": dist, "workload": "N=2048, d=4096, K=4, r=16 (4-modality benchmark)",
                  "group_sizes_first_batch": groups[0], "apply_us": round(res["apply"], 3),
                  "step_us": round(res["step"], 3), "apply_GBps": round(algo / (res["apply"] * 1e-6) / 1e9, 1),
                  "frac_of_measured": round(algo / (res["apply"] * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                  "l2": f"inputs larger than L2 ({N_BATCHES} resident batches, back to back)"})
    elif args.mode == "crossover_topk":
        for d_in, d_out, K, batches in ((4096, 4096, 4, (1, 8, 32, 128, 512, 2048)),
                                        (4096, 4096, 8, (1, 8, 32, 128, 512, 2048)),
                                        (2048, 6144, 4, (512, 1024, 2048, 4096, 8192))):
            for b in batches:
                k = 2
                g_ = torch.Generator().manual_seed(b + K)
                x = (torch.randn(b, d_in, generator=g_)).to(torch.bfloat16).to(dev)
                A = (torch.randn(K, d_in, 16, generator=g_) / math.sqrt(d_in)).to(torch.bfloat16).to(dev)
                B = (torch.randn(K, 16, d_out, generator=g_) / 4).to(torch.bfloat16).to(dev)
                y = torch.randn(b, d_out, generator=g_).to(dev)
                ids = torch.stack([torch.randperm(K, generator=g_)[:k] for _ in range(b)]).to(torch.int32).to(dev)
                w = torch.softmax(torch.randn(b, k, generator=g_), dim=1).to(dev)
                counts = torch.empty(K, dtype=torch.int32, device=dev)
                offsets = torch.empty(K + 1, dtype=torch.int32, device=dev)
                perm = torch.empty(b * k, dtype=torch.int32, device=dev)
                row = {"mode": "crossover_topk", "d_in": d_in, "d_out": d_out, "K": K, "k": k, "batch": b,
                       "auto": m.molora_select_path(torch.bfloat16, b, d_in, d_out, K, 16, k)}
                for path in ("scalar", "grouped", "dense"):
                    def fn(path=path):
                        if path == "grouped":
                            m.molora_dispatch(ids, K, counts=counts, offsets=offsets, perm=perm)
                        m.molora_lora_apply(x, A, B, ids, y, 2.0, w=w, counts=counts, offsets=offsets, perm=perm,
                                            path=path)
                    ms = _replay_ms(_graph(fn, stream), stream, 30, flush)
                    row[f"{path}_us_p50"] = round(_pct(ms, 0.5) * 1e3, 2)
                    row[f"{path}_us_warm"] = round(_loop_us(fn, stream), 3)
                row["fastest"] = min(("scalar", "grouped", "dense"), key=lambda p_: row[f"{p_}_us_warm"])
                emit(row)
    elif args.mode == "decode_step":
        for b in (1, 32, 160, 512):
            wls = [workloads.make("decode_sweep", seed=100 + i, N=b, K=16) for i in range(4)]
            ins = [dict(tok=w_.tok.to(dev), starts=w_.starts.to(dev), x=w_.x.to(dev), A=w_.A.to(dev),
                        B=w_.B.to(dev), y=w_.y0.to(dev)) for w_ in wls]
            adapter = torch.empty(b, dtype=torch.int32, device=dev)
            row = {"mode": "decode_step", "batch": b, "K": 16, "d": 4096, "r": 16, "path": "scalar"}
            for flag in (0, 1):
                state = {"i": 0}

                def step(flag=flag, state=state):
                    d_ = ins[state["i"] % 4]
                    state["i"] += 1
                    if flag:
                        m.molora_route_vocab_ex(d_["tok"], d_["starts"], m.INPUTS_READY, adapter=adapter)
                    else:
                        m.molora_route_vocab(d_["tok"], d_["starts"], adapter=adapter)
                    m.molora_lora_apply(d_["x"], d_["A"], d_["B"], adapter, d_["y"], 2.0, path="scalar")
                row["step_us_inputs_ready" if flag else "step_us"] = round(_loop_us(step, stream), 3)
            emit(row)
    elif args.mode == "crossover_stacked":
        d = 4096
        for K, r in ((16, 16), (4, 64), (32, 16), (8, 64), (64, 16), (16, 64)):
            for k in (1, 2, 4):
                for b in (1024, 2048, 4096, 8192):
                    g_ = torch.Generator().manual_seed(b + 7 * K + r + k)
                    x = torch.randn(b, d, generator=g_).to(torch.bfloat16).to(dev)
                    A = (torch.randn(K, d, r, generator=g_) / math.sqrt(d)).to(torch.bfloat16).to(dev)
                    B = (torch.randn(K, r, d, generator=g_) / math.sqrt(r)).to(torch.bfloat16).to(dev)
                    y = torch.randn(b, d, generator=g_).to(dev)
                    ids = torch.stack([torch.randperm(K, generator=g_)[:k] for _ in range(b)]).to(torch.int32).to(dev)
                    w = torch.softmax(torch.randn(b, k, generator=g_), dim=1).to(dev)
                    counts = torch.empty(K, dtype=torch.int32, device=dev)
                    offsets = torch.empty(K + 1, dtype=torch.int32, device=dev)
                    perm = torch.empty(b * k, dtype=torch.int32, device=dev)
                    need = m.molora_workspace_bytes(b, d, d, K, r, k, path="stacked")
                    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
                    row = {"mode": "crossover_stacked", "d": d, "K": K, "r": r, "k": k, "batch": b,
                           "auto_with_ws": m.molora_select_path(torch.bfloat16, b, d, d, K, r, k)}

                    def grouped():
                        m.molora_dispatch(ids, K, counts=counts, offsets=offsets, perm=perm)
                        m.molora_lora_apply(x, A, B, ids, y, 2.0, w=w, counts=counts, offsets=offsets, perm=perm,
                                            path="grouped")

                    def stacked():
                        m.molora_lora_apply(x, A, B, ids, y, 2.0, w=w, path="stacked", ws=ws)

                    for name, fn in (("grouped", grouped), ("stacked", stacked)):
                        row[f"{name}_us_warm"] = round(_loop_us(fn, stream, n=20, reps=3), 3)
                    row["faster"] = "stacked" if row["stacked_us_warm"] < row["grouped_us_warm"] else "grouped"
                    emit(row)
                    del x, A, B, y, ids, w, ws
    elif args.mode == "crossover":
        for r, dist in ((r, dist) for r in (int(v) for v in args.ranks.split(",")) for dist in ("uniform", "zipf")):
            for K in (4, 8, 16, 32, 64):
                for b in (1, 8, 32, 64, 128, 160, 256, 384, 512, 768, 1024, 1536, 2048):
                    wl = workloads.make("decode_sweep", N=b, K=K, r=r, dist=dist)
                    tok, starts = wl.tok.to(dev), wl.starts.to(dev)
                    x, A, B, y = wl.x.to(dev), wl.A.to(dev), wl.B.to(dev), wl.y0.to(dev)
                    adapter = torch.empty(b, dtype=torch.int32, device=dev)
                    counts = torch.empty(K, dtype=torch.int32, device=dev)
                    offsets = torch.empty(K + 1, dtype=torch.int32, device=dev)
                    perm = torch.empty(b, dtype=torch.int32, device=dev)
                    row = {"mode": "crossover", "dist": dist, "K": K, "r": r, "batch": b}
                    for path in ("scalar", "grouped"):
                        def fn(path=path):
                            # each path with the routing it needs: the token-major scalar apply
                            # takes the ids as they are; the grouped apply needs the dispatch
                            if path == "scalar":
                                m.molora_route_vocab(tok, starts, adapter=adapter)
                            else:
                                m.molora_route_vocab_dispatch(tok, starts, adapter=adapter, counts=counts,
                                                              offsets=offsets, perm=perm)
                            m.molora_lora_apply(x, A, B, adapter, y, wl.scale, counts=counts, offsets=offsets,
                                                perm=perm, path=path)
                        ms = _replay_ms(_graph(fn, stream), stream, 30, flush)
                        row[f"{path}_us_p50"] = round(_pct(ms, 0.5) * 1e3, 2)
                        row[f"{path}_us_warm"] = round(_loop_us(fn, stream), 3)
                    row["distinct_adapters"] = int(torch.unique(adapter).numel())
                    row["faster"] = "grouped" if row["grouped_us_warm"] < row["scalar_us_warm"] else "scalar"
                    emit(row)
    elif args.mode == "topk":
        peak = measured_peaks()[0].get("hbm_gbs")
        arms = set(args.topk_arms.split(","))
        for k in (int(v) for v in args.topk_k.split(",")):
            wl = workloads.make("topk_scaling", k=k)
            x, W1, W2, A, B, y = (wl.x.to(dev), wl.W1.to(dev), wl.W2.to(dev), wl.A.to(dev), wl.B.to(dev),
                                  wl.y0.to(dev))
            ids = torch.empty(wl.N, k, dtype=torch.int32, device=dev)
            w = torch.empty(wl.N, k, dtype=torch.float32, device=dev)
            counts = torch.empty(wl.K, dtype=torch.int32, device=dev)
            offsets = torch.empty(wl.K + 1, dtype=torch.int32, device=dev)
            perm = torch.empty(wl.N * k, dtype=torch.int32, device=dev)
            need = m.molora_workspace_bytes(wl.N, wl.d_in, wl.d_out, wl.K, wl.r, k, router=True)
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

            def fused():  # router + stacked apply: x read once, one y update per token
                m.molora_router_lora_apply(x, W1, W2, A, B, k, y, wl.scale, ids=ids, w=w, want_logits=False, ws=ws)

            def grouped():  # router -> dispatch -> grouped apply (k gathers and k reductions per token)
                m.molora_router_topk(x, W1, W2, k, ids=ids, w=w, want_logits=False)
                m.molora_dispatch(ids, wl.K, counts=counts, offsets=offsets, perm=perm)
                m.molora_lora_apply(x, A, B, ids, y, wl.scale, w=w, counts=counts, offsets=offsets, perm=perm,
                                    path="grouped")
            # algorithmic bytes: x once, y read + written, every adapter's A and B, W1, ids and w
            nbytes = (wl.N * wl.d_in * 2 + 2 * wl.N * wl.d_out * 4 + wl.K * (wl.d_in * wl.r + wl.r * wl.d_out) * 2
                      + wl.d_in * 64 * 2 + wl.N * 2 * k * 4)
            res = {}
            for name, fn, reps in (("fused_stacked", fused, args.replays), ("grouped", grouped, min(args.replays, 200))):
                if name not in arms:
                    continue
                g_arm = _graph(fn, stream)
                clocks = ClockSampler(0)
                clocks.start()
                ms = _replay_ms(g_arm, stream, reps)
                clk = clocks.stop()
                p50, p99 = _pct(ms, 0.5), _pct(ms, 0.99)
                res[name] = {"p50_ms": round(p50, 5), "p99_ms": round(p99, 5), "replays": reps, "clocks": clk,
                             "tokens_per_s_p50": round(wl.N / (p50 * 1e-3), 1),
                             "GBps_p50": round(nbytes / (p50 * 1e-3) / 1e9, 1),
                             "frac_of_measured_hbm": round(nbytes / (p50 * 1e-3) / 1e9 / peak, 3) if peak else None}
            if "router" in arms:
                r_ms = _replay_ms(_graph(lambda: m.molora_router_topk(x, W1, W2, k, ids=ids, w=w, want_logits=False),
                                         stream), stream, min(args.replays, 200))
                rb = wl.N * wl.d_in * 2 + wl.d_in * 64 * 2 + 64 * wl.K * 2 + wl.N * 2 * k * 4  # x, W1, W2, ids, w
                res["router_alone_us_p50"] = round(_pct(r_ms, 0.5) * 1e3, 2)
                res["router_alone_us_p99"] = round(_pct(r_ms, 0.99) * 1e3, 2)
                res["router_alone_GBps_p50"] = round(rb / (_pct(r_ms, 0.5) * 1e-3) / 1e9, 1)
                res["router_alone_frac_of_measured_hbm"] = (round(rb / (_pct(r_ms, 0.5) * 1e-3) / 1e9 / peak, 3)
                                                            if peak else None)
                # back to back in one graph (no per-call graph launch), x from DRAM
                lus, nbx = _router_loop(m, wl, k, stream, dev)
                res["router_b2b_loop"] = {"us_per_call": round(lus, 2), "GBps": round(rb / (lus * 1e-6) / 1e9, 1),
                                          "frac_of_measured_hbm": round(rb / (lus * 1e-6) / 1e9 / peak, 3) if peak else None,
                                          "timing": f"30 calls in one CUDA graph over {nbx} x batches (> L2)"}
            emit({"mode": "topk", "workload": "N=8192, d=4096, K=8, r=64, router d->64->K", "k": k,
                  "algorithmic_bytes": nbytes, **res,
                  "l2": "not flushed (back-to-back replays; 344 MB of inputs and outputs exceed the L2)"})
    elif args.mode == "router":
        wl = workloads.make("topk_mlp")
        x, W1, W2, A, B, y = (wl.x.to(dev), wl.W1.to(dev), wl.W2.to(dev), wl.A.to(dev), wl.B.to(dev),
                              wl.y0.to(dev))
        logits = torch.empty(wl.N, wl.K, dtype=torch.float32, device=dev)
        ids = torch.empty(wl.N, wl.k, dtype=torch.int32, device=dev)
        w = torch.empty(wl.N, wl.k, dtype=torch.float32, device=dev)
        counts = torch.empty(wl.K, dtype=torch.int32, device=dev)
        offsets = torch.empty(wl.K + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(wl.N * wl.k, dtype=torch.int32, device=dev)
        g_router = _graph(lambda: m.molora_router_topk(x, W1, W2, wl.k, logits=logits, ids=ids, w=w), stream)

        def path_grouped():
            m.molora_router_topk(x, W1, W2, wl.k, logits=logits, ids=ids, w=w)
            m.molora_dispatch(ids, wl.K, counts=counts, offsets=offsets, perm=perm)
            m.molora_lora_apply(x, A, B, ids, y, wl.scale, w=w, counts=counts, offsets=offsets, perm=perm,
                                path="grouped")

        def path_dense():  # no dispatch: the dense apply reads ids and w directly
            m.molora_router_topk(x, W1, W2, wl.k, logits=logits, ids=ids, w=w)
            m.molora_lora_apply(x, A, B, ids, y, wl.scale, w=w, path="dense")

        def path_fused():  # router and dense apply in one kernel: x is read once
            m.molora_router_lora_apply(x, W1, W2, A, B, wl.k, y, wl.scale, logits=logits, ids=ids, w=w, use_ws=False)

        ws = torch.empty(max(256, m.molora_workspace_bytes(wl.N, wl.d_in, wl.d_out, wl.K, wl.r, wl.k, path="stacked")),
                         dtype=torch.uint8, device=dev)

        def path_stacked():  # router in the stacked shrink, then the expand GEMM: x read once
            m.molora_router_lora_apply(x, W1, W2, A, B, wl.k, y, wl.scale, logits=logits, ids=ids, w=w, ws=ws)

        r_ms = _replay_ms(g_router, stream, 100, flush)
        res = {}
        # the router alone back to back (no flush), 200 replays
        peak = measured_peaks()[0].get("hbm_gbs")
        rb = wl.N * wl.d_in * 2 + wl.d_in * 64 * 2 + wl.N * (wl.K + 2 * wl.k) * 4
        rms = _replay_ms(g_router, stream, 200)
        res["b2b_router"] = {"p50_us": round(_pct(rms, 0.5) * 1e3, 2), "p99_us": round(_pct(rms, 0.99) * 1e3, 2),
                             "GBps_p50": round(rb / (_pct(rms, 0.5) * 1e-3) / 1e9, 1),
                             "frac_of_measured_hbm": (round(rb / (_pct(rms, 0.5) * 1e-3) / 1e9 / peak, 3)
                                                      if peak else None),
                             "timing": "one graph replay per call, events around each (graph launch included)"}
        lus, nbx = _router_loop(m, wl, wl.k, stream, dev)
        res["router_b2b_loop"] = {"us_per_call": round(lus, 2), "GBps": round(rb / (lus * 1e-6) / 1e9, 1),
                                  "frac_of_measured_hbm": round(rb / (lus * 1e-6) / 1e9 / peak, 3) if peak else None,
                                  "timing": f"30 calls in one CUDA graph over {nbx} x batches (> L2)"}
        for name, fn in (("grouped", path_grouped), ("dense", path_dense), ("fused", path_fused),
                         ("fused_stacked", path_stacked)):
            res[f"path_{name}_us_p50"] = round(_pct(_replay_ms(_graph(fn, stream), stream, 100, flush), 0.5) * 1e3, 2)
        # the two one-pass paths back to back (no flush), 200 replays: p50, p99 and the fraction of
        # measured HBM for x once, y read + written, A, B, W1, logits, ids and w
        nbytes = (wl.N * wl.d_in * 2 + 2 * wl.N * wl.d_out * 4 + wl.K * (wl.d_in * wl.r + wl.r * wl.d_out) * 2
                  + wl.d_in * 64 * 2 + wl.N * (wl.K + 2 * wl.k) * 4)
        for name, fn in (("fused", path_fused), ("fused_stacked", path_stacked)):
            ms = _replay_ms(_graph(fn, stream), stream, 200)
            p50, p99 = _pct(ms, 0.5), _pct(ms, 0.99)
            res[f"b2b_{name}"] = {"p50_us": round(p50 * 1e3, 2), "p99_us": round(p99 * 1e3, 2),
                                  "tokens_per_s_p50": round(wl.N / (p50 * 1e-3), 1),
                                  "frac_of_measured_hbm": round(nbytes / (p50 * 1e-3) / 1e9 / peak, 3) if peak else None}
        # the one-kernel path as the main line times it: 20 calls in one CUDA graph over three
        # (x, y) batches (350 MB, more than the L2), one event pair around the replay
        gb = torch.Generator().manual_seed(8765)
        lb = [(x, y)] + [(torch.randn(x.shape, generator=gb).to(x.dtype).to(dev),
                          torch.randn(y.shape, generator=gb).to(dev)) for _ in range(2)]
        st = {"i": 0}

        def fused_rot():
            xb, yb = lb[st["i"] % len(lb)]
            st["i"] += 1
            m.molora_router_lora_apply(xb, W1, W2, A, B, wl.k, yb, wl.scale, logits=logits, ids=ids, w=w,
                                       use_ws=False)
        lus = _loop_us(fused_rot, stream, n=20, reps=7)
        res["b2b_fused_loop"] = {"us_per_call": round(lus, 2), "tokens_per_s": round(wl.N / (lus * 1e-6), 1),
                                 "frac_of_measured_hbm": round(nbytes / (lus * 1e-6) / 1e9 / peak, 3) if peak else None,
                                 "timing": "20 calls in one CUDA graph over 3 (x, y) batches (> L2)"}
        res["algorithmic_bytes"] = nbytes
        path_grouped()  # ids, w, counts, offsets and perm for the apply-only graphs
        torch.cuda.synchronize()
        for name in ("grouped", "dense"):
            g_ap = _graph(lambda name=name: m.molora_lora_apply(x, A, B, ids, y, wl.scale, w=w, counts=counts,
                                                                 offsets=offsets, perm=perm, path=name), stream)
            res[f"apply_{name}_us_p50"] = round(_pct(_replay_ms(g_ap, stream, 100, flush), 0.5) * 1e3, 2)
        auto = m.molora_select_path(torch.bfloat16, wl.N, wl.d_in, wl.d_out, wl.K, wl.r, wl.k)
        best = res[f"path_{auto}_us_p50"]
        rb = wl.N * wl.d_in * 2 + wl.d_in * 64 * 2 + wl.N * (wl.K + 2 * wl.k) * 4
        emit({"mode": "router", "workload": "N=4096, d_in=2048, d_out=6144, K=4, r=16, k=2",
              "router_us_p50": round(_pct(r_ms, 0.5) * 1e3, 2),
              "router_GBps": round(rb / (_pct(r_ms, 0.5) * 1e-3) / 1e9, 1),
              "router_tflops": round(2 * wl.N * wl.d_in * 64 / (_pct(r_ms, 0.5) * 1e-3) / 1e12, 1),
              **res, "auto_path": auto, "path_us_p50": best,
              "fused_tokens_per_s": round(wl.N / (res["path_fused_us_p50"] * 1e-6), 1),
              "path_tokens_per_s": round(wl.N / (best * 1e-6), 1), "l2": "flushed between replays"})
    elif args.mode == "kernels":
        # single-kernel invocations at the shapes where AUTO uses them, for per-kernel rooflines
        # and ncu captures: the scalar apply at decode batches (d = 4096, r = 16, K = 16 hot-set
        # adapters, top-1 uniform) and the CUDA-core router on fp32 x (the learned-router shape)
        peak = measured_peaks()[0].get("hbm_gbs")
        for b in (160, 512):
            wl = workloads.make("decode_sweep", N=b, K=16)
            x, A, B, y = wl.x.to(dev), wl.A.to(dev), wl.B.to(dev), wl.y0.to(dev)
            adapter = m.molora_route_vocab(wl.tok.to(dev), wl.starts.to(dev))
            torch.cuda.synchronize()
            used = int((torch.bincount(adapter.cpu().long(), minlength=wl.K) > 0).sum().item())
            us = _loop_us(lambda: m.molora_lora_apply(x, A, B, adapter, y, wl.scale, path="scalar"), stream)
            nbytes = b * wl.d_in * 2 + 2 * b * wl.d_out * 4 + used * (wl.d_in * wl.r + wl.r * wl.d_out) * 2 + b * 4
            emit({"mode": "kernels", "kernel": "lora_scalar_kernel",
                  "workload": f"batch {b}, d_in=d_out=4096, K=16 hot-set adapters ({used} touched), r=16, top-1",
                  "us_per_call": round(us, 3), "algorithmic_bytes": nbytes,
                  "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                  "frac_of_measured_hbm": round(nbytes / (us * 1e-6) / 1e9 / peak, 3) if peak else None,
                  "timing": "50 calls back to back in one CUDA graph (the hot set stays in L2)"})
        wl = workloads.make("topk_mlp", dtype=torch.float32)
        x, W1, W2 = wl.x.to(dev), wl.W1.to(dev), wl.W2.to(dev)
        ids = torch.empty(wl.N, wl.k, dtype=torch.int32, device=dev)
        w = torch.empty(wl.N, wl.k, dtype=torch.float32, device=dev)
        us = _loop_us(lambda: m.molora_router_topk(x, W1, W2, wl.k, ids=ids, w=w, want_logits=False), stream, n=20)
        nbytes = wl.N * wl.d_in * 4 + wl.d_in * 64 * 4 + 64 * wl.K * 4 + wl.N * 2 * wl.k * 4
        emit({"mode": "kernels", "kernel": "router_scalar_kernel",
              "workload": "fp32 x, N=4096, d_in=2048 -> 64 -> K=4, top-2", "us_per_call": round(us, 3),
              "algorithmic_bytes": nbytes, "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
              "frac_of_measured_hbm": round(nbytes / (us * 1e-6) / 1e9 / peak, 3) if peak else None,
              "timing": "20 calls back to back in one CUDA graph (x is 33.6 MB: L2-resident)"})
    elif args.mode == "cv":
        for dist, b in ((dist, b) for dist in ("uniform", "zipf") for b in (32, 64, 128, 256)):
            wl = workloads.make("decode_sweep", N=b, K=16, dist=dist)
            tok, starts = wl.tok.to(dev), wl.starts.to(dev)
            x, A, B, y = wl.x.to(dev), wl.A.to(dev), wl.B.to(dev), wl.y0.to(dev)
            adapter = torch.empty(b, dtype=torch.int32, device=dev)
            counts = torch.empty(wl.K, dtype=torch.int32, device=dev)
            offsets = torch.empty(wl.K + 1, dtype=torch.int32, device=dev)
            perm = torch.empty(b, dtype=torch.int32, device=dev)

            def step():
                m.molora_route_vocab_dispatch(tok, starts, adapter=adapter, counts=counts, offsets=offsets, perm=perm)
                m.molora_lora_apply(x, A, B, adapter, y, wl.scale, counts=counts, offsets=offsets, perm=perm)
            g = _graph(step, stream)

            def spread(fn, n=1000):
                with torch.cuda.stream(stream):
                    for _ in range(50):
                        fn()
                    stream.synchronize()
                    ts = []
                    for _ in range(n):
                        t0 = time.perf_counter()
                        fn()
                        stream.synchronize()
                        ts.append((time.perf_counter() - t0) * 1e6)
                ts.sort()
                mean = statistics.fmean(ts)
                return {"mean_us": round(mean, 2), "p50_us": round(_pct(ts, 0.5), 2), "p99_us": round(_pct(ts, 0.99), 2),
                        "cv": round(statistics.pstdev(ts) / mean, 3)}
            emit({"mode": "cv", "batch": b, "K": wl.K, "r": wl.r, "dist": dist, "eager": spread(step), "graph": spread(g.replay),
                  "timing": "host clock around launch + synchronize, 1000 steps after 50 warm-up"})
    elif args.mode == "perseq":
        for r in (int(v) for v in args.ranks.split(",")):
            wl = workloads.make(WORKLOAD, r=r)
            tok, starts = wl.tok.to(dev), wl.starts.to(dev)
            x, A, B, y = wl.x.to(dev), wl.A.to(dev), wl.B.to(dev), wl.y0.to(dev)
            adapter = torch.empty(wl.N, dtype=torch.int32, device=dev)
            counts = torch.empty(wl.K, dtype=torch.int32, device=dev)
            offsets = torch.empty(wl.K + 1, dtype=torch.int32, device=dev)
            perm = torch.empty(wl.N, dtype=torch.int32, device=dev)

            def per_token():
                m.molora_route_vocab_dispatch(tok, starts, adapter=adapter, counts=counts, offsets=offsets, perm=perm)
                m.molora_lora_apply(x, A, B, adapter, y, wl.scale, counts=counts, offsets=offsets, perm=perm)

            def per_sequence():
                m.molora_route_vocab(tok, starts, adapter=adapter)
                for a in range(wl.K):
                    m.molora_lora_apply_masked_pass(x, A, B, adapter, a, y, wl.scale)
            t_ms = _replay_ms(_graph(per_token, stream), stream, 100, flush)
            s_ms = _replay_ms(_graph(per_sequence, stream), stream, 100, flush)
            emit({"mode": "perseq", "workload": f"N=2048, d=4096, K=4, r={r} (4-modality benchmark shape)",
                  "per_token_us_p50": round(_pct(t_ms, 0.5) * 1e3, 2),
                  "per_sequence_us_p50": round(_pct(s_ms, 0.5) * 1e3, 2),
                  "passes": {"per_token": 1, "per_sequence": wl.K},
                  "speedup": round(_pct(s_ms, 0.5) / _pct(t_ms, 0.5), 2), "l2": "flushed between replays"})
    return 0


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.mode != "step":
        return run_mode(args) if rank == 0 else 0
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    res = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
