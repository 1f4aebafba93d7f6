"""Throughput of the affine group-quantized mat-vec (qmv) on one GB300.

One step = one qmv call on the 12B-class decode projection (N=15360, K=3840,
4-bit affine, group 64, bf16 scale/bias/x, fp32 accumulate, bf16 y), M = 1.
The same measurement at M = 13 (the streamed kernel) is reported beside it,
and under "mxfp4" the mxfp4 mode (E2M1 codes, one E8M0 scale per 32) on the
same shape at M = 1 and M = 13.

Device timing: the K steps run as CUDA-graph replays on one stream,
bracketed by CUDA events; each step reads a different one of R copies of the
weights whose total exceeds twice the L2 size, so weights come from HBM.
``value`` = algorithmic bytes per call / device time per call (GB/s), the
bytes being W + scales + biases + x + y (weights read once for all M).

``e2e``: the same calls through the public Python API, each step copying x
from pinned host memory and reading y back to pinned host memory.

``--impl reference`` times the CPU oracle (fp32 factored form, all host
cores) on the same workload instead: the oracle is the reference arm here.

Launch: ``python bench.py [--gpus N --steps K --warmup W]``; for N > 1 under
torchrun each rank runs its own replica (the path has no exchange step) and
rank 0 prints the whole-job line.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "qmv achieved HBM GB/s & % of GB300 roofline at M=1 and M=13 (µs/call)"
WORKLOAD = "proj_15360x3840_4b_g64"
MX_WORKLOAD = "proj_15360x3840_mxfp4"
KERNEL_SOURCES = ["qmv_kernel.cuh", "qmv_plan.h", "qmv_launch.cuh", "qmv_api.cu"]
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes per launch of qmv_m1 (dram__bytes_read.sum + dram__bytes_write.sum)
# from one ncu capture of the bench workload, keyed by a hash of the kernel
# sources it was taken on; a changed kernel reports null until recaptured.
NCU_TRAFFIC = {"8863dc143765fe42": 33252096}


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "group_quantized_mat_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def algorithmic_bytes(N, K, M, bits, gs):
    return N * K * bits // 8 + 4 * N * (K // gs) + 2 * M * (K + N)


def mx_algorithmic_bytes(N, K, M):
    """mxfp4: 4-bit codes, one scale byte per 32, bf16 x and y."""
    return N * K // 2 + N * (K // 32) + 2 * M * (K + N)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's `value` (timed-region milliseconds): the
    job's time. One rank: the value itself."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_call: int, calls_per_rank: int, world: int, job_ms: float) -> float:
    """Whole-job throughput: the bytes all ranks processed over the job's time."""
    return world * calls_per_rank * bytes_per_call / (job_ms * 1e-3) / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- GPU arm
EXTRA_STEPS = 2000        # calls per side measurement (at most --steps)
WARM_CALLS = 2000         # untimed calls queued right before every timed region
SWEEP_MS = (1, 2, 4, 5, 10, 13, 16)
STACK = ("l27b_5120x5120_4b_g64", "l27b_1024x5120_4b_g64", "l27b_17408x5120_4b_g64", "l27b_5120x17408_4b_g64")
TWO_BIT = ("proj_15360x3840_2b_g64", "proj_15360x3840_2b_g128")
CHUNK = 500               # calls per captured graph


def run_gpu(args, rank, world, local_rank):
    import torch

    import group_quantized_mat_gb300 as g
    import synth
    from group_quantized_mat_gb300 import build as libbuild

    libbuild.build()
    g.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.Stream(device=dev)

    def tdev(a):
        a = a.view(np.int16) if a.dtype == np.uint16 else a.view(np.int32)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    cache = {}

    def problem(name):
        """R rotating device copies of the workload's weights, scales and biases
        (R * bytes > 2x L2, so every call reads its weights from HBM), and 16
        activation vectors."""
        if name not in cache:
            w = synth.WORKLOADS[name]
            inp = synth.make_inputs(w["N"], w["K"], 16, w["bits"], w["group_size"], seed=0)
            w_host = g.qmv_pack(inp.q, w["bits"])
            set_bytes = w_host.nbytes + inp.scales.nbytes + inp.biases.nbytes
            R = max(2, int(np.ceil(2.0 * l2 / set_bytes)) + 1)
            sets = [(tdev(w_host), tdev(inp.scales), tdev(inp.biases)) for _ in range(R)]
            cache[name] = dict(w, R=R, set_bytes=set_bytes, sets=sets, x=tdev(inp.x), inp=inp)
        return cache[name]

    def timed(call, steps, clocks=False):
        """`warmup` plain calls; then `steps` calls captured as CUDA graphs of
        at most CHUNK calls. The timed replays are enqueued right behind
        untimed replays of at least WARM_CALLS calls, with no host
        synchronization in between, so the GPU is busy when the start event
        runs and the host's graph submissions overlap GPU work; the events on
        the launch stream bracket exactly `steps` calls. Returns (job
        milliseconds, clock summary or None, timing description)."""
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                call(i)
        torch.cuda.synchronize()
        n_chunks, rem = divmod(steps, CHUNK)
        graphs = []
        with torch.cuda.stream(stream):
            for size in ([CHUNK] if n_chunks else []) + ([rem] if rem else []):
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=stream):
                    for i in range(size):
                        call(i)
                graphs.append(gr)
            for gr in graphs:  # uploads the graphs
                gr.replay()
        torch.cuda.synchronize()
        big = graphs[0] if n_chunks else None
        tail = graphs[-1] if rem else None
        warm = big if big is not None else tail
        warm_reps = max(3, -(-WARM_CALLS // (CHUNK if big is not None else rem)))
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        clk = ClockSampler(local_rank) if clocks else None
        if clk:
            clk.__enter__()
        with torch.cuda.stream(stream):
            for _ in range(warm_reps):
                warm.replay()
            start.record(stream)
            for _ in range(n_chunks):
                big.replay()
            if tail is not None:
                tail.replay()
            end.record(stream)
        torch.cuda.synchronize()
        if clk:
            clk.__exit__(None, None, None)
        if world > 1:
            torch.distributed.barrier()
        ms = max_over_ranks(start.elapsed_time(end), world, dev)
        desc = (f"{steps} calls timed as {n_chunks} CUDA-graph replays of {CHUNK} calls"
                + (f" and one of {rem}" if n_chunks and rem else "" if n_chunks else f" (one replay of {rem})")
                + f", enqueued behind {warm_reps} untimed replays of the same graph with no host sync between;"
                  " CUDA events on the launch stream")
        return ms, (clk.summary() if clk else None), desc

    def measure(name, M, flags=0, steps=None, clocks=False):
        pr = problem(name)
        N, K, bits, gs, R, sets = pr["N"], pr["K"], pr["bits"], pr["group_size"], pr["R"], pr["sets"]
        x = pr["x"][:M].contiguous()
        y = torch.empty((M, N), dtype=torch.int16, device=dev)

        def call(i):
            wq, s, b = sets[i % R]
            if flags:
                g.qmv_run_ex(wq, s, b, x, y, M, N, K, bits, gs, flags=flags, stream=stream)
            else:
                g.qmv_run(wq, s, b, x, y, M, N, K, bits, gs, stream=stream)

        steps = args.steps if steps is None else steps
        ms, ck, desc = timed(call, steps, clocks)
        return dict(ms=ms, steps=steps, clocks=ck, timing=desc, N=N, K=K, bits=bits, gs=gs, M=M, R=R,
                    set_bytes=pr["set_bytes"])

    def measure_stack(M, steps):
        """One step = the four matrices of the 27B-class layer in turn."""
        prs = [problem(n) for n in STACK]
        xs = [pr["x"][:M].contiguous() for pr in prs]
        ys = [torch.empty((M, pr["N"]), dtype=torch.int16, device=dev) for pr in prs]

        def call(i):
            for pr, x, y in zip(prs, xs, ys):
                wq, s, b = pr["sets"][i % pr["R"]]
                g.qmv_run(wq, s, b, x, y, M, pr["N"], pr["K"], pr["bits"], pr["group_size"], stream=stream)

        ms, _, _ = timed(call, steps)
        return ms

    def measure_e2e(M, steps):
        pr = problem(WORKLOAD)
        N, K, bits, gs, R, sets = pr["N"], pr["K"], pr["bits"], pr["group_size"], pr["R"], pr["sets"]
        x_host = torch.from_numpy(pr["inp"].x[:M].view(np.int16).copy()).pin_memory()
        y_host = torch.empty((M, N), dtype=torch.int16).pin_memory()
        x = torch.empty((M, K), dtype=torch.int16, device=dev)
        y = torch.empty((M, N), dtype=torch.int16, device=dev)

        def step(i):
            wq, s, b = sets[i % R]
            x.copy_(x_host, non_blocking=True)
            g.qmv_run(wq, s, b, x, y, M, N, K, bits, gs, stream=stream)
            y_host.copy_(y, non_blocking=True)

        with torch.cuda.stream(stream):
            for i in range(min(args.warmup, 50)):
                step(i)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(steps):
                step(i)
            end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / steps, M * K * 2, M * N * 2

    head1 = measure(WORKLOAD, 1, clocks=True)
    head13 = measure(WORKLOAD, 13, clocks=True)

    # side measurements: the MTP verify sweep on both projection shapes, the
    # same 13 vectors as 13 one-vector launches, the 27B-class stack, the
    # 2-bit variants, and the opt-in programmatic-dependency launch
    xs = min(args.steps, EXTRA_STEPS)
    sweep = {}
    for name in (WORKLOAD, "down_3840x15360_4b_g64"):
        sweep[name] = {M: (head1 if (name == WORKLOAD and M == 1) else head13 if (name == WORKLOAD and M == 13)
                           else measure(name, M, steps=xs)) for M in SWEEP_MS}
    per_column = {name: measure(name, 13, flags=g.FORCE_M1_PER_COLUMN, steps=xs)
                  for name in (WORKLOAD, "down_3840x15360_4b_g64")}
    stack = {name: {M: measure(name, M, steps=xs) for M in (1, 13)} for name in STACK}
    stack_step = {M: measure_stack(M, xs) for M in (1, 13)}
    two_bit = {name: {M: measure(name, M, steps=xs) for M in (1, 13)} for name in TWO_BIT}
    pdl = measure(WORKLOAD, 1, flags=g.PDL, steps=xs)
    for name in list(cache):
        if name != WORKLOAD:
            del cache[name]

    # the mxfp4 mode on the same projection shape
    mxw = synth.MX_WORKLOADS[MX_WORKLOAD]
    mN, mK = mxw["N"], mxw["K"]
    minp = synth.make_mxfp4_inputs(mN, mK, 16, seed=0)
    mw_host = g.qmv_pack(minp.codes, 4)
    mset_bytes = mw_host.nbytes + minp.scales.nbytes
    mR = max(2, int(np.ceil(2.0 * l2 / mset_bytes)) + 1)
    msets = [(tdev(mw_host), torch.from_numpy(np.ascontiguousarray(minp.scales)).to(dev)) for _ in range(mR)]
    mx_steps = min(args.steps, 50000)

    def measure_mx(M):
        x = tdev(minp.x[:M])
        y = torch.empty((M, mN), dtype=torch.int16, device=dev)

        def call(i):
            wq, sc = msets[i % mR]
            g.qmv_mxfp4_run(wq, sc, x, y, M, mN, mK, stream=stream)

        return timed(call, mx_steps, clocks=(M == 13))

    mx_ms1, _, _ = measure_mx(1)
    mx_ms13, mx_clocks13, _ = measure_mx(13)
    del msets
    e2e_steps = min(args.steps, 3000)
    e2e_ms, h2d, d2h = measure_e2e(1, e2e_steps)
    pr = problem(WORKLOAD)
    return dict(N=pr["N"], K=pr["K"], bits=pr["bits"], gs=pr["group_size"], R=pr["R"], set_bytes=pr["set_bytes"],
                l2=l2, ms1=head1["ms"], ms13=head13["ms"], clocks1=head1["clocks"], clocks13=head13["clocks"],
                timing=head1["timing"], e2e_ms=e2e_ms, e2e_steps=e2e_steps, h2d=h2d, d2h=d2h,
                sweep=sweep, per_column=per_column, stack=stack, stack_step=stack_step, two_bit=two_bit, pdl=pdl,
                extra_steps=xs,
                mx=dict(N=mN, K=mK, R=mR, set_bytes=mset_bytes, steps=mx_steps, ms1=mx_ms1, ms13=mx_ms13,
                        clocks13=mx_clocks13),
                sm_count=torch.cuda.get_device_properties(dev).multi_processor_count)


def call_summary(m, peak, fma_peak_tflops):
    """µs per call, GB/s and fractions of one side measurement."""
    us = m["ms"] * 1e3 / m["steps"]
    nbytes = algorithmic_bytes(m["N"], m["K"], m["M"], m["bits"], m["gs"])
    gbs = nbytes / (us * 1e-6) / 1e9
    d = {"us_per_call": round(us, 3), "achieved_gbs": round(gbs, 2), "hbm_frac": round(gbs / peak, 4)}
    if m["M"] > 1:
        tflops = 2.0 * m["N"] * m["K"] * m["M"] / (us * 1e-6) / 1e12
        d.update(fp32_tflops=round(tflops, 2), fp32_frac=round(tflops / fma_peak_tflops, 4))
    return d


def side_summary(r, peak, fma_peak_tflops):
    """The extra objects of the bench line (issue #1289 "Step 1" and
    "Acceptance criteria": the verify sweep and the recovered gap; PR #1681
    "What lands": the 27B-class stack; PR #159 "What": 2-bit, groups 64/128)."""
    us = lambda m: m["ms"] * 1e3 / m["steps"]
    sweep = {}
    for name, by_m in r["sweep"].items():
        t1 = us(by_m[1])
        sweep[name] = {f"m{M}": dict(call_summary(m, peak, fma_peak_tflops), ratio_to_m1=round(us(m) / t1, 3))
                       for M, m in by_m.items()}
    gap = {}
    for name, pc in r["per_column"].items():
        t_stream, t1, t_pc = us(r["sweep"][name][13]), us(r["sweep"][name][1]), us(pc)
        gap[name] = {"m13_streamed_us": round(t_stream, 3), "m13_as_13_launches_us": round(t_pc, 3),
                     "m1_us": round(t1, 3), "speedup_vs_13_launches": round(t_pc / t_stream, 3),
                     "recovered_frac": round((t_pc - t_stream) / (t_pc - t1), 4) if t_pc > t1 else None}
    stack = {name: {f"m{M}": call_summary(m, peak, fma_peak_tflops) for M, m in by_m.items()}
             for name, by_m in r["stack"].items()}
    for M, ms in r["stack_step"].items():
        nbytes = sum(algorithmic_bytes(r["stack"][n][M]["N"], r["stack"][n][M]["K"], M, 4, 64) for n in STACK)
        t = ms * 1e3 / r["extra_steps"]
        stack[f"stack_m{M}"] = {"us_per_step": round(t, 3), "bytes_per_step": nbytes,
                                "achieved_gbs": round(nbytes / (t * 1e-6) / 1e9, 2),
                                "hbm_frac": round(nbytes / (t * 1e-6) / 1e9 / peak, 4)}
    two_bit = {name: {f"m{M}": call_summary(m, peak, fma_peak_tflops) for M, m in by_m.items()}
               for name, by_m in r["two_bit"].items()}
    pdl = dict(call_summary(r["pdl"], peak, fma_peak_tflops),
               note="QMV_PDL (opt-in): each call may start streaming weights under the previous call's tail")
    return {"steps_each": r["extra_steps"], "mtp_sweep": sweep, "recovered_gap": gap, "stack_27b": stack,
            "two_bit": two_bit, "pdl_m1": pdl}


# --------------------------------------------------------------------------- CPU oracle
def oracle_timing(N, K, M, bits, gs, seconds=10.0, rows=None, repeats=None, threads=None):
    """fp32 factored oracle on `threads` host cores (all of them by default);
    returns (seconds per run, threads used, rows, runs)."""
    import synth
    from oracle import Oracle
    o = Oracle(0)
    inp = synth.make_inputs(N, K, M, bits, gs, seed=0)
    rows = N if rows is None else rows
    wq = o.pack(inp.q[:rows], bits)
    s, b = inp.scales[:rows], inp.biases[:rows]
    threads = len(os.sched_getaffinity(0)) if threads is None else int(threads)
    o.qmv_f32_factored(wq, s, b, inp.x, bits, gs, nthreads=threads)  # warm
    runs, t0 = 0, time.perf_counter()
    used = threads
    while True:
        _, _, used = o.qmv_f32_factored(wq, s, b, inp.x, bits, gs, nthreads=threads)
        runs += 1
        el = time.perf_counter() - t0
        if (repeats is not None and runs >= repeats) or (repeats is None and el >= seconds):
            break
    return el / runs, used, rows, runs


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import synth
    w = synth.WORKLOADS[WORKLOAD]
    N, K, bits, gs, M = w["N"], w["K"], w["bits"], w["group_size"], 1
    t_full, threads, _, _ = oracle_timing(N, K, M, bits, gs, repeats=1)
    budget = 60.0
    rows = int(max(1, min(N, N * budget / max(1e-9, (args.steps + args.warmup) * t_full))))
    if args.warmup:
        oracle_timing(N, K, M, bits, gs, rows=rows, repeats=args.warmup)
    t_step, threads, rows, runs = oracle_timing(N, K, M, bits, gs, rows=rows, repeats=args.steps)
    nbytes = algorithmic_bytes(rows, K, M, bits, gs)
    gbs = nbytes / t_step / 1e9
    sample = f"rows 0..{rows - 1} of the {N}x{K} 4-bit g64 problem, M=1, per step; {runs} steps"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; distributions of the tiny workload)",
        "config": {"workload": WORKLOAD, "N": N, "K": K, "M": M, "bits": bits, "group_size": gs},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def run_profile(args):
    """Plain launches of one workload for ncu: `warmup` untimed calls, then
    `steps` calls, each on a fresh weight copy (no graphs, no clock sampling)."""
    import torch

    import group_quantized_mat_gb300 as g
    import synth
    from group_quantized_mat_gb300 import build as libbuild

    libbuild.build()
    g.load()
    if args.workload in synth.MX_WORKLOADS:
        w = synth.MX_WORKLOADS[args.workload]
        N, K, M = w["N"], w["K"], args.M
        inp = synth.make_mxfp4_inputs(N, K, M, seed=0)
        codes = torch.from_numpy(g.qmv_pack(inp.codes, 4).view(np.int32))
        sets = [(codes.cuda(), torch.from_numpy(inp.scales).cuda()) for _ in range(2)]
        x = torch.from_numpy(inp.x.view(np.int16)).cuda()
        y = torch.empty((M, N), dtype=torch.int16, device="cuda")
        for i in range(args.warmup + args.steps):
            wd, sd = sets[i % 2]
            g.qmv_mxfp4_run(wd, sd, x, y, M, N, K)
        torch.cuda.synchronize()
        print(json.dumps({"profile": args.workload, "M": M, "launches": args.warmup + args.steps,
                          "bytes_per_launch": mx_algorithmic_bytes(N, K, M)}))
        return
    w = synth.WORKLOADS[args.workload]
    N, K, bits, gs, M = w["N"], w["K"], w["bits"], w["group_size"], args.M
    inp = synth.make_inputs(N, K, M, bits, gs, seed=0)
    wq = g.qmv_pack(inp.q, bits)

    def tdev(a):
        a = a.view(np.int16) if a.dtype == np.uint16 else a.view(np.int32)
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    copies = 2
    sets = [(tdev(wq), tdev(inp.scales), tdev(inp.biases)) for _ in range(copies)]
    x = tdev(inp.x)
    y = torch.empty((M, N), dtype=torch.int16, device="cuda")
    for i in range(args.warmup + args.steps):
        wd, sd, bd = sets[i % copies]
        g.qmv_run(wd, sd, bd, x, y, M, N, K, bits, gs)
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.workload, "M": M, "launches": args.warmup + args.steps,
                      "bytes_per_launch": algorithmic_bytes(N, K, M, bits, gs)}))


def mx_oracle_timing(K, rows=256, seconds=2.0):
    """The mxfp4 oracle (fp64 dequantize-then-dot, one thread) on `rows` rows of
    the workload's shape and distribution, M = 1: (seconds per run, runs)."""
    import synth
    from oracle import Oracle
    o = Oracle(0)
    inp = synth.make_mxfp4_inputs(rows, K, 1, seed=0)
    wq = o.pack(inp.codes, 4)
    o.mxfp4_qmv_f64(wq, inp.scales, inp.x)  # warm
    runs, t0 = 0, time.perf_counter()
    while True:
        o.mxfp4_qmv_f64(wq, inp.scales, inp.x)
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return el / runs, runs


def mx_summary(mx, peak, fma_peak_tflops, cpu=None):
    """The mxfp4 mode's side measurement (same shape, E2M1 codes + E8M0 scales).
    `cpu` = (rows, seconds per run, runs) of the oracle timed beside it, or None."""
    N, K, steps = mx["N"], mx["K"], mx["steps"]
    out = {"workload": MX_WORKLOAD, "N": N, "K": K, "steps": steps, "kernel": "qmv_mxfp4<V> (V = M)",
           "l2": f"inputs > L2: {mx['R']} rotating copies of {mx['set_bytes'] / 1e6:.1f} MB"}
    if cpu is not None:
        rows, t, runs = cpu
        out["cpu_oracle"] = {"value": round(mx_algorithmic_bytes(rows, K, 1) / t / 1e9, 5), "unit": "GB/s",
                             "cores": 1, "kind": "oracle",
                             "sample": f"{rows} rows x {K}, M=1, fp64 dequantize-then-dot, {runs} runs"}
    for M, ms in ((1, mx["ms1"]), (13, mx["ms13"])):
        us = ms * 1e3 / steps
        nbytes = mx_algorithmic_bytes(N, K, M)
        gbs = nbytes / (us * 1e-6) / 1e9
        d = {"us_per_call": round(us, 3), "achieved_gbs": round(gbs, 2), "hbm_frac": round(gbs / peak, 4),
             "bytes_per_launch": nbytes}
        if M > 1:
            tflops = 2.0 * N * K * M / (us * 1e-6) / 1e12
            d.update(fp32_tflops=round(tflops, 2), fp32_frac=round(tflops / fma_peak_tflops, 4),
                     ratio_to_m1=round(ms / mx["ms1"], 3), clocks=mx["clocks13"])
        out[f"m{M}"] = d
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", action="store_true", help="plain launches for ncu (see run_profile)")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")

    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    r = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        N, K, bits, gs = r["N"], r["K"], r["bits"], r["gs"]
        b1 = algorithmic_bytes(N, K, 1, bits, gs)
        b13 = algorithmic_bytes(N, K, 13, bits, gs)
        us1 = r["ms1"] * 1e3 / args.steps
        us13 = r["ms13"] * 1e3 / args.steps
        gbs1 = whole_job_gbs(b1, args.steps, 1, r["ms1"])  # per GPU
        gbs13 = whole_job_gbs(b13, args.steps, 1, r["ms13"])
        peak, peak_kind = measured_peaks()
        cpu_t, cpu_threads, cpu_rows, cpu_runs = oracle_timing(N, K, 1, bits, gs, seconds=args.cpu_seconds)
        cpu_gbs = b1 / cpu_t / 1e9
        # the same oracle on one core, over the first 1/16 of the rows
        one_rows = max(1, N // 16)
        one_t, _, _, one_runs = oracle_timing(N, K, 1, bits, gs, seconds=min(3.0, args.cpu_seconds), rows=one_rows,
                                              threads=1)
        one_gbs = algorithmic_bytes(one_rows, K, 1, bits, gs) / one_t / 1e9
        e2e_gbs = b1 / (r["e2e_ms"] * 1e-3) / 1e9
        kh = kernel_hash()
        traffic = NCU_TRAFFIC.get(kh)
        # FP32-lane roofline for the streamed case: 2 flop per (element, vector)
        fma_peak_tflops = r["sm_count"] * 128 * 2 * 2.07e9 / 1e12
        flops13 = 2.0 * N * K * 13
        line = {
            "metric": METRIC,
            "value": round(whole_job_gbs(b1, args.steps, world, r["ms1"]), 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(r["ms1"] / args.steps, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded: q~U{0..15}, scale~U(0.001,0.02) bf16, bias=-8*scale+N(0,1e-3) bf16, x~N(0,1) bf16)",
            "config": {"workload": WORKLOAD, "N": N, "K": K, "M": 1, "bits": bits, "group_size": gs,
                       "l2": f"inputs > L2: {r['R']} rotating weight copies of {r['set_bytes'] / 1e6:.1f} MB "
                             f"({r['R'] * r['set_bytes'] / 1e6:.0f} MB) vs L2 {r['l2'] / 1e6:.0f} MB",
                       "timing": r["timing"],
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "us_per_call": round(us1, 3),
            "roofline": {"bound": "hbm", "achieved": round(gbs1, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs1 / peak, 4), "traffic": traffic,
                         "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "kernel": "qmv_m1<4,64>", "bytes_per_launch": b1},
            "m13": {"us_per_call": round(us13, 3), "achieved_gbs": round(gbs13, 2),
                    "hbm_frac": round(gbs13 / peak, 4), "ratio_to_m1": round(us13 / us1, 3),
                    "fp32_tflops": round(flops13 / (us13 * 1e-6) / 1e12, 2),
                    "fp32_lane_peak_tflops": round(fma_peak_tflops, 1),
                    "fp32_frac": round(flops13 / (us13 * 1e-6) / 1e12 / fma_peak_tflops, 4),
                    "kernel": "qmv_streamed<4,64,13>", "bytes_per_launch": b13, "clocks": r["clocks13"]},
            "mxfp4": mx_summary(r["mx"], peak, fma_peak_tflops, cpu=(256, *mx_oracle_timing(r["mx"]["K"]))),
            "side": side_summary(r, peak, fma_peak_tflops),
            "clocks": r["clocks1"],
            "e2e": {"value": round(world * e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"], "us_per_step": round(r["e2e_ms"] * 1e3, 3),
                    "steps": r["e2e_steps"], "api": "group_quantized_mat_gb300.qmv_run (C ABI qmv_run)"},
            "gpu_launches": args.steps,
            "cpu_baseline": {"value": round(cpu_gbs, 4), "unit": "GB/s", "cores": cpu_threads, "kind": "oracle",
                             "sample": f"full {N}x{K} M=1 problem (fp32 factored oracle), {cpu_runs} runs",
                             "single_core": {"value": round(one_gbs, 4), "unit": "GB/s", "cores": 1,
                                             "sample": f"rows 0..{one_rows - 1} of the same problem, {one_runs} runs"}},
            "kernel_hash": kh,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
