#!/usr/bin/env python3
"""Benchmark: GEMM TFLOP/s on one GB300 (and N replicas under torchrun).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME | --workload MxNxK[:AB[:IO[:bias]]]]
                    [--opt NAME=VALUE ...]

A step is one C = A·B (+bias) through the library on resident device inputs.
Default workload: M = N = K = 8192, fp16 row-major A, column-major B, fp32 bias,
fp16 output (the shape the >= 70 % of dense fp16 tensor peak target is quoted
on).  Prints one JSON line (rank 0).

--impl reference times the CPU oracle (a plain fp64 triple loop on the host
cores) on a bounded sample of the same workload: the comparison arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "gemm8192_f16_bias_f16out"
L2_BYTES = 129 * 1024 * 1024
METRIC = "GEMM TFLOPS (1×GB300) and fraction of dense fp16/fp32 roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference", "cublas"], default="ours",
                    help="ours: this library; reference: the CPU oracle on a bounded sample; "
                         "cublas: torch.mm/addmm (cuBLAS) on the same operands and protocol, "
                         "for context only (the library never calls it)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="a named workload of dense_gemm_tmem_gb300/inputs.py, or a shape "
                         "MxNxK[:AB[:IO[:bias]]] (A/B r|c for row/column-major, I/O h|f "
                         "for fp16/fp32; default rc and hh), e.g. 2048x2048x2048:rc:hh")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--eager", action="store_true",
                    help="launch the timed steps one by one from the host instead of "
                         "replaying them as one CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target duration of the CPU-baseline sample")
    ap.add_argument("--opt", action="append", default=[], metavar="NAME=VALUE",
                    help="set a library option before timing, e.g. DYNAMIC_TILES=0 or "
                         "GROUP_M=4 (the GEMM_OPT_ names of include/gemm.h); repeatable")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def flops_of(M, N, K):
    return 2.0 * M * N * K


def slowest_rank_ms(elapsed_ms, device, dist=None):
    """The timed region's length on the slowest rank (all ranks get it): the
    whole job is done when the last replica is."""
    import torch
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, steps, step_flops, elapsed_ms):
    """Every rank's steps over the slowest rank's time (weak scaling: each
    replica runs the same workload)."""
    return world * steps * step_flops / (elapsed_ms * 1e-3) / 1e12


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def kernel_source_hash(files):
    """Hash of the listed kernel source files (in the listed order)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_gemm_tmem_gb300", "csrc")
    for fn in files:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


TRAFFIC_PLAN_KEYS = ("kernel", "tile_m", "tile_n", "grid", "group_m", "cluster_split", "k_group")


def recorded_traffic(workload, plan):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources of the kernel it names and with the same launch
    plan (the raster order and grid decide how much L2 reuse there is); else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f).get(workload)
        if not rec or rec.get("src_hash") != kernel_source_hash(rec["sources"]):
            return None
        if rec.get("plan") != {k: int(plan[k]) for k in TRAFFIC_PLAN_KEYS}:
            return None
    except (OSError, ValueError, KeyError):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            # the raw samples (the JSON line carries their summary)
            out_dir = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
            self.path = os.path.join(out_dir, "clocks_%d_%d.csv" % (os.getpid(), self.gpu))
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clocks not sampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# --------------------------------------------------------------- CPU oracle --
def oracle_sample(p, rows, cols, threads):
    """Times the oracle on rows x cols of the product (full K).  Returns
    (seconds, flops)."""
    import numpy as np

    import oracle
    Bs = p.B
    if cols is not None:
        Bs = np.ascontiguousarray(p.B[cols, :] if p.b_major == 1 else p.B[:, cols])
    bias = p.bias[cols] if (p.bias is not None and cols is not None) else p.bias
    t0 = time.perf_counter()
    oracle.gemm_rows(p.A, Bs, bias, a_major=p.a_major, b_major=p.b_major, rows=rows,
                     threads=threads)
    dt = time.perf_counter() - t0
    ncols = len(cols) if cols is not None else p.N
    return dt, flops_of(len(rows), ncols, p.K)


def cpu_baseline(p, seconds, threads):
    """The oracle as it stands on a bounded sample of the workload: `threads`
    rows at a time, all N columns, grown until about `seconds` of work."""
    import numpy as np
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(p.M, size=min(p.M, threads), replace=False)).astype(np.int64)
    dt, fl = oracle_sample(p, rows, None, threads)
    reps = 1
    total_t, total_f = dt, fl
    while total_t < seconds and reps < 64:
        rows = np.sort(rng.choice(p.M, size=min(p.M, threads), replace=False)).astype(np.int64)
        dt, fl = oracle_sample(p, rows, None, threads)
        total_t += dt
        total_f += fl
        reps += 1
    return {"value": total_f / total_t / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": "%d calls x %d rows of the %dx%dx%d product (all %d columns, full K), "
                      "fp64 accumulation, %.1f s" % (reps, len(rows), p.M, p.N, p.K, p.N, total_t)}


def host_link(dev, hA, hB, hbias, hC, dev_set, step_flops, per_launch_s, reps=3):
    """The host link the end-to-end steps travel over, measured with the same
    pinned buffers: one step's inputs host -> device, its output device ->
    host, and both directions at once on two streams (CUDA events, best of
    `reps`).  The bound is the step rate the link (or the kernel, if slower)
    allows when one step's copies overlap the previous step's compute, as
    the pipelined end-to-end steps do."""
    import torch
    A, Bd, bias, C = dev_set
    ins = [(A, hA), (Bd, hB)] + ([(bias, hbias)] if hbias is not None else [])
    bytes_in = sum(h.numel() * h.element_size() for _, h in ins)
    bytes_out = hC.numel() * hC.element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(streams_work):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            cur = torch.cuda.current_stream(dev)
            e0.record(cur)
            for st, work in streams_work:
                st.wait_stream(cur)
                with torch.cuda.stream(st):
                    work()
            for st, _ in streams_work:
                cur.wait_stream(st)
            e1.record(cur)
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1) * 1e-3)
        return best

    def copy_in():
        for d, h in ins:
            d.copy_(h, non_blocking=True)

    def copy_out():
        hC.copy_(C, non_blocking=True)

    t_in = timed([(s_in, copy_in)])
    t_out = timed([(s_out, copy_out)])
    t_both = timed([(s_in, copy_in), (s_out, copy_out)])
    step_s = max(t_both, per_launch_s)
    return {"h2d_gbs": bytes_in / t_in / 1e9, "d2h_gbs": bytes_out / t_out / 1e9,
            "both_gbs": (bytes_in + bytes_out) / t_both / 1e9,
            "bound_tflops": step_flops / step_s / 1e12,
            "bound_basis": "one step's copies in both directions at once, overlapping the "
                           "previous step's kernel (or the kernel, if slower)"}


# --------------------------------------------------------------- cuBLAS arm --
def cublas_step(p, sets):
    """One step of the context arm: cuBLAS (through torch) on one set of the
    same device operands.  fp32 inputs run with TF32 off; a bias is added in
    the output type.  fp16 inputs with an fp32 output are computed with an
    fp16 output instead (its own buffer), which writes half the bytes."""
    import torch
    torch.backends.cuda.matmul.allow_tf32 = False
    copies = len(sets)
    in_t = sets[0][0].dtype
    outs = [C if C.dtype == in_t else torch.empty(C.shape, dtype=in_t, device=C.device)
            for _, _, _, C in sets]
    biases = [None if b is None else b.to(in_t) for _, _, b, _ in sets]

    def step(i, s):
        A, Bd, _, _ = sets[i % copies]
        Aop = A if p.a_major == 0 else A.t()
        Bop = Bd if p.b_major == 0 else Bd.t()
        with torch.cuda.stream(s):
            if biases[i % copies] is not None:
                torch.addmm(biases[i % copies], Aop, Bop, out=outs[i % copies])
            else:
                torch.mm(Aop, Bop, out=outs[i % copies])
    return step


# ------------------------------------------------------------ reference arm --
def run_reference(args):
    import numpy as np

    import oracle
    from dense_gemm_tmem_gb300 import inputs
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = inputs.workload(args.workload)
    p = w.make()
    threads = oracle.host_threads()
    rng = np.random.default_rng(11)
    budget = 100.0  # seconds for the whole --steps/--warmup run
    per_step = budget / max(1, args.steps + args.warmup)
    rows = np.sort(rng.choice(p.M, size=min(p.M, threads), replace=False)).astype(np.int64)
    # calibrate: cost per column of a `threads`-row sample
    cols = np.arange(min(p.N, 64), dtype=np.int64)
    dt, _ = oracle_sample(p, rows, cols, threads)
    per_col = dt / len(cols)
    ncols = int(max(8, min(p.N, per_step / max(per_col, 1e-9))))
    ncols -= ncols % 8 if ncols > 8 else 0
    cols = np.sort(rng.choice(p.N, size=ncols, replace=False)).astype(np.int64)
    for _ in range(args.warmup):
        oracle_sample(p, rows, cols, threads)
    times, fl = [], 0.0
    for _ in range(args.steps):
        dt, f = oracle_sample(p, rows, cols, threads)
        times.append(dt)
        fl += f
    total = sum(times)
    value = fl / total / 1e12
    sample = ("%d rows x %d columns of the %dx%dx%d product per step (full K), fp64 "
              "accumulation" % (len(rows), ncols, p.M, p.N, p.K))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "M": p.M, "N": p.N, "K": p.K,
                   "description": w.description},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm --
def run_ours(args):
    import numpy as np
    import torch

    from dense_gemm_tmem_gb300 import binding as B
    from dense_gemm_tmem_gb300 import inputs
    from dense_gemm_tmem_gb300.gemm import Gemm

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = inputs.workload(args.workload)
    p = w.make()
    cublas = args.impl == "cublas"
    g = None if cublas else Gemm(dev)
    opts = {}
    for kv in ([] if cublas else args.opt):
        name, _, value = kv.partition("=")
        opts[name.upper()] = int(value)
        g.set_option(getattr(B, "GEMM_OPT_" + name.upper()), int(value))
    tdt = {inputs.F16: torch.float16, inputs.F32: torch.float32}
    in_t, out_t = tdt[p.in_dtype], tdt[p.out_dtype]
    esz_in = 2 if p.in_dtype == inputs.F16 else 4
    esz_out = 2 if p.out_dtype == inputs.F16 else 4
    bytes_a = p.A.size * esz_in
    bytes_b = p.B.size * esz_in
    bytes_c = p.M * p.N * esz_out
    bytes_bias = 0 if p.bias is None else p.bias.size * 4
    step_bytes = bytes_a + bytes_b + bytes_c + bytes_bias
    # inputs smaller than 3x L2: rotate through enough copies that each step
    # reads operands no earlier step left in L2
    copies = 1 if step_bytes > 3 * L2_BYTES else int(np.ceil(3 * L2_BYTES / step_bytes))
    hA = torch.from_numpy(p.A).pin_memory()
    hB = torch.from_numpy(p.B).pin_memory()
    hbias = torch.from_numpy(p.bias).pin_memory() if p.bias is not None else None
    sets = []
    for _ in range(copies):
        A = hA.to(dev, non_blocking=True)
        Bd = hB.to(dev, non_blocking=True)
        bias = hbias.to(dev, non_blocking=True) if hbias is not None else None
        C = torch.empty((p.M, p.N), dtype=out_t, device=dev)
        sets.append((A, Bd, bias, C))
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    if cublas:
        plan = None
        launches_per_step = 0  # none of this library's kernels
        step = cublas_step(p, sets)
    else:
        plan = g.plan(p.M, p.N, p.K, p.a_major, p.b_major,
                      B.GEMM_F16 if p.in_dtype == inputs.F16 else B.GEMM_F32,
                      B.GEMM_F16 if p.out_dtype == inputs.F16 else B.GEMM_F32)
        launches_per_step = 0 if plan["kernel"] == B.GEMM_KERNEL_NONE else 1

        def step(i, s):
            A, Bd, bias, C = sets[i % copies]
            g.run(A, Bd, C, bias, p.a_major, p.b_major, stream=s)

    def check():
        if g is not None:
            g.status(stream)

    for i in range(args.warmup):
        step(i, stream)
    check()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # The K timed steps are recorded once as a CUDA graph and replayed on the
    # launching stream: every step's kernel runs in full, without the host's
    # per-call launch latency between them (which would dominate microsecond
    # kernels).  --eager launches them one by one instead.
    graph = None
    if not args.eager:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap, capture_error_mode="relaxed"):
            for i in range(args.steps):
                step(i, cap)
        torch.cuda.synchronize(dev)
        graph.replay()  # one untimed replay
        torch.cuda.synchronize(dev)
        check()

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)  # first sample lands before the region
    barrier()
    ev[0].record(stream)
    if graph is not None:
        graph.replay()
        ev[args.steps].record(stream)
    else:
        for i in range(args.steps):
            step(i, stream)
            ev[i + 1].record(stream)
    barrier()
    clocks = sampler.stop()
    check()
    elapsed_ms = ev[0].elapsed_time(ev[args.steps])
    if graph is not None:
        per_launch_ms = [elapsed_ms / args.steps]  # back-to-back launches inside the replay
    else:
        per_launch_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    elapsed_ms = slowest_rank_ms(elapsed_ms, dev, dist)
    step_flops = flops_of(p.M, p.N, p.K)
    value = whole_job_tflops(world, args.steps, step_flops, elapsed_ms)

    # roofline of the one kernel per step
    avg_launch_s = statistics.mean(per_launch_ms) * 1e-3
    peaks, peak_src = load_peaks()
    region_s = elapsed_ms * 1e-3
    if p.in_dtype == inputs.F16:
        # The sustained peak was taken as a long loop under the power cap: it
        # is the denominator for a region of a second or more, or for one whose
        # clock samples show the power cap holding the SM clock down.
        ck = clocks or {}
        capped = ("sw_power_cap" in (ck.get("reasons") or []) and ck.get("sm_mhz") and
                  ck.get("sm_max_mhz") and ck["sm_mhz"] < 0.95 * ck["sm_max_mhz"])
        sustained = region_s >= 1.0 or bool(capped)
        peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        ridge = peak * 1e12 / (peaks["hbm_gbs"] * 1e9)  # flop per byte
        intensity = step_flops / step_bytes
        if intensity >= ridge:
            roof = {"bound": "tensor", "achieved": step_flops / avg_launch_s / 1e12,
                    "peak": peak, "unit": "TFLOP/s",
                    "peak_source": "%s dense bf16 %s (fp16 dense rate is the same)"
                                   % (peak_src, "sustained" if sustained else "burst")}
        else:
            # below the ridge: the operands' bytes bound the kernel
            roof = {"bound": "hbm", "achieved": step_bytes / avg_launch_s / 1e9,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "peak_source": "%s copy bandwidth" % peak_src,
                    "tflops": step_flops / avg_launch_s / 1e12}
        roof["intensity_flop_per_byte"] = intensity
        roof["ridge_flop_per_byte"] = ridge
    else:
        # fp32 CUDA-core path: SMs x 128 FMA lanes x 2 flop x max SM clock
        props = torch.cuda.get_device_properties(dev)
        peak = props.multi_processor_count * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": step_flops / avg_launch_s / 1e12, "peak": peak,
                "unit": "TFLOP/s", "peak_source": "SMs x 128 FP32 lanes x 2 x max SM clock"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    traffic = None if cublas else recorded_traffic(args.workload, plan)
    roof["traffic"] = traffic
    roof["algorithmic_bytes"] = step_bytes

    # end to end through the C ABI with host buffers: every step is one
    # gemm_run_host call, which copies A, B and bias in from pinned host
    # memory, runs, and copies C back, all on its stream.  Steps alternate
    # between two handles on two streams, so step i+1's inputs travel while
    # step i computes and its result comes back.
    e2e = None
    if not args.no_e2e and not cublas:
        hs = [g, Gemm(dev)]
        for name, value in opts.items():
            hs[1].set_option(getattr(B, "GEMM_OPT_" + name), value)
        ss = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
        hCs = [torch.empty((p.M, p.N), dtype=out_t).pin_memory() for _ in range(2)]

        def e2e_step(i):
            k = i % 2
            hs[k].run_host(hA, hB, hCs[k], hbias, p.a_major, p.b_major, stream=ss[k])

        e_steps = max(3, min(args.steps, 50))
        for i in range(2):
            e2e_step(i)
        for s in ss:
            s.synchronize()
        barrier()
        t0 = time.perf_counter()
        for i in range(e_steps):
            e2e_step(i)
        for s in ss:
            s.synchronize()
        barrier()
        e_ms = slowest_rank_ms((time.perf_counter() - t0) * 1e3, dev, dist)
        for h, s in zip(hs, ss):
            h.status(s)
        for h in hs[1:]:
            h.close()
        e2e = {"value": whole_job_tflops(world, e_steps, step_flops, e_ms),
               "unit": "TFLOP/s", "h2d_bytes_per_step": bytes_a + bytes_b + bytes_bias,
               "d2h_bytes_per_step": bytes_c, "steps": e_steps,
               "api": "gemm_run_host (pinned host buffers)",
               "pipelining": "two handles on two streams, alternating steps",
               "link": host_link(dev, hA, hB, hbias, hCs[0], sets[0], step_flops,
                                 per_launch_s=avg_launch_s)}
        e2e["link"]["frac"] = e2e["value"] / e2e["link"]["bound_tflops"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu and not cublas:
        import oracle
        cpu = cpu_baseline(p, args.cpu_seconds, oracle.host_threads())

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16" if p.in_dtype == inputs.F16
            else "f32", "data": "synthetic",
            "config": {
                "workload": args.workload, "M": p.M, "N": p.N, "K": p.K,
                "a_major": "row" if p.a_major == 0 else "col",
                "b_major": "row" if p.b_major == 0 else "col",
                "out_dtype": p.out_dtype, "bias": p.bias is not None,
                "accumulate": "f32", "description": w.description,
                "parallelism": "replicas x%d" % world,
                "timing": "eager launches" if graph is None
                else "the K steps replayed as one CUDA graph on the launching stream",
                "l2": ("inputs exceed L2 (%d MiB per step)" % (step_bytes >> 20)) if copies == 1
                else "rotating %d input copies (%d MiB) so each step misses L2"
                     % (copies, (copies * step_bytes) >> 20),
                **({"plan": {k: plan[k] for k in ("kernel", "swap_ab", "tile_m", "tile_n",
                                                  "tile_k", "stages", "grid", "dp_tiles",
                                                  "sk_tiles")}} if plan else {}),
                **({"options": opts} if opts else {}),
            },
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "roofline": roof,
            "cpu_baseline": cpu,
        }
        if cublas:
            line = {"impl": "cublas", **line,
                    "note": "cuBLAS through torch.mm / torch.addmm on the same operands and "
                            "protocol, for context only (the library never calls it); a bias is "
                            "added in the output type; fp16 inputs with fp32 output are "
                            "computed with fp16 output"}
        print(json.dumps(line), flush=True)
    if g is not None:
        g.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
