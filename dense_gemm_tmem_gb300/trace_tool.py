"""Phase timeline of back-to-back launches, from the kernels' own trace stamps.

    python -m dense_gemm_tmem_gb300.trace_tool --workload skinny_m16_4096

Records `--launches` launches of one workload as a CUDA graph, each launch
writing its own rows of %globaltimer stamps (gemm_set_trace), replays the
graph once, and prints the median time of each phase over the launches:
the gap between one launch's last CTA exit and the next one's first CTA
entry, setup, the first TMA load, the main loop, the epilogue and, for the
cluster split, the on-chip reduction.  The stamps have the timer's
granularity (about a quarter of a microsecond on GB300).
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import binding as B
from . import inputs
from .gemm import Gemm

# per-CTA trace slots (include/gemm.h, gemm_set_trace)
START, FIRST_LOAD, FIRST_DATA, MMA_DONE, LAST_ACCUM, END = range(6)
CLUSTER_DONE, ENTRY, EXIT = B.TRACE_CLUSTER_DONE, B.TRACE_ENTRY, B.TRACE_EXIT
PARKED, REDUCED = B.TRACE_CLUSTER_PARKED, B.TRACE_CLUSTER_REDUCED


def _stat(t, i, k, how):
    v = t[i, :, k]
    v = v[v > 0]
    return how(v) if len(v) else np.nan


def phases(t: np.ndarray) -> dict:
    """Mean over launches 1.. of each phase in microseconds; t holds
    (launches, ctas, slots) nanosecond stamps.  A phase's ends are averaged
    over the CTAs (and the launches), which resolves phases shorter than the
    timer's tick: the stamps fall at every offset from the ticks."""
    rows = []
    for i in range(1, t.shape[0]):
        med = lambda k: _stat(t, i, k, np.mean)  # noqa: E731
        first_entry = _stat(t, i, ENTRY, np.min)
        rows.append({
            "gap_after_previous_launch": first_entry - _stat(t, i - 1, EXIT, np.max),
            "entry_to_setup_done": med(START) - med(ENTRY),
            "setup_to_first_load": med(FIRST_LOAD) - med(START),
            "first_load_to_first_data": med(FIRST_DATA) - med(FIRST_LOAD),
            "main_loop": med(MMA_DONE) - med(FIRST_DATA),
            "epilogue": _stat(t, i, END, np.max) - med(MMA_DONE),
            "cluster_park_wait": med(PARKED) - med(END),
            "cluster_reduce": med(REDUCED) - med(PARKED),
            "cluster_finish": med(CLUSTER_DONE) - med(REDUCED),
            "end_to_exit": _stat(t, i, EXIT, np.max) - _stat(t, i, END, np.max),
            "entry_to_exit": _stat(t, i, EXIT, np.max) - first_entry,
        })
    out = {}
    for k in rows[0]:
        vals = [r[k] for r in rows if not np.isnan(r[k])]
        if vals:
            out[k] = round(float(np.mean(vals)) / 1e3, 3)
    return out


def run(workload: str, launches: int, pdl: int, device: int = 0, opts=None) -> dict:
    dev = torch.device("cuda", device)
    g = Gemm(dev)
    for name, value in (opts or {}).items():
        g.set_option(getattr(B, "GEMM_OPT_" + name.upper()), int(value))
    w = inputs.workload(workload)
    p = w.make()
    A = torch.from_numpy(p.A).to(dev)
    Bm = torch.from_numpy(p.B).to(dev)
    bias = torch.from_numpy(p.bias).to(dev) if p.bias is not None else None
    odt = torch.float16 if p.out_dtype == inputs.F16 else torch.float32
    C = torch.empty((p.M, p.N), dtype=odt, device=dev)
    g.set_option(B.GEMM_OPT_PDL, pdl)
    plan = g.plan(p.M, p.N, p.K, p.a_major, p.b_major,
                  B.GEMM_F16 if p.in_dtype == inputs.F16 else B.GEMM_F32,
                  B.GEMM_F16 if p.out_dtype == inputs.F16 else B.GEMM_F32)
    grid = plan["grid"]
    bufs = torch.zeros((launches, grid, B.TRACE_SLOTS), dtype=torch.int64, device=dev)
    for _ in range(3):
        g.run(A, Bm, C, bias, p.a_major, p.b_major)
    torch.cuda.synchronize(dev)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap, capture_error_mode="relaxed"):
        for i in range(launches):
            B.gemm_set_trace(g.handle, bufs[i].data_ptr(), grid)
            g.run(A, Bm, C, bias, p.a_major, p.b_major, stream=cap)
    B.gemm_set_trace(g.handle, None, 0)
    graph.replay()
    torch.cuda.synchronize(dev)
    bufs.zero_()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    g.status()
    t = bufs.cpu().numpy().astype(np.float64)
    res = {"workload": workload, "pdl": pdl, "grid": grid, "kernel": plan["kernel"],
           "tile": [plan["tile_m"], plan["tile_n"]], "cluster_split": plan["cluster_split"],
           "us_per_launch": round(e0.elapsed_time(e1) * 1e3 / launches, 2),
           "mean_phase_us": phases(t)}
    g.close()
    return res


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="skinny_m16_4096",
                    help="a named workload (dense_gemm_tmem_gb300/inputs.py) or a shape "
                         "MxNxK[:AB[:IO[:bias]]]")
    ap.add_argument("--launches", type=int, default=20)
    ap.add_argument("--pdl", type=int, default=0, choices=[0, 1],
                    help="programmatic dependent launch (1 overlaps each launch's setup with "
                         "the previous launch, which makes the phases harder to read)")
    ap.add_argument("--opt", action="append", default=[], metavar="NAME=VALUE",
                    help="set a library option (a GEMM_OPT_ name of include/gemm.h); repeatable")
    a = ap.parse_args()
    opts = dict(kv.split("=", 1) for kv in a.opt)
    res = run(a.workload, a.launches, a.pdl, opts=opts)
    if opts:
        res["options"] = opts
    print(json.dumps(res))


if __name__ == "__main__":
    main()
