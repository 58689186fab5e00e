"""Checks the tile picker against forced alternatives on fp16 shapes.

    python -m dense_gemm_tmem_gb300.picker_check
    python -m dense_gemm_tmem_gb300.picker_check --shape 4096x4096x4096 --shape 1024x2048x4096
    python -m dense_gemm_tmem_gb300.picker_check --splits --shape 512x512x1024

For each M x N x K (row-major A, column-major B, fp16 output, no bias) it
times the picker's plan and the same product forced onto the two-SM kernel,
the one-SM kernel with whole tiles, and the one-SM Stream-K split (with
--splits: instead, cluster splits of 2, 4 and 8 CTAs over 64- and 128-wide
tiles), each as a replayed CUDA graph of back-to-back launches with inputs
rotated through enough copies to miss L2, and prints TFLOP/s and µs per
launch with each plan's kernel, tile width and grid.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import binding as B
from .gemm import Gemm

DEFAULT_SHAPES = ["2048x2048x2048", "4096x4096x4096", "1024x2048x4096", "1536x1536x4096",
                  "1024x1024x8192", "2048x1024x2048", "1280x5120x1024", "768x4096x4096",
                  "1536x2048x2048", "512x4096x8192"]
VARIANTS = [("picker", {}),
            ("two_sm", {B.GEMM_OPT_FORCE_KERNEL: B.GEMM_KERNEL_TC2}),
            ("one_sm_whole", {B.GEMM_OPT_FORCE_KERNEL: B.GEMM_KERNEL_TC}),
            ("one_sm_streamk", {B.GEMM_OPT_FORCE_KERNEL: B.GEMM_KERNEL_STREAMK})]
SPLIT_VARIANTS = [("picker", {})] + [
    ("csplit%d_w%d" % (cs, w), {B.GEMM_OPT_FORCE_KERNEL: B.GEMM_KERNEL_SPLITC,
                                B.GEMM_OPT_FORCE_TILE_N: w, B.GEMM_OPT_CLUSTER_SPLIT: cs})
    for w in (64, 128) for cs in (2, 4, 8)]
L2_BYTES = 129 * 10**6


def _graph_us(dev, fn, launches):
    for i in range(3):
        fn(i, torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap, capture_error_mode="relaxed"):
        for i in range(launches):
            fn(i, cap)
    graph.replay()
    torch.cuda.synchronize(dev)
    best = float("inf")
    for _ in range(2):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1) * 1e3 / launches)
    return best


def check(shape: str, g: Gemm, variants=VARIANTS) -> dict:
    M, N, K = (int(x) for x in shape.lower().split("x"))
    dev = g.device
    copies = max(1, int(np.ceil(3 * L2_BYTES / ((M * K + K * N + M * N) * 2))))
    sets = [(torch.empty((M, K), dtype=torch.float16, device=dev).uniform_(-1, 1),
             torch.empty((N, K), dtype=torch.float16, device=dev).uniform_(-1, 1),
             torch.empty((M, N), dtype=torch.float16, device=dev)) for _ in range(copies)]
    flops = 2.0 * M * N * K
    launches = max(10, min(200, int(2e5 / max(1.0, flops / 1.5e12 * 1e6))))
    out = {}
    for name, opts in variants:
        for o, v in opts.items():
            g.set_option(o, v)
        try:
            plan = g.plan(M, N, K, 0, 1, B.GEMM_F16, B.GEMM_F16)

            def fn(i, s):
                A, Bm, C = sets[i % copies]
                g.run(A, Bm, C, None, 0, 1, stream=s)
            us = _graph_us(dev, fn, launches)
            out[name] = {"tflops": round(flops / us / 1e6, 1), "us": round(us, 2),
                         "kernel": plan["kernel"], "tile_n": plan["tile_n"], "grid": plan["grid"]}
        except B.GemmError as e:
            out[name] = {"unsupported": str(e)}
        finally:
            for o in opts:
                g.set_option(o, -1)
    g.status()
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--shape", action="append", help="MxNxK (repeatable)")
    ap.add_argument("--splits", action="store_true", help="cluster-split variants instead")
    args = ap.parse_args()
    g = Gemm(torch.device("cuda", 0))
    for shape in args.shape or DEFAULT_SHAPES:
        print(shape, json.dumps(check(shape, g, SPLIT_VARIANTS if args.splits else VARIANTS)),
              flush=True)
        torch.cuda.empty_cache()
    g.close()


if __name__ == "__main__":
    main()
