"""Times this library against cuBLAS on the large fp16 GEMMs, for context.

    python -m dense_gemm_tmem_gb300.cublas_compare              # both shapes, short and long runs
    python -m dense_gemm_tmem_gb300.cublas_compare --only ours --launches 4    # a few plain launches (for ncu)
    python -m dense_gemm_tmem_gb300.cublas_compare --only cublas --launches 4

A measurement tool only: the library never calls cuBLAS.  The comparison
side is `torch.addmm` / `torch.mm` (cuBLAS) on the same fp16 operands (an
fp16 bias there, since cuBLAS adds the bias in the output type).  Shapes:
8192^3 with A row-major, B column-major, bias, fp16 output; 16384^3 row/row,
fp16 output.  Both sides are replayed as CUDA graphs over input copies that
together exceed L2, interleaved, with a pause between runs so that each
starts from the same clock; "short" is about 30 ms of launches, "long" about
300 ms (power-capped).  Prints TFLOP/s per side and run length.
"""
from __future__ import annotations

import argparse
import json
import time

import torch

from .gemm import Gemm

L2_BYTES = 129 * 10**6
SHAPES = [(8192, True, True), (16384, False, False)]  # (n, B column-major, bias)
LAYOUT_SHAPES = [(8192, True, False), (8192, False, False), (16384, True, False)]


def _operands(n, bcol, copies, dev):
    return [(torch.empty((n, n), dtype=torch.float16, device=dev).normal_(),
             torch.empty((n, n), dtype=torch.float16, device=dev).normal_(),  # (N,K) if bcol
             torch.empty((n, n), dtype=torch.float16, device=dev)) for _ in range(copies)]


def _launchers(g, sets, bcol, bias32, bias16):
    copies = len(sets)

    def ours(i, s):
        A, Bs, C = sets[i % copies]
        g.run(A, Bs, C, bias32, 0, 1 if bcol else 0, stream=s)

    def cublas(i, s):
        A, Bs, C = sets[i % copies]
        with torch.cuda.stream(s):
            Bm = Bs.t() if bcol else Bs
            if bias16 is not None:
                torch.addmm(bias16, A, Bm, out=C)
            else:
                torch.mm(A, Bm, out=C)
    return {"ours": ours, "cublas": cublas}


def _graph(fn, launches, dev):
    for i in range(3):
        fn(i, torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(torch.cuda.current_stream(dev))
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=cap, capture_error_mode="relaxed"):
        for i in range(launches):
            fn(i, cap)
    gr.replay()
    torch.cuda.synchronize(dev)
    return gr


def compare(dev, shapes=SHAPES) -> None:
    g = Gemm(dev)
    for n, bcol, bias in shapes:
        copies = max(2, -(-3 * L2_BYTES // (3 * n * n * 2)))
        sets = _operands(n, bcol, copies, dev)
        b32 = torch.randn(n, device=dev) if bias else None
        fns = _launchers(g, sets, bcol, b32, b32.half() if bias else None)
        flops = 2.0 * n ** 3
        per_ms = flops / 1.6e15 * 1e3
        runs = {"short": max(5, int(30 / per_ms)), "long": max(20, int(300 / per_ms))}
        graphs = {(w, r): _graph(fns[w], k, dev) for w in fns for r, k in runs.items()}
        res = {}
        for _ in range(2):
            for w in fns:
                for r, k in runs.items():
                    time.sleep(1.0)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                    graphs[(w, r)].replay()
                    e1.record()
                    torch.cuda.synchronize(dev)
                    us = e0.elapsed_time(e1) * 1e3 / k
                    res.setdefault("%s_%s" % (w, r), []).append(round(flops / us / 1e6, 1))
        g.status()
        print("%d^3 B %s%s" % (n, "col" if bcol else "row", " +bias" if bias else ""), json.dumps(res),
              "launches: %s" % json.dumps(runs), flush=True)
        del sets, graphs
        torch.cuda.empty_cache()
    g.close()


def plain(dev, which: str, launches: int, n: int) -> None:
    """A few plain launches of one side on the 8192^3-style operands (for ncu)."""
    g = Gemm(dev)
    sets = _operands(n, True, 1, dev)
    b32 = torch.randn(n, device=dev)
    fn = _launchers(g, sets, True, b32, b32.half())[which]
    for i in range(launches):
        fn(i, torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    g.status()
    g.close()
    print("ok", which, launches)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--only", choices=["ours", "cublas"])
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--n", type=int, default=8192)
    ap.add_argument("--layouts", action="store_true",
                    help="B row- vs column-major without bias (8192^3, and 16384^3 column-major)")
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    if a.only:
        plain(dev, a.only, a.launches, a.n)
    else:
        compare(dev, LAYOUT_SHAPES if a.layouts else SHAPES)


if __name__ == "__main__":
    main()
