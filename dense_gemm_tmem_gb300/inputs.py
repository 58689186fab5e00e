"""Seeded synthetic inputs and the named workloads.

This module only draws numbers and names shapes: it holds none of the
product's arithmetic, and both the CUDA path and the CPU oracle consume what
it returns.  Values are drawn in binary64 with numpy's PCG64 generator (the
same stream on x86 and Arm) and rounded once, to nearest-even, to the storage
type.

Storage conventions: A (M x K) is stored as an (M, K) array when row-major and
as a (K, M) array (Aᵀ row-major) when column-major; B (K x N) is stored as
(K, N) when row-major and (N, K) when column-major.  ``major`` 0 = row-major,
1 = column-major.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

ROW, COL = 0, 1
F16, F32 = "f16", "f32"
_NP = {F16: np.float16, F32: np.float32}
_CHUNK = 1 << 22  # elements drawn per generator call, fixed so streams repeat


def _draw(shape, seed, kind, lo=-1, hi=1):
    rng = np.random.default_rng(seed)
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        if kind == "uniform":
            out[s:e] = rng.uniform(lo, hi, size=e - s)
        elif kind == "normal":
            out[s:e] = rng.standard_normal(size=e - s)
        elif kind == "int":
            out[s:e] = rng.integers(lo, hi + 1, size=e - s)
        else:
            raise ValueError(kind)
    return out.reshape(shape)


def draw(shape, seed, kind="uniform", dtype=F16, lo=-1, hi=1):
    """``shape`` values from ``kind`` ∈ {uniform (U[lo,hi]), normal (N(0,1)),
    int (integers lo..hi)}, rounded once to ``dtype``."""
    x = _draw(tuple(shape), seed, kind, lo, hi)
    return x.astype(_NP[dtype])


def storage_shape_a(M, K, major):
    return (M, K) if major == ROW else (K, M)


def storage_shape_b(K, N, major):
    return (K, N) if major == ROW else (N, K)


@dataclass
class Problem:
    """One GEMM instance in storage form (numpy, host)."""
    name: str
    M: int
    N: int
    K: int
    A: np.ndarray
    B: np.ndarray
    bias: np.ndarray | None
    a_major: int
    b_major: int
    in_dtype: str
    out_dtype: str
    info: dict = field(default_factory=dict)


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    a_major: int
    b_major: int
    in_dtype: str
    out_dtype: str
    dist: str        # "uniform" or "normal"
    bias: bool
    seed_base: int   # A: 1000+seed_base, B: 2000+seed_base, bias: 3000+seed_base
    description: str

    def make(self, kind: str | None = None, M: int | None = None,
             N: int | None = None, K: int | None = None) -> Problem:
        """Draws the inputs.  ``kind`` overrides the distribution (e.g. "int"
        for the exact-integer variant); M/N/K override the shape (same seeds)."""
        M = self.M if M is None else M
        N = self.N if N is None else N
        K = self.K if K is None else K
        return make_problem(self.name, M, N, K, self.a_major, self.b_major,
                            self.in_dtype, self.out_dtype, kind or self.dist,
                            self.bias, self.seed_base)


def int_range(in_dtype):
    """Integer value range of the exact variant: {-1,0,1} for fp16 (so that
    sums at K=8192 stay inside fp16's exact-integer range), {-2..2} for fp32."""
    return (-1, 1) if in_dtype == F16 else (-2, 2)


def make_problem(name, M, N, K, a_major, b_major, in_dtype, out_dtype, kind,
                 with_bias, seed_base) -> Problem:
    if kind == "int":
        lo, hi = int_range(in_dtype)
        blo, bhi = -2, 2
    else:
        lo, hi, blo, bhi = -1, 1, -1, 1
    A = draw(storage_shape_a(M, K, a_major), 1000 + seed_base, kind, in_dtype, lo, hi)
    B = draw(storage_shape_b(K, N, b_major), 2000 + seed_base, kind, in_dtype, lo, hi)
    bias = None
    if with_bias:
        bias = draw((N,), 3000 + seed_base, kind, F32, blo, bhi)
    return Problem(name, M, N, K, A, B, bias, a_major, b_major, in_dtype,
                   out_dtype, {"kind": kind, "seed_base": seed_base})


WORKLOADS = {
    w.name: w for w in [
        Workload("gemm512_f16_f32out", 512, 512, 512, ROW, ROW, F16, F32,
                 "uniform", False, 1,
                 "M=N=K=512, fp16 row-major A and B, U[-1,1], fp32 output"),
        Workload("sgemm2048_f32", 2048, 2048, 2048, ROW, ROW, F32, F32,
                 "uniform", False, 2,
                 "M=N=K=2048 fp32 row-major A and B, U[-1,1], fp32 output (CUDA-core path)"),
        Workload("gemm8192_f16_bias_f16out", 8192, 8192, 8192, ROW, COL, F16, F16,
                 "normal", True, 3,
                 "M=N=K=8192, fp16 row-major A, column-major B, N(0,1), fp32 bias, fp16 output"),
        Workload("skinny_m1_4096", 1, 4096, 4096, ROW, ROW, F16, F32, "uniform",
                 False, 4, "M=1, N=K=4096 fp16 row-major, U[-1,1], fp32 output"),
        Workload("skinny_m16_4096", 16, 4096, 4096, ROW, ROW, F16, F32, "uniform",
                 False, 4, "M=16, N=K=4096 fp16 row-major, U[-1,1], fp32 output"),
        Workload("skinny_m64_4096", 64, 4096, 4096, ROW, ROW, F16, F32, "uniform",
                 False, 4, "M=64, N=K=4096 fp16 row-major, U[-1,1], fp32 output"),
        Workload("skinny_m128_4096", 128, 4096, 4096, ROW, ROW, F16, F32, "uniform",
                 False, 4, "M=128, N=K=4096 fp16 row-major, U[-1,1], fp32 output"),
        Workload("gemm16384_f16_f16out", 16384, 16384, 16384, ROW, ROW, F16, F16,
                 "uniform", False, 5,
                 "M=N=K=16384 fp16 row-major A and B, U[-1,1], fp16 output"),
        Workload("tile128_f16_f32out", 128, 128, 64, ROW, COL, F16, F32, "uniform", False, 6,
                 "a 128 x 128 output with K=64 (one k-block): the fixed cost of a launch"),
    ]
}


def shape_workload(spec: str) -> Workload:
    """A workload named by its shape: ``MxNxK[:AB[:IO[:bias]]]`` with A and B
    each ``r`` (row-major) or ``c`` (column-major), I and O each ``h`` (fp16)
    or ``f`` (fp32); the defaults are ``rc`` and ``hh``.  Inputs are U[-1,1]
    (bias included) from the seeds of base 7.  ``4096x4096x1024:rc:hf`` is
    row-major A, column-major B, fp16 in, fp32 out, no bias."""
    parts = spec.split(":")
    try:
        M, N, K = (int(x) for x in parts[0].lower().split("x"))
    except ValueError:
        raise ValueError("workload %r: neither a named workload nor MxNxK" % spec) from None
    lay = parts[1] if len(parts) > 1 else "rc"
    io = parts[2] if len(parts) > 2 else "hh"
    bias = len(parts) > 3 and parts[3] == "bias"
    if (len(lay) != 2 or any(c not in "rc" for c in lay) or len(io) != 2
            or any(c not in "hf" for c in io) or len(parts) > 4
            or (len(parts) == 4 and not bias) or min(M, N, K) < 0):
        raise ValueError("shape %r: want MxNxK[:AB[:IO[:bias]]], A/B in r|c, I/O in h|f"
                         % spec)
    maj = {"r": ROW, "c": COL}
    dt = {"h": F16, "f": F32}
    name = "shape_%dx%dx%d_%s_%s%s" % (M, N, K, lay, io, "_bias" if bias else "")
    desc = "M=%d N=%d K=%d, %s A, %s B, %s in, %s out%s, U[-1,1]" % (
        M, N, K, "row-major" if lay[0] == "r" else "column-major",
        "row-major" if lay[1] == "r" else "column-major", dt[io[0]], dt[io[1]],
        ", fp32 bias" if bias else "")
    return Workload(name, M, N, K, maj[lay[0]], maj[lay[1]], dt[io[0]], dt[io[1]],
                    "uniform", bias, 7, desc)


def workload(name: str) -> Workload:
    """A named workload of ``WORKLOADS``, or a shape spec (``shape_workload``)."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    return shape_workload(name)
