"""Shared pieces of the GPU tests: running a Problem through the C-ABI and
the acceptance gates."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dense_gemm_tmem_gb300 import binding as B
from dense_gemm_tmem_gb300 import inputs

TDT = {inputs.F16: torch.float16, inputs.F32: torch.float32}


def to_dev(p: inputs.Problem, dev):
    A = torch.from_numpy(p.A).to(dev)
    Bt = torch.from_numpy(p.B).to(dev)
    bias = torch.from_numpy(p.bias).to(dev) if p.bias is not None else None
    return A, Bt, bias


def run(g, p: inputs.Problem, dev, *, check_status=True):
    """Runs p through the library; returns C on the device."""
    A, Bt, bias = to_dev(p, dev)
    C = g(A, Bt, bias, p.a_major, p.b_major, out_dtype=TDT[p.out_dtype])
    if check_status:
        g.status()
    return C


def as_f64(C: torch.Tensor, rows=None) -> np.ndarray:
    if rows is not None:
        C = C[torch.as_tensor(np.asarray(rows), device=C.device)]
    return C.double().cpu().numpy()


def abs_scale(p: inputs.Problem, rows=None) -> np.ndarray:
    """sum_k |A[i,k] B[k,j]| (+|bias_j|), the natural scale of each element's
    rounding error, from the oracle on |A|, |B|."""
    bias = np.abs(p.bias) if p.bias is not None else None
    return oracle.gemm_rows(np.abs(p.A), np.abs(p.B), bias, a_major=p.a_major,
                            b_major=p.b_major, rows=rows)


def f16_gate(p: inputs.Problem) -> float:
    """max-abs-error gate for fp16 inputs with fp32 accumulation:
    1e-2 * sqrt(K) * max|a| * max|b|."""
    amax = float(np.abs(p.A).max()) if p.A.size else 0.0
    bmax = float(np.abs(p.B).max()) if p.B.size else 0.0
    return 1e-2 * np.sqrt(max(p.K, 1)) * amax * bmax


def check_f16_path(got: np.ndarray, ref: np.ndarray, p: inputs.Problem, rows=None):
    """The gate, plus the element-wise relative bound the arithmetic allows:
    |Δ| <= 1e-3 * sum|a b| (+ half an fp16 ulp of the result for fp16 output)."""
    err = np.abs(got - ref)
    gate = f16_gate(p)
    assert err.max(initial=0.0) <= gate, (err.max(), gate)
    scale = abs_scale(p, rows)
    slack = 1e-3 * scale
    if p.out_dtype == inputs.F16:
        slack = slack + np.abs(ref) * 2.0 ** -11
    bad = err > slack + 1e-30
    assert not bad.any(), ("element-wise bound", int(bad.sum()), float(err[bad].max()))
    return float(err.max(initial=0.0)), gate


def check_f32_path(got: np.ndarray, ref: np.ndarray):
    """fp32 path: relative error <= 1e-5, read as both the Frobenius ratio and
    max|Δ| / max|C|."""
    d = got - ref
    nref = np.linalg.norm(ref)
    if nref == 0:
        assert np.abs(d).max(initial=0.0) == 0
        return 0.0
    fro = np.linalg.norm(d) / nref
    mx = np.abs(d).max() / np.abs(ref).max()
    assert fro <= 1e-5 and mx <= 1e-5, (fro, mx)
    return max(fro, mx)


def check(got, ref, p, rows=None):
    if p.in_dtype == inputs.F16:
        return check_f16_path(got, ref, p, rows)
    return check_f32_path(got, ref)


def sample_rows(M: int, seed: int, tile: int = 128):
    """One seeded row per 128-row tile, plus rows 0, M-1 and the last row of
    the first tile: every tile row, TMEM lane quarter and column is covered."""
    rng = np.random.default_rng(seed)
    rows = {0, M - 1, min(M - 1, tile - 1)}
    for t0 in range(0, M, tile):
        rows.add(int(rng.integers(t0, min(M, t0 + tile))))
    return np.array(sorted(rows), dtype=np.int64)


def set_opts(g, **kw):
    names = {"kernel": B.GEMM_OPT_FORCE_KERNEL, "tile_n": B.GEMM_OPT_FORCE_TILE_N,
             "grid": B.GEMM_OPT_FORCE_GRID, "swap": B.GEMM_OPT_FORCE_SWAP_AB,
             "min_split": B.GEMM_OPT_MIN_SPLIT_ITERS, "group_m": B.GEMM_OPT_GROUP_M,
             "pair": B.GEMM_OPT_PAIR, "csplit": B.GEMM_OPT_CLUSTER_SPLIT,
             "pair_split": B.GEMM_OPT_PAIR_SPLIT, "tma_store": B.GEMM_OPT_TMA_STORE,
             "bias_init": B.GEMM_OPT_BIAS_INIT, "dyn": B.GEMM_OPT_DYNAMIC_TILES,
             "stages": B.GEMM_OPT_STAGES, "tile_m": B.GEMM_OPT_TILE_M,
             "k_group": B.GEMM_OPT_K_GROUP}
    for k, v in kw.items():
        g.set_option(names[k], v)


def reset_opts(g):
    for opt in (B.GEMM_OPT_FORCE_KERNEL, B.GEMM_OPT_FORCE_TILE_N, B.GEMM_OPT_FORCE_GRID,
                B.GEMM_OPT_FORCE_SWAP_AB, B.GEMM_OPT_MIN_SPLIT_ITERS, B.GEMM_OPT_GROUP_M,
                B.GEMM_OPT_PAIR, B.GEMM_OPT_CLUSTER_SPLIT, B.GEMM_OPT_PAIR_SPLIT,
                B.GEMM_OPT_TMA_STORE, B.GEMM_OPT_BIAS_INIT, B.GEMM_OPT_DYNAMIC_TILES,
                B.GEMM_OPT_STAGES, B.GEMM_OPT_TILE_M, B.GEMM_OPT_K_GROUP):
        g.set_option(opt, -1)
