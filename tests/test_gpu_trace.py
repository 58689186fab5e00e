"""Phase tracing of the tensor-core kernels: stamps are ordered within each
CTA, the unit counts match the host's work partition, and tracing does not
change the result."""
import numpy as np
import pytest
import torch

from dense_gemm_tmem_gb300 import binding as B
from dense_gemm_tmem_gb300 import inputs
from dense_gemm_tmem_gb300.gemm import Gemm

from gpu_helpers import TDT, set_opts, to_dev

pytestmark = pytest.mark.gpu

(START, FIRST_LOAD, FIRST_DATA, MMA_DONE, LAST_ACCUM, END, UNITS, CLUSTER_DONE, ENTRY, EXIT,
 PARKED, REDUCED) = range(12)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


@pytest.mark.parametrize("M,N,K,kernel", [
    (16, 4096, 4096, -1),                        # swapped, cluster split
    (1024, 19 * 256, 512, B.GEMM_KERNEL_TC2),     # one wave of CTA pairs
    (600, 1000, 1480, B.GEMM_KERNEL_TC),          # whole tiles, one SM each
])
def test_trace_stamps(dev, M, N, K, kernel):
    g = Gemm(dev)
    if kernel >= 0:
        set_opts(g, kernel=kernel)
    p = inputs.make_problem("tr", M, N, K, 0, 0, inputs.F16, inputs.F32, "uniform", True, 300)
    A, Bt, bias = to_dev(p, dev)
    plain = g(A, Bt, bias)
    pl = g.plan(M, N, K)
    grid = pl["grid"]
    buf = torch.zeros((grid, B.TRACE_SLOTS), dtype=torch.int64, device=dev)
    assert B.gemm_set_trace(g.handle, buf.data_ptr(), grid) == B.GEMM_OK
    traced = g(A, Bt, bias)
    g.status()
    assert B.gemm_set_trace(g.handle, None, 0) == B.GEMM_OK
    assert torch.equal(plain, traced)
    t = buf.cpu().numpy()
    rc, plan = B.gemm_query_plan(g.handle, M, N, K, B.layout(0, 0, B.GEMM_F16, B.GEMM_F32))
    pair = plan.kernel == B.GEMM_KERNEL_TC2
    for cta in range(grid):
        row = t[cta]
        unit_owner = cta // 2 if pair else cta
        n_units = len(B.gemm_work_units(plan, unit_owner))
        assert row[UNITS] == n_units
        if n_units == 0:
            continue
        assert 0 < row[ENTRY] <= row[START] <= row[FIRST_LOAD] <= row[END] <= row[EXIT]
        if plan.kernel == B.GEMM_KERNEL_SPLITC:
            assert row[END] <= row[PARKED] <= row[REDUCED] <= row[CLUSTER_DONE] <= row[EXIT]
        assert row[LAST_ACCUM] <= row[END]
        if not pair or cta % 2 == 0:  # the CTA that issues the MMAs
            assert row[FIRST_LOAD] <= row[FIRST_DATA] <= row[MMA_DONE] <= row[LAST_ACCUM]
        else:
            assert row[FIRST_DATA] == 0 and row[MMA_DONE] == 0
    span_us = (t[:, END].max() - t[:, START].min()) / 1e3
    assert 0 < span_us < 1e5
    g.close()


def test_trace_buffer_too_small_is_skipped(dev):
    g = Gemm(dev)
    buf = torch.zeros((4, B.TRACE_SLOTS), dtype=torch.int64, device=dev)
    assert B.gemm_set_trace(g.handle, buf.data_ptr(), 4) == B.GEMM_OK
    p = inputs.make_problem("tr", 16, 4096, 4096, 0, 0, inputs.F16, inputs.F32, "uniform",
                            False, 301)
    A, Bt, _ = to_dev(p, dev)
    g(A, Bt)
    g.status()
    assert int(buf.abs().sum().item()) == 0  # 152 CTAs do not fit in 4 rows: no stamps
    assert B.gemm_set_trace(g.handle, None, 5) == B.GEMM_ERR_INVALID_ARG
    g.close()


def test_trace_tool_timeline(dev):
    """The timeline tool reads back stamps from every launch of a replayed graph."""
    from dense_gemm_tmem_gb300 import trace_tool
    res = trace_tool.run("tile128_f16_f32out", 6, 0)
    ph = res["mean_phase_us"]
    assert 1 <= res["grid"] <= 8 and res["us_per_launch"] > 0  # a few whole tiles
    for k in ("entry_to_setup_done", "setup_to_first_load", "main_loop", "epilogue",
              "entry_to_exit"):
        assert 0 <= ph[k] < 1000, (k, ph)
    res = trace_tool.run("skinny_m16_4096", 4, 1)
    assert res["kernel"] == B.GEMM_KERNEL_SPLITC and "cluster_reduce" in res["mean_phase_us"]
