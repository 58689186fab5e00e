"""The allocation-free entry point, gemm_run_noalloc, against gemm_run.

Some callers cannot allocate device memory (a plugin living inside an
application whose allocator owns the GPU's memory, or a latency-critical path
that must not synchronise on cudaMalloc/cudaFree).  gemm_run_noalloc serves
them with scratch compiled into the library.  Each case calls it twice in a
row (the second call finds the first call's partial tiles and counters still
in the shared array) and checks both results against the CPU oracle at the
gates every other GPU test uses, and against gemm_run's result within the same
tolerance; where both entry points run the same plan the results must be
bit-identical.

This file is collected last on purpose, and builds everything it needs itself
so it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_tmem_gb300 import binding as B
from dense_gemm_tmem_gb300 import inputs
from dense_gemm_tmem_gb300.gemm import Gemm

from gpu_helpers import TDT, check, sample_rows, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # (M, N, K, a_major, b_major, out, bias)
    (16, 4096, 192, 0, 0, inputs.F32, True),      # Stream-K split: partial tiles and tile
                                                  # counters in the shared array
    (16, 2048, 192, 0, 1, inputs.F16, True),      # the same, column-major B, fp16 output
    (16, 4096, 4096, 0, 0, inputs.F32, False),    # skinny: swapped operands, cluster split
    (512, 512, 512, 0, 0, inputs.F32, False),     # whole 128 x 64 tiles
    (1280, 5120, 1024, 0, 1, inputs.F16, True),   # CTA pairs, whole 256 x 256 tiles
    (296, 520, 200, 1, 0, inputs.F16, True),      # ragged tiles, MN-major A
    (8, 8, 0, 0, 0, inputs.F32, True),            # K = 0: bias only
]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


@pytest.mark.parametrize("case", CASES)
def test_noalloc_matches_gemm_run_twice(dev, case):
    M, N, K, am, bm, odt, with_bias = case
    p = inputs.make_problem("na", M, N, K, am, bm, inputs.F16, odt, "uniform", with_bias, 200 + M)
    A, Bt, bias = to_dev(p, dev)
    g = Gemm(dev)
    ref = g(A, Bt, bias, am, bm, out_dtype=TDT[odt])
    g.status()
    ref_plan = g.plan(M, N, K, am, bm, B.GEMM_F16,
                      B.GEMM_F16 if odt == inputs.F16 else B.GEMM_F32)
    if K == 192:  # these shapes run the split that keeps its partials in the array
        assert ref_plan["kernel"] == B.GEMM_KERNEL_STREAMK and ref_plan["workspace_bytes"] > 0
    lay = B.layout(am, bm, B.GEMM_F16, B.GEMM_F16 if odt == inputs.F16 else B.GEMM_F32)
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = []
    for _ in range(2):
        C = torch.full((M, N), float("nan"), dtype=TDT[odt], device=dev)
        rc = B.gemm_run_noalloc(M, N, K, A.data_ptr(), Bt.data_ptr(),
                                bias.data_ptr() if bias is not None else None, C.data_ptr(),
                                lay, stream.cuda_stream, status.data_ptr())
        assert rc == B.GEMM_OK, B.gemm_strerror(rc)
        outs.append(C)
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0
    # the oracle on every row of the smaller cases, on one row per 128-row
    # tile (plus the edges) of the larger ones
    rows = None if M * N * K <= (1 << 31) else sample_rows(M, 17)
    exact = oracle.gemm_rows(p.A, p.B, p.bias, a_major=am, b_major=bm, rows=rows)
    pick = (lambda X: X) if rows is None else (lambda X: X[rows])
    want = pick(ref.double().cpu().numpy())
    check(want, exact, p, rows)  # gemm_run itself passes the gates here
    same_plan = ref_plan["workspace_bytes"] <= (16 << 20)
    for C in outs:
        got = C.double().cpu().numpy()
        assert not np.isnan(got).any()
        check(pick(got), exact, p, rows)
        # and within the same tolerance of gemm_run's result
        check(pick(got), want, p, rows)
        if same_plan:
            assert torch.equal(C, ref)
    g.close()


def test_noalloc_rejects_what_it_cannot_run(dev):
    lay32 = B.layout(0, 0, B.GEMM_F32, B.GEMM_F32)
    x = torch.zeros((64, 64), dtype=torch.float32, device=dev)
    rc = B.gemm_run_noalloc(64, 64, 64, x.data_ptr(), x.data_ptr(), None, x.data_ptr(), lay32,
                            torch.cuda.current_stream(dev).cuda_stream)
    assert rc == B.GEMM_ERR_UNSUPPORTED
    lay = B.layout(0, 0, B.GEMM_F16, B.GEMM_F32)
    rc = B.gemm_run_noalloc(-1, 64, 64, None, None, None, None, lay, None)
    assert rc == B.GEMM_ERR_INVALID_ARG
