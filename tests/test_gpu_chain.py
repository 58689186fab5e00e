"""Back-to-back launches that depend on each other.

The tensor-core kernels are launched with programmatic dependent launch: a
kernel's prologue may overlap the previous kernel on the stream, and it
touches global memory only after that kernel has completed.  A chain where
each product is the next product's operand (and, with the split paths, where
consecutive launches share the handle's workspace and counters) must give the
same numbers as the oracle, launched eagerly or replayed as a CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_tmem_gb300 import binding as B
from dense_gemm_tmem_gb300 import inputs
from dense_gemm_tmem_gb300.gemm import Gemm

from gpu_helpers import set_opts

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def chain_reference(A0, mats):
    """fp16 chain on the oracle: X_{i+1} = fp16(X_i · W_i), exact for these data."""
    X = A0
    for W in mats:
        Y = oracle.gemm(X, W)
        assert np.abs(Y).max() <= 2048  # integers below 2^11 are exact in fp16
        X = Y.astype(np.float16)
    return X.astype(np.float64)


@pytest.mark.parametrize("opts,M", [({}, 384), ({"kernel": B.GEMM_KERNEL_STREAMK}, 384),
                                    ({"kernel": B.GEMM_KERNEL_SPLITC, "csplit": 4}, 384),
                                    ({"kernel": B.GEMM_KERNEL_TC2}, 384),
                                    ({"tile_m": 64}, 384),   # 64-row tiles
                                    ({}, 16)])               # swapped skinny cluster split
@pytest.mark.parametrize("graph", [False, True])
def test_dependent_chain(dev, opts, M, graph):
    g = Gemm(dev)
    set_opts(g, **opts)
    N, steps = 512, 6
    A0 = inputs.draw((M, N), 400, "int", inputs.F16, -1, 1)
    # sparse {-1,0,1} weights keep every intermediate a small integer
    rng = np.random.default_rng(401)
    mats = []
    for i in range(steps):
        W = np.zeros((N, N), np.float16)
        idx = rng.integers(0, N, size=(N, 2))
        W[idx[:, 0], np.arange(N)] = 1
        W[idx[:, 1], np.arange(N)] += rng.choice([-1, 1], size=N).astype(np.float16)
        mats.append(W)
    ref = chain_reference(A0, mats)
    X = [torch.from_numpy(A0).to(dev)] + [torch.empty((M, N), dtype=torch.float16, device=dev)
                                          for _ in range(steps)]
    Ws = [torch.from_numpy(W).to(dev) for W in mats]
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))

    def launch_all():
        for i in range(steps):
            g.run(X[i], Ws[i], X[i + 1], stream=s)

    if graph:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s, capture_error_mode="relaxed"):
            launch_all()
        for t in X[1:]:
            t.zero_()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(s):
            gr.replay()
    else:
        with torch.cuda.stream(s):
            launch_all()
    g.status(s)
    got = X[-1].double().cpu().numpy()
    assert np.array_equal(got, ref)
    g.close()
