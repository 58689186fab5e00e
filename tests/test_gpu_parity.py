"""GPU parity: every kernel family against the CPU oracle, element by element,
on seeded inputs that span several tiles with ragged tails; closed-form inputs
(permutations, integers) that must come out exact; edge cases; determinism;
and the full-size workloads on sampled rows."""
import numpy as np
import pytest
import torch

import golden_values
import oracle
from dense_gemm_tmem_gb300 import binding as B
from dense_gemm_tmem_gb300 import inputs
from dense_gemm_tmem_gb300.gemm import Gemm

from gpu_helpers import (as_f64, check, reset_opts, run, sample_rows, set_opts, to_dev, TDT)

pytestmark = pytest.mark.gpu
F16, F32 = inputs.F16, inputs.F32
TC, SK, SIMT, TC2, SPLITC = (B.GEMM_KERNEL_TC, B.GEMM_KERNEL_STREAMK, B.GEMM_KERNEL_SIMT,
                              B.GEMM_KERNEL_TC2, B.GEMM_KERNEL_SPLITC)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def g(dev):
    h = Gemm(dev)
    yield h
    h.close()


@pytest.fixture(autouse=True)
def _clean_options(request):
    yield
    if "g" in request.fixturenames:
        reset_opts(request.getfixturevalue("g"))


def problem(M, N, K, am, bm, idt, odt, bias, seed, kind="uniform"):
    return inputs.make_problem("t", M, N, K, am, bm, idt, odt, kind, bias, seed)


def full_check(g, dev, p):
    C = run(g, p, dev)
    ref = oracle.gemm(p.A, p.B, p.bias, a_major=p.a_major, b_major=p.b_major)
    return check(as_f64(C), ref, p)


# ---------------------------------------------------------------- layouts --
@pytest.mark.parametrize("kernel", [-1, TC, SK])
@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("odt", [F16, F32])
@pytest.mark.parametrize("bias", [False, True])
def test_tc_layouts_ragged(g, dev, kernel, am, bm, odt, bias):
    """296 x 520 x 200: 3 tile rows (the last 40 high), 3 tile columns of 256
    (the last 8 wide), 4 k-blocks (the last 8 deep), all four storage pairs."""
    set_opts(g, kernel=kernel)
    p = problem(296, 520, 200, am, bm, F16, odt, bias, 10 + am + 2 * bm)
    full_check(g, dev, p)


@pytest.mark.parametrize("case", [
    ("tc", 296, 520, 200, 0, 1, {"kernel": TC}),
    ("tc_persistent", 600, 1000, 328, 1, 0, {"kernel": TC, "grid": 5}),
    ("streamk", 392, 600, 1480, 0, 1, {"kernel": SK, "grid": 37}),
    ("pair", 520, 776, 1032, 0, 0, {"kernel": TC2}),
    ("pair_persistent", 1000, 1000, 1480, 0, 1, {"kernel": TC2, "grid": 6}),
    ("pair_split", 520, 776, 2056, 0, 1, {"kernel": TC2, "pair_split": 1, "grid": 14}),
    ("csplit", 296, 520, 2048, 0, 1, {"kernel": SPLITC, "csplit": 4}),
    ("swapped", 16, 2048, 4096, 0, 0, {}),
    ("swapped_sk", 40, 3000, 1000, 0, 1, {"kernel": SK, "swap": 1, "grid": 29}),
])
@pytest.mark.parametrize("odt", [F16, F32])
def test_bias_as_reduction_init(g, dev, case, odt):
    """GEMM_OPT_BIAS_INIT: each tile's reduction starts from the bias seeded
    into the accumulator (split tiles: only the k-block-0 part carries it)."""
    name, M, N, K, am, bm, opts = case
    set_opts(g, bias_init=1, **opts)
    p = problem(M, N, K, am, bm, F16, odt, True, 200 + len(name) + (odt == F32))
    full_check(g, dev, p)


def test_bias_as_reduction_init_exact(g, dev):
    """Integer-valued inputs and bias: seeding the reduction with the bias
    gives the same exact values as adding it last."""
    for opts in ({"kernel": TC}, {"kernel": SK, "grid": 23}, {"kernel": TC2},
                 {"kernel": SPLITC, "csplit": 8}):
        set_opts(g, bias_init=1, **opts)
        p = problem(384, 520, 1024, 0, 1, F16, F32, True, 210, kind="int")
        ref = oracle.gemm(p.A, p.B, p.bias, b_major=1)
        assert np.array_equal(as_f64(run(g, p, dev)), ref)
        reset_opts(g)


@pytest.mark.parametrize("kernel", [TC, SK, TC2])
@pytest.mark.parametrize("odt", [F16, F32])
def test_plain_store_path(g, dev, kernel, odt):
    """The epilogue's plain-store path on an output the TMA could take
    (GEMM_OPT_TMA_STORE = 0): same results as the TMA-store path."""
    set_opts(g, kernel=kernel, tma_store=0)
    p = problem(296, 520, 200, 0, 1, F16, odt, True, 160 + (odt == F32))
    full_check(g, dev, p)


@pytest.mark.parametrize("kernel", [TC, SK, TC2])
@pytest.mark.parametrize("odt", [F16, F32])
def test_tma_store_path_forced(g, dev, kernel, odt):
    """GEMM_OPT_TMA_STORE = 1: TMA stores even where the default takes plain
    stores (fp32 output on a single wave of tiles)."""
    set_opts(g, kernel=kernel, tma_store=1)
    p = problem(296, 520, 200, 0, 1, F16, odt, True, 162 + (odt == F32))
    full_check(g, dev, p)


@pytest.mark.parametrize("kernel,grid,odt,want", [
    (TC2, 4, F16, 1),    # 20 pair tiles on 2 pairs: 10 per pair, TMA stores
    (TC2, 6, F16, 0),    # on 3 pairs: 6.7 per pair, plain stores
    (TC2, 10, F32, 1),   # on 5 pairs: 4 per pair
    (TC2, 12, F32, 0),   # on 6 pairs: 3.3 per pair
    (TC, 8, F16, 1),     # 80 one-SM 128 x 128 tiles on 8 CTAs
    (TC, 20, F32, 1),
    (TC, 40, F32, 0),
])
def test_default_store_path_by_waves(g, dev, kernel, grid, odt, want):
    """The default store path follows the waves per CTA (per pair): TMA stores
    from 10 output tiles per CTA for fp16 output and from 4 for fp32, plain
    stores below; either way the oracle's result."""
    odt_b = B.GEMM_F16 if odt == F16 else B.GEMM_F32
    M, N, K = 1280, 1024, 192
    set_opts(g, kernel=kernel, grid=grid, tile_n=(-1 if kernel == TC2 else 128))
    pl = g.plan(M, N, K, 0, 1, B.GEMM_F16, odt_b)
    assert (pl["kernel"], pl["grid"], pl["tma_store"]) == (kernel, grid, want), pl
    p = problem(M, N, K, 0, 1, F16, odt, True, 440 + grid + (odt == F32))
    full_check(g, dev, p)


@pytest.mark.parametrize("kernel", [TC, TC2])
@pytest.mark.parametrize("odt", [F16, F32])
def test_output_pitch_not_16_bytes(g, dev, kernel, odt):
    """C rows of 536 or 1064 bytes: no TMA store; the plain stores write C."""
    N = 268 if odt == F16 else 266
    set_opts(g, kernel=kernel)
    p = problem(300, N, 200, 0, 1, F16, odt, True, 165 + (odt == F32))
    full_check(g, dev, p)


@pytest.mark.parametrize("tile_n,bm", [(32, 1), (64, 0), (64, 1)])
@pytest.mark.parametrize("kernel", [TC, SK])
@pytest.mark.parametrize("odt", [F16, F32])
def test_narrow_tiles(g, dev, tile_n, bm, kernel, odt):
    """32- and 64-column tiles without swapping (a row-major B needs 64)."""
    set_opts(g, kernel=kernel, tile_n=tile_n)
    p = problem(300, 520, 328, 0, bm, F16, odt, True, 220 + tile_n + bm)
    pl = g.plan(300, 520, 328, 0, bm, B.GEMM_F16, B.GEMM_F16 if odt == F16 else B.GEMM_F32)
    assert pl["tile_n"] == tile_n and pl["swap_ab"] == 0
    full_check(g, dev, p)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("kernel", [TC, SK])
def test_tc_tile_widths(g, dev, tile_n, kernel):
    set_opts(g, kernel=kernel, tile_n=tile_n)
    p = problem(400, 776, 328, 0, 0, F16, F32, True, 21)
    full_check(g, dev, p)


@pytest.mark.parametrize("M", [1, 3, 16, 40, 64, 100, 128])
@pytest.mark.parametrize("bm", [0, 1])
@pytest.mark.parametrize("odt", [F16, F32])
def test_swapped_skinny(g, dev, M, bm, odt):
    """Skinny M runs with swapped operands (Cᵀ = Bᵀ·Aᵀ) and a transposed store:
    by the picker's choice up to M = 64, forced beyond."""
    if M > 64:
        set_opts(g, swap=1)
    p = problem(M, 1000, 520, 0, bm, F16, odt, True, 30 + M)
    pl = g.plan(M, 1000, 520, 0, bm, B.GEMM_F16, B.GEMM_F16 if odt == F16 else B.GEMM_F32)
    assert pl["swap_ab"] == 1
    full_check(g, dev, p)


@pytest.mark.parametrize("tile_n", [16, 32, 64, 128])
@pytest.mark.parametrize("kernel", [TC, SK])
def test_swapped_tile_widths(g, dev, tile_n, kernel):
    set_opts(g, kernel=kernel, tile_n=tile_n, swap=1)
    p = problem(72, 640, 1032, 0, 0, F16, F32, True, 41)
    full_check(g, dev, p)


@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("odt", [F16, F32])
@pytest.mark.parametrize("bias", [False, True])
def test_tile64_layouts_ragged(g, dev, am, bm, odt, bias):
    """64-row tiles (the M = 64 MMA: 16 rows per TMEM lane quarter) on 296 x
    520 x 200: 5 tile rows (the last 40 high), 9 tile columns (the last 8
    wide), 4 k-blocks (the last 8 deep), every layout, bias and output type."""
    set_opts(g, tile_m=64)
    p = problem(296, 520, 200, am, bm, F16, odt, bias, 300 + 2 * am + bm)
    pl = g.plan(296, 520, 200, am, bm, B.GEMM_F16, B.GEMM_F16 if odt == F16 else B.GEMM_F32)
    assert (pl["tile_m"], pl["kernel"]) == (64, TC)
    full_check(g, dev, p)


@pytest.mark.parametrize("tile_n,bm", [(32, 1), (64, 0), (128, 0), (128, 1)])
@pytest.mark.parametrize("grid,stages", [(-1, -1), (5, 3)])
def test_tile64_widths_rings_and_waves(g, dev, tile_n, bm, grid, stages):
    """64-row tiles of every width on 200 x 296 x 2000 (32 k-blocks, more than
    the ring holds), once one tile per CTA and once 5 CTAs walking all tiles
    with a 3-stage ring (both accumulators and every ring phase wrap around)."""
    set_opts(g, tile_m=64, tile_n=tile_n, grid=grid, stages=stages)
    p = problem(200, 296, 2000, 0, bm, F16, F32, True, 310 + tile_n + grid)
    pl = g.plan(200, 296, 2000, 0, bm)
    assert (pl["kernel"], pl["tile_m"], pl["tile_n"]) == (TC, 64, tile_n)
    if grid > 0:
        assert pl["grid"] == grid and pl["stages"] == stages
    full_check(g, dev, p)


@pytest.mark.parametrize("am,bm,tile_n", [(0, 0, 64), (0, 1, 32), (1, 0, 128), (1, 1, 64),
                                          (0, 1, 128)])
def test_tile64_k_groups(g, dev, am, bm, tile_n):
    """64-row tiles with 1, 2 and 4 k-blocks per TMA copy (3-D boxes for a
    K-major operand, deeper boxes for an MN-major one) on 296 x 520 x 320:
    5 k-blocks, so the last group is short.  Every grouping gives the same
    bits (the MMAs run in the same k order) and matches the oracle."""
    p = problem(296, 520, 320, am, bm, F16, F32, True, 330 + 2 * am + bm)
    ref = oracle.gemm(p.A, p.B, p.bias, a_major=am, b_major=bm)
    outs = []
    for kg in (1, 2, 4):
        set_opts(g, tile_m=64, tile_n=tile_n, k_group=kg)
        pl = g.plan(296, 520, 320, am, bm)
        assert (pl["kernel"], pl["tile_m"], pl["tile_n"], pl["k_group"]) == (TC, 64, tile_n, kg)
        C = run(g, p, dev)
        check(as_f64(C), ref, p)
        outs.append(C.cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("kg,stages", [(2, 4), (4, 4), (4, 8)])
def test_tile64_k_groups_ring_wrap(g, dev, kg, stages):
    """Groups of k-blocks through a short ring: 5 CTAs walk all 20 tiles of
    200 x 296 x 1024 (16 k-blocks each), so ring phases and accumulators wrap
    many times."""
    set_opts(g, tile_m=64, tile_n=64, grid=5, stages=stages, k_group=kg)
    p = problem(200, 296, 1024, 0, 1, F16, F16, True, 340 + kg + stages)
    pl = g.plan(200, 296, 1024, 0, 1, B.GEMM_F16, B.GEMM_F16)
    assert (pl["tile_m"], pl["grid"], pl["stages"], pl["k_group"]) == (64, 5, stages, kg)
    full_check(g, dev, p)


def test_tile64_k_groups_mn_major_ragged_k(g, dev):
    """Both operands MN-major with K = 200 (not a multiple of 64): 4 k-blocks
    in one copy per operand, the zeros past K filled by the TMA unit."""
    set_opts(g, tile_m=64)
    p = problem(256, 384, 200, 1, 0, F16, F32, False, 350)
    pl = g.plan(256, 384, 200, 1, 0)
    assert (pl["tile_m"], pl["k_group"]) == (64, 4)
    full_check(g, dev, p)


ONE_SM_K_GROUP_CASES = [
    # name, M, N, K, am, bm, odt, opts
    ("whole_256", 520, 776, 1088, 0, 1, F16, {"kernel": TC, "tile_n": 256}),
    ("whole_128_mn", 520, 776, 1088, 1, 0, F32, {"kernel": TC, "tile_n": 128}),
    ("whole_64_rr", 520, 776, 1088, 0, 0, F32, {"kernel": TC, "tile_n": 64}),
    ("whole_cc", 520, 776, 1088, 1, 1, F16, {"kernel": TC}),
    ("streamk", 384, 512, 1088, 0, 1, F32, {"kernel": SK, "grid": 23}),
    ("csplit_push", 512, 512, 1088, 0, 1, F32, {"kernel": SPLITC, "csplit": 4, "tile_n": 64}),
    ("csplit_park", 512, 512, 1088, 0, 0, F16, {"kernel": SPLITC, "csplit": 4, "tile_n": 128}),
    ("skinny", 16, 1024, 2048, 0, 0, F32, {}),
    ("skinny_col", 40, 1536, 1024, 0, 1, F16, {}),
]


@pytest.mark.parametrize("case", ONE_SM_K_GROUP_CASES, ids=[c[0] for c in ONE_SM_K_GROUP_CASES])
def test_one_sm_k_groups(g, dev, case):
    """The 128-row one-SM kernel with 2 and 4 k-blocks per stage and TMA copy
    against 1: whole tiles of every width and layout, Stream-K ranges that
    start and end inside groups, cluster splits (pushed and parked partials)
    whose ranks' ranges are not multiples of the group, and swapped skinny
    products.  K = 1088 gives 17 k-blocks (a short last group).  Every
    grouping gives the same bits and matches the oracle."""
    _, M, N, K, am, bm, odt, opts = case
    odt_b = B.GEMM_F16 if odt == F16 else B.GEMM_F32
    p = problem(M, N, K, am, bm, F16, odt, True, 360 + M % 97)
    outs = []
    for kg in (1, 2, 4):
        set_opts(g, k_group=kg, tile_m=128, **opts)
        pl = g.plan(M, N, K, am, bm, B.GEMM_F16, odt_b)
        assert pl["tile_m"] == 128 and pl["kernel"] != TC2
        assert pl["k_group"] in (1, kg) and pl["stages"] % pl["k_group"] == 0
        if kg > 1 and pl["stages"] >= 2 * kg:
            assert pl["k_group"] == kg
        outs.append(run(g, p, dev).cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref = oracle.gemm(p.A, p.B, p.bias, a_major=am, b_major=bm)
    check(as_f64(outs[2]), ref, p)


def test_tile64_unaligned_output(g, dev):
    """64-row tiles writing a C whose rows are not 16-byte aligned (the
    element-wise store path)."""
    set_opts(g, tile_m=64)
    p = problem(130, 70, 136, 0, 1, F16, F32, True, 320)
    A, Bt, bias = to_dev(p, dev)
    big = torch.empty(p.M * p.N + 1, dtype=torch.float32, device=dev)
    C = big[1:].view(p.M, p.N)
    g.run(A, Bt, C, bias, 0, 1)
    g.status()
    check(as_f64(C), oracle.gemm(p.A, p.B, p.bias, b_major=1), p)


@pytest.mark.parametrize("kernel,tile_n,stages,want", [
    (TC, -1, 1, 1), (TC, -1, 2, 2), (SK, -1, 3, 3),
    (SPLITC, 64, 1, 1),     # partials pushed into the staging area: any ring
    (SPLITC, 128, 1, 3),    # parked in the ring: it must hold 128 x 132 fp32
    (SPLITC, 128, 3, 3)])
def test_short_rings(g, dev, kernel, tile_n, stages, want):
    """The one-SM kernel with a ring of 1 to 3 stages (a launch may use fewer
    stages than the ring holds): every stage is refilled many times.  A
    cluster split that parks its partial in the ring keeps enough stages to
    hold it, whatever is asked."""
    set_opts(g, kernel=kernel, tile_n=tile_n, stages=stages)
    p = problem(296, 520, 1000, 0, 1, F16, F32, True, 180 + stages)
    assert g.plan(296, 520, 1000, 0, 1)["stages"] == want
    full_check(g, dev, p)


def test_lean_ring_for_wide_cluster_split(g, dev):
    """A cluster split over more than half the SMs runs with a ring short
    enough for two CTAs per SM where the kernel's registers allow it and the
    ring still keeps enough loads in flight (so the next launch's CTAs start
    beside this one's): skinny M = 16 (16-wide swapped tiles, 5 stages, one
    k-block per copy: a short ring keeps its stages single)."""
    w = inputs.WORKLOADS["skinny_m16_4096"]
    pl = g.plan(w.M, w.N, w.K, w.a_major, w.b_major, B.GEMM_F16, B.GEMM_F32)
    assert pl["kernel"] == SPLITC and pl["grid"] > 76
    assert (pl["stages"], pl["k_group"]) == (5, 1)
    full_check(g, dev, w.make())


@pytest.mark.parametrize("grid", [1, 5, 37, 152])
def test_split_grid_sizes(g, dev, grid):
    """Stream-K with awkward CTA counts: ranges start and end mid-tile."""
    set_opts(g, kernel=SK, grid=grid)
    p = problem(392, 600, 1480, 0, 1, F16, F32, True, 50 + grid)
    full_check(g, dev, p)


@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("odt", [F16, F32])
@pytest.mark.parametrize("bias", [False, True])
def test_pair_layouts_ragged(g, dev, am, bm, odt, bias):
    """Two-SM kernel on 296 x 520 x 200: the second pair tile has 40 valid rows,
    all in the leader CTA, so the peer CTA computes only zero-filled rows."""
    set_opts(g, kernel=TC2)
    p = problem(296, 520, 200, am, bm, F16, odt, bias, 110 + am + 2 * bm)
    pl = g.plan(296, 520, 200, am, bm, B.GEMM_F16, B.GEMM_F16 if odt == F16 else B.GEMM_F32)
    assert pl["kernel"] == TC2 and pl["tile_m"] == 256
    full_check(g, dev, p)


@pytest.mark.parametrize("grid", [2, 6, 150])
def test_pair_grid_sizes(g, dev, grid):
    """16 pair tiles on 1, 3 or 75 CTA pairs: each pair walks many tiles, both
    accumulators and every pipeline phase wrap around."""
    set_opts(g, kernel=TC2, grid=grid)
    p = problem(1000, 1000, 1480, 0, 1, F16, F32, True, 120 + grid)
    assert g.plan(1000, 1000, 1480, 0, 1)["grid"] == min(grid, 32)
    full_check(g, dev, p)


@pytest.mark.parametrize("odt", [F16, F32])
def test_pair_dynamic_matches_static(g, dev, odt):
    """Two-SM kernel over several waves of whole tiles (9 x 17 pair tiles,
    ragged on both sides): with GEMM_OPT_DYNAMIC_TILES = 1 the pairs take
    tiles from a counter at run time; with 0 (the default), in the static
    order.  A tile's k order depends on the tile alone, so both give the same
    bits, which match the oracle; the counter resets itself at the end of a
    launch, so a second launch gives them again."""
    p = problem(2048 + 40, 4096 + 8, 1032, 0, 1, F16, odt, True, 160)
    set_opts(g, kernel=TC2, dyn=1)
    assert g.plan(p.M, p.N, p.K, 0, 1, B.GEMM_F16,
                  B.GEMM_F16 if odt == F16 else B.GEMM_F32)["dp_tiles"] == 9 * 17
    C_dyn = run(g, p, dev)
    C_dyn2 = run(g, p, dev)
    set_opts(g, dyn=0)
    C_st = run(g, p, dev)
    assert torch.equal(C_dyn, C_dyn2) and torch.equal(C_dyn, C_st)
    rows = sample_rows(p.M, 13)
    check(as_f64(C_dyn, rows), oracle.gemm_rows(p.A, p.B, p.bias, b_major=1, rows=rows), p, rows)


@pytest.mark.parametrize("am,bm,odt", [(0, 1, F16), (0, 0, F32), (1, 0, F16), (1, 1, F32)])
@pytest.mark.parametrize("split", [False, True])
def test_pair_k_groups(g, dev, am, bm, odt, split):
    """Two-SM kernel with 2 or 3 k-blocks per stage and TMA copy (3-D boxes
    for a K-major operand, deeper boxes for an MN-major one) against 1, on
    1040 x 1040 x 1088: 17 k-blocks, so the last group is short.  Whole tiles:
    25 pair tiles on 3 pairs, every other wave walking k backwards; split: a
    Stream-K split over 7 pairs, whose ranges start and end inside groups.
    Both groupings give the same bits (the same k order) and match the
    oracle."""
    M = N = 1040
    K = 1088
    odt_b = B.GEMM_F16 if odt == F16 else B.GEMM_F32
    p = problem(M, N, K, am, bm, F16, odt, True, 170 + 2 * am + bm + 4 * split)
    opts = dict(kernel=TC2, pair_split=1, grid=14) if split else dict(kernel=TC2, grid=6)
    outs = []
    for kg in (1, 2, 3):
        set_opts(g, k_group=kg, **opts)
        pl = g.plan(M, N, K, am, bm, B.GEMM_F16, odt_b)
        assert (pl["kernel"], pl["k_group"], pl["sk_tiles"] > 0) == (TC2, kg, split)
        outs.append(run(g, p, dev).cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref = oracle.gemm(p.A, p.B, p.bias, a_major=am, b_major=bm)
    check(as_f64(outs[1]), ref, p)


@pytest.mark.parametrize("grid", [2, 10, 38, 152])
def test_pair_split_grid_sizes(g, dev, grid):
    """Two-SM Stream-K: every pair tile's k-blocks split over grid / 2 pairs;
    ranges start and end mid-tile and each CTA half is added by the last pair
    to arrive."""
    set_opts(g, kernel=TC2, pair_split=1, grid=grid)
    p = problem(520, 776, 2056, 0, 1, F16, F32, True, 90 + grid)
    pl = g.plan(520, 776, 2056, 0, 1)
    assert pl["kernel"] == TC2 and (pl["dp_tiles"], pl["sk_tiles"]) == (0, 12)
    full_check(g, dev, p)


@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("odt", [F16, F32])
def test_pair_split_layouts(g, dev, am, bm, odt):
    set_opts(g, kernel=TC2, pair_split=1, grid=22)
    p = problem(296, 520, 2048, am, bm, F16, odt, True, 150 + 4 * am + 2 * bm + (odt == F32))
    full_check(g, dev, p)


def test_pair_tail_split(g, dev):
    """Whole pair tiles first, then the last two waves split: 20 pair tiles on
    6 pairs -> 12 whole, 8 split."""
    set_opts(g, kernel=TC2, pair_split=2, grid=12)
    pl = g.plan(1000, 1200, 1000, 0, 1, B.GEMM_F16, B.GEMM_F16)
    assert (pl["dp_tiles"], pl["sk_tiles"], pl["grid"]) == (12, 8, 12)
    p = problem(1000, 1200, 1000, 0, 1, F16, F16, True, 95)
    full_check(g, dev, p)


@pytest.mark.parametrize("csplit", [2, 4, 8])
@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("odt", [F16, F32])
def test_cluster_split_layouts(g, dev, csplit, am, bm, odt):
    """Each tile's 17 k-blocks split over a cluster of 2, 4 or 8 CTAs (ranges
    of 2 or 3 k-blocks), partials added in distributed shared memory."""
    set_opts(g, kernel=SPLITC, csplit=csplit)
    p = problem(296, 520, 1032, am, bm, F16, odt, True, 140 + csplit + am + 2 * bm)
    pl = g.plan(296, 520, 1032, am, bm, B.GEMM_F16, B.GEMM_F16 if odt == F16 else B.GEMM_F32)
    assert pl["kernel"] == SPLITC and pl["cluster_split"] == csplit
    full_check(g, dev, p)


@pytest.mark.parametrize("csplit", [2, 4, 8])
@pytest.mark.parametrize("am,bm", [(0, 0), (1, 1)])
@pytest.mark.parametrize("odt", [F16, F32])
def test_cluster_split_narrow_unswapped(g, dev, csplit, am, bm, odt):
    """64-column unswapped tiles split over clusters (the parked partials of a
    64-wide tile, rows of 68 floats), with ragged M, N and K."""
    set_opts(g, kernel=SPLITC, csplit=csplit, tile_n=64)
    p = problem(296, 200, 1032, am, bm, F16, odt, True, 170 + csplit + am)
    pl = g.plan(296, 200, 1032, am, bm, B.GEMM_F16, B.GEMM_F16 if odt == F16 else B.GEMM_F32)
    assert pl["kernel"] == SPLITC and pl["cluster_split"] == csplit and pl["tile_n"] == 64
    full_check(g, dev, p)


@pytest.mark.parametrize("M,N,K,w", [(512, 512, 1024, 64), (384, 384, 2048, 64),
                                     (256, 256, 1024, 64), (512, 1024, 2048, 64),
                                     (1024, 1024, 2048, 128)])
def test_cluster_split_picker_widths(g, dev, M, N, K, w):
    """The picker's own cluster splits (width and size by per-CTA cost)."""
    p = problem(M, N, K, 0, 1, F16, F32, True, 180 + M + K)
    pl = g.plan(M, N, K, 0, 1, B.GEMM_F16, B.GEMM_F32)
    assert pl["kernel"] == SPLITC and pl["tile_n"] == w and pl["swap_ab"] == 0
    full_check(g, dev, p)


@pytest.mark.parametrize("tile_n", [16, 32, 64, 128])
@pytest.mark.parametrize("csplit", [2, 4, 8])
@pytest.mark.parametrize("odt", [F16, F32])
def test_cluster_split_swapped(g, dev, tile_n, csplit, odt):
    """Swapped cluster splits: tiles of up to 64 columns push their partials
    to the owning CTA, wider ones are read from the peers."""
    set_opts(g, kernel=SPLITC, csplit=csplit, tile_n=tile_n, swap=1)
    p = problem(72, 640, 1032, 0, 0, F16, odt, True, 150 + tile_n + (odt == F32))
    full_check(g, dev, p)


def test_split_many_contributors(g, dev):
    """One output tile whose 256 k-blocks are split over 128 CTAs (2 each):
    the fixup adds 128 partials in batches."""
    set_opts(g, kernel=SK, grid=128)
    p = problem(128, 128, 16384, 0, 0, F16, F32, True, 61)
    pl = g.plan(128, 128, 16384)
    assert pl["kernel"] == SK and pl["grid"] == 128
    full_check(g, dev, p)


# ---------------------------------------------------------- closed forms --
@pytest.mark.parametrize("kernel", [TC, SK, TC2, SPLITC])
@pytest.mark.parametrize("bm", [0, 1])
def test_permutation_rows_exact(g, dev, kernel, bm):
    """A = P: C must be B's rows permuted, exactly (catches swizzle, descriptor
    and lane-mapping mistakes, which permute or mix elements)."""
    set_opts(g, kernel=kernel)
    n = 512
    perm = np.random.default_rng(7).permutation(n)
    P = np.zeros((n, n), np.float16)
    P[np.arange(n), perm] = 1
    Bs = inputs.draw(inputs.storage_shape_b(n, 384, bm), 71, "uniform", F16)
    Bl = Bs if bm == 0 else Bs.T
    p = inputs.Problem("perm", n, 384, n, P, Bs, None, 0, bm, F16, F32)
    got = as_f64(run(g, p, dev))
    assert np.array_equal(got, Bl[perm].astype(np.float64))


@pytest.mark.parametrize("kernel", [TC, SK, TC2, SPLITC])
def test_permutation_columns_exact(g, dev, kernel):
    set_opts(g, kernel=kernel)
    n = 512
    perm = np.random.default_rng(8).permutation(n)
    P = np.zeros((n, n), np.float16)
    P[np.arange(n), perm] = 1
    A = inputs.draw((264, n), 72, "uniform", F16)
    p = inputs.Problem("permc", 264, n, n, A, P, None, 0, 0, F16, F16)
    got = as_f64(run(g, p, dev))
    assert np.array_equal(got, A[:, np.argsort(perm)].astype(np.float64))


@pytest.mark.parametrize("case", [
    ("tc", 384, 512, 1024, 0, 1, F16, F32, {"kernel": TC}),
    ("tc16", 384, 512, 1024, 0, 0, F16, F16, {"kernel": TC}),
    ("sk", 384, 512, 1024, 1, 0, F16, F32, {"kernel": SK, "grid": 23}),
    ("sk16", 256, 768, 2048, 0, 1, F16, F16, {"kernel": SK}),
    ("swap", 16, 2048, 4096, 0, 0, F16, F32, {}),
    ("simt", 200, 300, 500, 0, 0, F32, F32, {}),
    ("simt_col", 200, 300, 500, 1, 1, F32, F32, {}),
    ("simt_split", 300, 420, 1000, 1, 0, F32, F32, {"grid": 23}),
    ("simt_f16", 300, 420, 1000, 1, 0, F16, F16, {"kernel": SIMT, "grid": 23}),
    ("pair", 520, 776, 1032, 0, 1, F16, F32, {"kernel": TC2}),
    ("pair16", 296, 520, 2048, 1, 0, F16, F16, {"kernel": TC2, "grid": 4}),
    ("pair_split", 520, 776, 1032, 0, 1, F16, F32, {"kernel": TC2, "pair_split": 1, "grid": 14}),
    ("csplit", 296, 520, 2048, 0, 1, F16, F32, {"kernel": SPLITC, "csplit": 8}),
    ("csplit_swap", 16, 2048, 4096, 0, 0, F16, F16, {"kernel": SPLITC, "csplit": 4}),
])
def test_integer_inputs_exact(g, dev, case):
    """Integer-valued inputs: every partial sum is an integer below 2^24, so
    any summation order gives the exact result: values must match exactly
    (+0 and -0 count as equal)."""
    name, M, N, K, am, bm, idt, odt, opts = case
    set_opts(g, **opts)
    p = problem(M, N, K, am, bm, idt, odt, True, 80, kind="int")
    ref = oracle.gemm(p.A, p.B, p.bias, a_major=am, b_major=bm)
    assert np.abs(ref).max() <= 2048
    assert np.array_equal(as_f64(run(g, p, dev)), ref)


def test_all_ones_gives_k(g, dev):
    M, N, K = 300, 264, 1000
    p = inputs.Problem("ones", M, N, K, np.ones((M, K), np.float16), np.ones((K, N), np.float16),
                       None, 0, 0, F16, F32)
    assert np.array_equal(as_f64(run(g, p, dev)), np.full((M, N), float(K)))


_GOLDEN_CASES = [
    (1, 1, F16, {}), (1, 1, F32, {}), (300, 264, F16, {"kernel": TC}),
    (520, 776, F16, {"kernel": TC2}), (384, 512, F16, {"kernel": SK, "grid": 23}),
    (16, 2048, F16, {"kernel": SPLITC, "csplit": 2}), (200, 300, F32, {}),
    (300, 420, F16, {"kernel": SIMT, "grid": 23})]


# fp32 operands give fp32 output only
@pytest.mark.parametrize("M,N,idt,opts,odt", [
    c + (odt,) for c in _GOLDEN_CASES for odt in (F16, F32) if c[2] == F16 or odt == F32])
def test_golden_block_sum(g, dev, M, N, idt, opts, odt):
    """Every output is the pages' worked reduction 0 + 1 + ... + 255 = 32640
    (tests/golden/block_sum_arange256.txt): each row of A is the ramp
    0..K-1 and B (column-major) is all ones; exact in any summation order."""
    gv = golden_values.load("block_sum_arange256.txt")
    K = int(gv["K"])
    set_opts(g, **opts)
    npdt = np.float16 if idt == F16 else np.float32
    A = np.tile(np.arange(K, dtype=npdt), (M, 1))
    p = inputs.Problem("golden", M, N, K, A, np.ones((N, K), npdt), None, 0, 1, idt, odt)
    assert np.array_equal(as_f64(run(g, p, dev)), np.full((M, N), gv["C"]))


# ------------------------------------------------------------ edge cases --
@pytest.mark.parametrize("odt", [F16, F32])
def test_k_zero_gives_bias(g, dev, odt):
    bias = torch.arange(40, dtype=torch.float32, device=dev) - 7.5
    A = torch.empty((33, 0), dtype=torch.float16, device=dev)
    Bt = torch.empty((0, 40), dtype=torch.float16, device=dev)
    C = g(A, Bt, bias, out_dtype=TDT[odt])
    g.status()
    assert torch.equal(C.float(), bias.expand(33, 40).to(TDT[odt]).float())
    C = g(A, Bt, None, out_dtype=TDT[odt])
    g.status()
    assert torch.count_nonzero(C) == 0


def test_empty_outputs_are_noops(g, dev):
    for M, N in ((0, 16), (16, 0)):
        A = torch.zeros((M, 8), dtype=torch.float16, device=dev)
        Bt = torch.zeros((8, N), dtype=torch.float16, device=dev)
        C = g(A, Bt)
        g.status()
        assert C.shape == (M, N)


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (300, 8, 64), (8, 8, 4096), (129, 264, 8)])
def test_tiny_and_thin(g, dev, M, N, K):
    p = problem(M, N, K, 0, 0, F16, F32, True, 90 + M)
    full_check(g, dev, p)


def test_fp16_alignment_rules(g, dev):
    A = torch.zeros((64, 104), dtype=torch.float16, device=dev)
    Bt = torch.zeros((100, 64), dtype=torch.float16, device=dev)
    C = torch.empty((64, 64), dtype=torch.float32, device=dev)
    with pytest.raises(ValueError):
        g.run(A[:, :100], Bt, C)  # not contiguous -> rejected before the C-ABI


@pytest.mark.parametrize("odt", [F16, F32])
def test_fp16_odd_leading_dims_run_on_cuda_cores(g, dev, odt):
    """lda = K = 100 breaks the TMA stride rule: the CUDA-core kernel runs it
    with fp32 accumulation."""
    ocode = B.GEMM_F16 if odt == F16 else B.GEMM_F32
    assert g.plan(70, 64, 100, 0, 0, B.GEMM_F16, ocode)["kernel"] == SIMT
    p = problem(70, 64, 100, 0, 0, F16, odt, True, 170 + (odt == F32))
    full_check(g, dev, p)


@pytest.mark.parametrize("odt", [F16, F32])
def test_fp16_unaligned_bases_run_on_cuda_cores(g, dev, odt):
    """A and B based 2 bytes past a 16-byte boundary: the TMA cannot read them,
    the CUDA-core kernel does."""
    M, N, K = 130, 264, 200
    p = problem(M, N, K, 0, 1, F16, odt, True, 175 + (odt == F32))
    A, Bt, bias = to_dev(p, dev)
    af = torch.zeros(A.numel() + 1, dtype=torch.float16, device=dev)
    af[1:] = A.flatten()
    bf = torch.zeros(Bt.numel() + 1, dtype=torch.float16, device=dev)
    bf[1:] = Bt.flatten()
    C = torch.empty((M, N), dtype=TDT[odt], device=dev)
    ocode = B.GEMM_F16 if odt == F16 else B.GEMM_F32
    rc = B.gemm_run(g.handle, M, N, K, af[1:].data_ptr(), bf[1:].data_ptr(), bias.data_ptr(),
                    C.data_ptr(), B.layout(0, 1, B.GEMM_F16, ocode),
                    torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0
    g.status()
    check(as_f64(C), oracle.gemm(p.A, p.B, p.bias, b_major=1), p)


@pytest.mark.parametrize("tile", [64, 128])
@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("odt", [F16, F32])
def test_fp16_cuda_core_layouts(g, dev, tile, am, bm, odt):
    set_opts(g, kernel=SIMT, tile_n=tile)
    p = problem(130, 70, 96, am, bm, F16, odt, True, 180 + 4 * am + 2 * bm + (odt == F32))
    full_check(g, dev, p)


@pytest.mark.parametrize("grid", [3, 37, 304])
def test_fp16_cuda_core_split(g, dev, grid):
    set_opts(g, kernel=SIMT, grid=grid)
    p = problem(392, 600, 1480, 0, 1, F16, F16, True, 190 + grid)
    assert g.plan(392, 600, 1480, 0, 1, B.GEMM_F16, B.GEMM_F16)["grid"] == grid
    full_check(g, dev, p)


def test_unaligned_outputs_and_bias(g, dev):
    """C and bias have no alignment rule: offset both by one element."""
    p = problem(130, 264, 72, 0, 0, F16, F16, True, 95)
    A, Bt, bias = to_dev(p, dev)
    cflat = torch.zeros(130 * 264 + 1, dtype=torch.float16, device=dev)
    bflat = torch.zeros(265, dtype=torch.float32, device=dev)
    bflat[1:] = bias
    rc = B.gemm_run(g.handle, 130, 264, 72, A.data_ptr(), Bt.data_ptr(), bflat[1:].data_ptr(),
                    cflat[1:].data_ptr(), B.layout(0, 0, B.GEMM_F16, B.GEMM_F16),
                    torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0
    g.status()
    ref = oracle.gemm(p.A, p.B, p.bias)
    check(cflat[1:].view(130, 264).double().cpu().numpy(), ref, p)


@pytest.mark.parametrize("tile", [64, 128])
@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(130, 70, 33), (257, 129, 128), (5, 3, 2)])
def test_simt_layouts_ragged(g, dev, tile, am, bm, M, N, K):
    set_opts(g, tile_n=tile)
    p = problem(M, N, K, am, bm, F32, F32, True, 100 + M)
    full_check(g, dev, p)


@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("K", [16, 17, 1000, 1024])
@pytest.mark.parametrize("grid", [0, 7])
@pytest.mark.parametrize("tile", [64, 128])
def test_simt_interior_and_ragged_k(g, dev, am, bm, K, grid, tile):
    """fp32, every tile inside M and N: the unchecked interior loop (direct
    global-to-shared copies for operands stored m/n-contiguous) runs all
    whole k-blocks, the checked loop only a ragged last one; with a forced
    grid the k ranges of the split start and end inside tiles."""
    set_opts(g, tile_n=tile)
    if grid:
        set_opts(g, grid=grid)
    p = problem(256, 384, K, am, bm, F32, F32, True, 300 + K + 2 * am + bm)
    full_check(g, dev, p)


@pytest.mark.parametrize("tile", [64, 128])
@pytest.mark.parametrize("grid", [1, 5, 37, 304])
def test_simt_split_grid_sizes(g, dev, tile, grid):
    """fp32 Stream-K with awkward CTA counts: ranges start and end mid-tile and
    the last CTA to arrive adds the partials."""
    set_opts(g, tile_n=tile, grid=grid)
    p = problem(392, 600, 1480, 0, 1, F32, F32, True, 60 + grid)
    pl = g.plan(392, 600, 1480, 0, 1, B.GEMM_F32, B.GEMM_F32)
    assert pl["kernel"] == SIMT and pl["grid"] == grid
    full_check(g, dev, p)


@pytest.mark.parametrize("am,bm", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_simt_split_layouts(g, dev, am, bm):
    set_opts(g, grid=41)
    p = problem(300, 452, 1000, am, bm, F32, F32, True, 70 + 2 * am + bm)
    full_check(g, dev, p)


def test_simt_unaligned_pointers(g, dev):
    p = problem(100, 68, 36, 0, 0, F32, F32, False, 111)
    A, Bt, _ = to_dev(p, dev)
    af = torch.zeros(A.numel() + 1, dtype=torch.float32, device=dev)
    af[1:] = A.flatten()
    C = torch.empty((100, 68), dtype=torch.float32, device=dev)
    rc = B.gemm_run(g.handle, 100, 68, 36, af[1:].data_ptr(), Bt.data_ptr(), None, C.data_ptr(),
                    B.layout(0, 0, B.GEMM_F32, B.GEMM_F32),
                    torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0
    g.status()
    check(as_f64(C), oracle.gemm(p.A, p.B), p)


def test_fp32_to_fp16_unsupported(g, dev):
    A = torch.zeros((8, 8), dtype=torch.float32, device=dev)
    with pytest.raises(B.GemmError) as e:
        g(A, A, out_dtype=torch.float16)
    assert e.value.code == B.GEMM_ERR_UNSUPPORTED


def test_side_stream(g, dev):
    p = problem(256, 512, 256, 0, 1, F16, F32, True, 120)
    A, Bt, bias = to_dev(p, dev)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        C = g(A, Bt, bias, 0, 1, stream=s)
    g.status(s)
    check(as_f64(C), oracle.gemm(p.A, p.B, p.bias, b_major=1), p)


# ----------------------------------------------------------- determinism --
@pytest.mark.parametrize("kernel,grid", [(SK, -1), (SK, 29), (TC, -1), (TC2, -1), (SPLITC, -1)])
def test_bitwise_repeatable(g, dev, kernel, grid):
    set_opts(g, kernel=kernel, grid=grid)
    p = problem(520, 776, 2056, 0, 1, F16, F32, True, 130, kind="normal")
    A, Bt, bias = to_dev(p, dev)
    C1 = g(A, Bt, bias, 0, 1)
    C2 = g(A, Bt, bias, 0, 1)
    g.status()
    assert torch.equal(C1, C2)


def test_pair_split_bitwise_repeatable(g, dev):
    set_opts(g, kernel=TC2, pair_split=1, grid=14)
    p = problem(520, 776, 2056, 0, 1, F16, F32, True, 132, kind="normal")
    A, Bt, bias = to_dev(p, dev)
    C1 = g(A, Bt, bias, 0, 1)
    C2 = g(A, Bt, bias, 0, 1)
    g.status()
    assert torch.equal(C1, C2)


def test_simt_split_bitwise_repeatable(g, dev):
    set_opts(g, grid=29)
    p = problem(520, 776, 2056, 0, 0, F32, F32, True, 131, kind="normal")
    A, Bt, bias = to_dev(p, dev)
    C1 = g(A, Bt, bias, 0, 0)
    C2 = g(A, Bt, bias, 0, 0)
    g.status()
    assert torch.equal(C1, C2)


# ------------------------------------------------------ failure detection --
def test_wait_timeout_selftest(g, dev):
    """A bounded device wait that nothing completes must expire, be reported
    by gemm_status, and leave the handle and context usable."""
    s = torch.cuda.current_stream(dev).cuda_stream
    assert B.gemm_selftest_wait_timeout(g.handle, 5_000_000, s) == B.GEMM_OK
    assert B.gemm_status(g.handle, s) == B.GEMM_ERR_DEVICE_TIMEOUT
    assert B.gemm_status_detail(g.handle) == 6
    assert B.gemm_status(g.handle, s) == B.GEMM_OK
    p = problem(256, 256, 512, 0, 0, F16, F32, False, 140)
    full_check(g, dev, p)


@pytest.mark.parametrize("kernel,shape", [
    (TC, (1024, 1024, 8192)),     # one-SM kernel, whole tiles
    (SK, (512, 512, 65536)),      # one-SM kernel, Stream-K partials through the workspace
    (SPLITC, (512, 512, 32768)),  # one-SM kernel, cluster split (partials on chip)
    (TC2, (2048, 2048, 8192)),    # two-SM kernel (CTA pairs)
])
def test_real_kernel_wait_timeout(g, dev, kernel, shape):
    """Each CTA of these launches waits tens of microseconds for its first
    accumulator.  A wait limit of 1 us makes the kernels' own
    bounded waits give up mid-launch: gemm_status reports
    GEMM_ERR_DEVICE_TIMEOUT with the role whose wait expired first (TMA
    producer, MMA issuer or epilogue; never the clean-up, whose waits keep at
    least gemm_drain_limit_ns), and the next launch on the same handle, with
    the default limit, matches the oracle."""
    M, N, K = shape
    p = problem(M, N, K, 0, 1, F16, F32, True, 150 + kernel)
    set_opts(g, kernel=kernel)
    assert g.plan(M, N, K, 0, 1, B.GEMM_F16, B.GEMM_F32)["kernel"] == kernel
    A, Bt, bias = to_dev(p, dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    g.set_option(B.GEMM_OPT_WAIT_LIMIT_NS, 1000)
    g(A, Bt, bias, 0, 1, out_dtype=torch.float32)
    assert B.gemm_status(g.handle, s) == B.GEMM_ERR_DEVICE_TIMEOUT
    assert B.gemm_status_detail(g.handle) in (1, 2, 3, 4)
    g.set_option(B.GEMM_OPT_WAIT_LIMIT_NS, -1)
    C = g(A, Bt, bias, 0, 1, out_dtype=torch.float32)
    g.status()
    rows = sample_rows(M, 9)
    check(as_f64(C, rows), oracle.gemm_rows(p.A, p.B, p.bias, b_major=1, rows=rows), p, rows)


def test_alloc_failure_injection(dev):
    """Allocation failures made on the host (gemm_inject_alloc_failure): each
    of gemm_create's three device allocations in turn fails with
    GEMM_ERR_ALLOC and leaves nothing allocated; a failed buffer growth in
    gemm_run_host returns GEMM_ERR_ALLOC and the handle keeps working, on
    device buffers and, once the failure is disarmed, on host buffers."""
    import ctypes
    lib = B.load()
    torch.cuda.synchronize(dev)
    free0 = torch.cuda.mem_get_info(dev)[0]
    try:
        for k in (1, 2, 3):
            assert B.gemm_inject_alloc_failure(k) == B.GEMM_OK
            h = ctypes.c_void_p()
            assert lib.gemm_create(ctypes.byref(h), dev.index) == B.GEMM_ERR_ALLOC
            assert not h.value
        assert B.gemm_inject_alloc_failure(0) == B.GEMM_OK
        torch.cuda.synchronize(dev)
        assert abs(torch.cuda.mem_get_info(dev)[0] - free0) < (4 << 20)  # the 38 MiB workspace is gone
        g = Gemm(dev)
        p = problem(300, 260, 200, 0, 1, F16, F32, True, 170)
        hA, hB, hbias = (torch.from_numpy(x).pin_memory() for x in (p.A, p.B, p.bias))
        hC = torch.empty((p.M, p.N), dtype=torch.float32).pin_memory()
        B.gemm_inject_alloc_failure(1)
        with pytest.raises(B.GemmError) as e:
            g.run_host(hA, hB, hC, hbias, 0, 1)
        assert e.value.code == B.GEMM_ERR_ALLOC
        B.gemm_inject_alloc_failure(0)
        full_check(g, dev, p)  # device buffers: unaffected
        g.run_host(hA, hB, hC, hbias, 0, 1)
        g.status()
        check(as_f64(hC), oracle.gemm(p.A, p.B, p.bias, b_major=1), p)
        g.close()
    finally:
        B.gemm_inject_alloc_failure(0)


# ------------------------------------------------- the named workloads --
def test_workload_512_full(g, dev):
    p = inputs.WORKLOADS["gemm512_f16_f32out"].make()
    full_check(g, dev, p)


def test_workload_tile128_full(g, dev):
    p = inputs.WORKLOADS["tile128_f16_f32out"].make()
    full_check(g, dev, p)


def test_workload_sgemm2048_full(g, dev):
    p = inputs.WORKLOADS["sgemm2048_f32"].make()
    pl = g.plan(2048, 2048, 2048, 0, 0, B.GEMM_F32, B.GEMM_F32)
    assert pl["kernel"] == SIMT and pl["sk_tiles"] == 256  # split over the resident CTAs
    full_check(g, dev, p)


@pytest.mark.parametrize("M", [1, 16, 64, 128])
def test_workload_skinny_full(g, dev, M):
    p = inputs.WORKLOADS["skinny_m%d_4096" % M].make()
    full_check(g, dev, p)


@pytest.mark.parametrize("name,kind", [("gemm8192_f16_bias_f16out", None),
                                       ("gemm8192_f16_bias_f16out", "int"),
                                       ("gemm16384_f16_f16out", None),
                                       ("gemm16384_f16_f16out", "int")])
def test_workload_large_sampled_rows(g, dev, name, kind):
    """Full-size launch (the configuration the benchmark times), checked on one
    seeded row per 128-row tile plus edge rows, all N columns each."""
    w = inputs.WORKLOADS[name]
    p = w.make(kind=kind)
    pl = g.plan(w.M, w.N, w.K, w.a_major, w.b_major, B.GEMM_F16, B.GEMM_F16)
    assert pl["kernel"] == TC2 and pl["tile_n"] == 256
    C = run(g, p, dev)
    rows = sample_rows(w.M, 7)
    got = as_f64(C, rows)
    del C
    ref = oracle.gemm_rows(p.A, p.B, p.bias, a_major=p.a_major, b_major=p.b_major, rows=rows)
    if kind == "int":
        assert np.abs(ref).max() <= 2048
        assert np.array_equal(got, ref)
    else:
        check(got, ref, p, rows)


# ------------------------------------------------------------- host buffers --
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("odt", [F16, F32])
def test_run_host_matches_oracle(g, dev, pinned, odt):
    """gemm_run_host: host operands copied in, the GEMM, the result copied out,
    all on one stream; pinned and pageable host memory."""
    p = problem(300, 520, 1000, 0, 1, F16, odt, True, 200 + pinned + 2 * (odt == F32))
    hA = torch.from_numpy(p.A)
    hB = torch.from_numpy(p.B)
    hbias = torch.from_numpy(p.bias)
    hC = torch.empty((p.M, p.N), dtype=TDT[odt])
    if pinned:
        hA, hB, hbias, hC = hA.pin_memory(), hB.pin_memory(), hbias.pin_memory(), hC.pin_memory()
    g.run_host(hA, hB, hC, hbias, p.a_major, p.b_major)
    g.status()
    check(as_f64(hC), oracle.gemm(p.A, p.B, p.bias, a_major=p.a_major, b_major=p.b_major), p)


def test_run_host_buffers_grow_and_fp32(g, dev):
    """The handle's device buffers grow to the largest problem and stay valid
    for smaller ones; the fp32 path runs through the same call."""
    for (M, N, K, idt) in [(64, 96, 40, F16), (700, 300, 900, F32), (64, 96, 40, F32)]:
        odt = F32
        p = problem(M, N, K, 0, 0, idt, odt, True, 210 + M)
        hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
        hA, hB, hbias = (torch.from_numpy(x).pin_memory() for x in (p.A, p.B, p.bias))
        g.run_host(hA, hB, hC, hbias, 0, 0)
        g.status()  # the copies read hA, hB, hbias until here
        check(as_f64(hC), oracle.gemm(p.A, p.B, p.bias), p)


def test_run_host_one_handle_two_streams(g, dev):
    """Two calls on one handle from two streams share its device buffers:
    the second call's copies wait for the first call's work, so both
    results are right."""
    ps = [problem(520, 392, 1032, 0, 1, F16, F32, True, 230 + i) for i in range(2)]
    ss = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    hCs = [torch.empty((p.M, p.N), dtype=torch.float32).pin_memory() for p in ps]
    # every host buffer stays referenced until both streams are done: the
    # copies run after the calls return
    hins = [[torch.from_numpy(x).pin_memory() for x in (p.A, p.B, p.bias)] for p in ps]
    for (hA, hB, hbias), s, hC in zip(hins, ss, hCs):
        g.run_host(hA, hB, hC, hbias, 0, 1, stream=s)
    for s in ss:
        g.status(s)
    for p, hC in zip(ps, hCs):
        check(as_f64(hC), oracle.gemm(p.A, p.B, p.bias, b_major=1), p)


def test_run_host_two_streams_regrow(g, dev):
    """A call on a second stream that needs larger device buffers than the
    handle holds: the host waits for the previous call's work before freeing
    the old buffers, so the first call (still running on its own stream) and
    the second both come out right."""
    ps = [problem(256, 384, 2048, 0, 1, F16, F32, True, 240),
          problem(1536, 1280, 2056, 0, 1, F16, F32, True, 241)]
    h = Gemm(dev)  # a fresh handle: no buffers yet
    try:
        ss = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
        hCs = [torch.empty((p.M, p.N), dtype=torch.float32).pin_memory() for p in ps]
        hins = [[torch.from_numpy(x).pin_memory() for x in (p.A, p.B, p.bias)] for p in ps]
        for (hA, hB, hbias), s, hC in zip(hins, ss, hCs):
            h.run_host(hA, hB, hC, hbias, 0, 1, stream=s)
        for s in ss:
            h.status(s)
        for i, (p, hC) in enumerate(zip(ps, hCs)):
            rows = None if i == 0 else sample_rows(p.M, 11)
            got = as_f64(hC) if rows is None else hC.double().numpy()[rows]
            check(got, oracle.gemm_rows(p.A, p.B, p.bias, b_major=1, rows=rows), p, rows)
    finally:
        h.close()
