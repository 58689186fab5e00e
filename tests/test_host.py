"""Host-side checks that need no GPU: the library loads and exports every
declared symbol, the tile picker, the Stream-K work partition against the
oracle's reading, the padded staging strides, and source/binary lints."""
import os
import re
import subprocess

import pytest

from dense_gemm_tmem_gb300 import binding as B
from oracle import schedule

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMS = 152
F16, F32 = B.GEMM_F16, B.GEMM_F32


@pytest.fixture(scope="module")
def lib():
    return B.load()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^(?:int|int64_t|const char \*)\s*(gemm_\w+)\(", txt, re.M)
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12 and "gemm_drain_limit_ns" in names
    for n in names:
        assert hasattr(lib, n), n


def test_no_library_gemm_or_cuda_driver_link(lib):
    """The product links no cuBLAS/CUTLASS and does not link libcuda directly."""
    out = subprocess.run(["nm", "-D", "--undefined-only", B.library_path()],
                         capture_output=True, text=True, check=True).stdout
    assert "cublas" not in out.lower() and "cutlass" not in out.lower()
    deps = subprocess.run(["ldd", B.library_path()], capture_output=True, text=True).stdout
    assert "libcuda.so" not in deps and "libcublas" not in deps


@pytest.mark.parametrize("src", ["simt.cu", "tc2.cu", "tc_n256.cu", "tc_n128.cu", "tc_small.cu", "tc_narrow.cu"])
def test_kernels_keep_registers_without_spills(src):
    """The hot kernels fit their registers: ptxas reports no spill stores (the
    128 x 128 CUDA-core kernel sits at the 128-register cap of 2 CTAs per SM,
    where a small change elsewhere can push it into local memory), except a
    few words in the CUDA-core fallback instantiations."""
    from dense_gemm_tmem_gb300 import build as bld
    try:
        nvcc = bld._nvcc()
    except Exception:
        pytest.skip("nvcc not found")
    csrc = os.path.join(os.path.dirname(bld.__file__), "csrc")
    r = subprocess.run([nvcc] + bld.NVCC_FLAGS + ["-Xptxas", "-v", "-c", os.path.join(csrc, src),
                        "-o", os.devnull], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    kernels = re.findall(r"Compiling entry function '(\S+)'.*?(\d+) bytes spill stores",
                         r.stderr, re.S)
    assert kernels, r.stderr[-2000:]
    for name, spill in kernels:
        # The CUDA-core kernels' fallback instantiations (an operand stored
        # k-contiguous or with unaligned rows keeps its staging registers
        # through the k loop) may spill a few words; the direct-copy ones the
        # aligned fp32 layouts run may not.
        fallback = "simt_sgemm_kernel" in name and not name.endswith("Lb1EEEvNS0_8SimtArgsE")
        assert int(spill) <= (32 if fallback else 0), (name, spill)


def test_sources_use_no_multicast_loads_or_wgmma():
    """No TMA multicast loads (every CTA fetches its own operand tiles), and no
    Hopper/legacy MMA forms.  A tcgen05.commit multicast (a completion signal to
    both CTAs of a pair) is not a load and is allowed."""
    csrc = os.path.join(ROOT, "dense_gemm_tmem_gb300", "csrc")
    for fn in os.listdir(csrc):
        txt = open(os.path.join(csrc, fn)).read()
        for line in txt.splitlines():
            if "cp.async.bulk" in line:
                assert "multicast" not in line, (fn, line)
        assert "wgmma" not in txt, fn
        assert "mma.sync" not in txt and "wmma::" not in txt, fn


def test_strerror(lib):
    assert B.gemm_strerror(0) == "GEMM_OK"
    assert "UNSUPPORTED" in B.gemm_strerror(-2)
    assert B.gemm_strerror(12345) == "unknown gemm status"


def plan(M, N, K, am=0, bm=0, idt=F16, odt=F32, sms=SMS):
    rc, p = B.gemm_plan_for(M, N, K, B.layout(am, bm, idt, odt), sms)
    return rc, p


def test_picker_large_square_two_sm_tiles():
    """Large shapes run on CTA pairs: 256 x 256 whole tiles on 76 pairs (8192^3:
    1024 pair tiles = 13 waves + 36; a Stream-K tail measured slower)."""
    rc, p = plan(8192, 8192, 8192, 0, 1, F16, F16)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_TC2
    assert (p.tile_m, p.tile_n, p.tile_k, p.stages) == (256, 256, 64, 6)
    assert (p.tiles_m, p.tiles_n, p.k_iters) == (32, 32, 128)
    assert (p.dp_tiles, p.sk_tiles, p.grid, p.workspace_bytes) == (1024, 0, SMS, 0)
    assert (p.swap_ab, p.a_mn_major, p.b_mn_major) == (0, 0, 0)
    assert p.group_m == 16  # raster groups of 4096 rows of A (16 pair tiles)
    rc, p = plan(16384, 16384, 16384, 0, 0, F16, F16)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_TC2 and p.b_mn_major == 1
    assert p.dp_tiles == 64 * 64 and p.sk_tiles == 0 and p.workspace_bytes == 0


def test_picker_pair_rule():
    # at least half as many pair tiles as pairs (38 of 76): the two-SM kernel,
    # whole tiles, even when the last wave is part-empty
    rc, p = plan(1280, 5120, 4096)  # 100 pair tiles: 1.3 waves
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_TC2
    assert (p.grid, p.dp_tiles, p.sk_tiles) == (SMS, 100, 0)
    rc, p = plan(2048, 2048, 4096)  # 64 pair tiles on 64 pairs
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_TC2 and (p.grid, p.dp_tiles) == (128, 64)
    rc, p = plan(1024, 19 * 256, 4096)  # one wave: 76 = 4 x 19
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_TC2 and p.grid == 152
    # shallow (K <= 1024) with at most one wave of pair tiles: one-SM 128 x 256
    # whole tiles instead
    rc, p = plan(2048, 2048, 1024)
    assert (p.kernel, p.tile_m, p.tile_n, p.grid, p.dp_tiles) == (B.GEMM_KERNEL_TC, 128, 256, 128, 128)
    rc, p = plan(1280, 5120, 1024)  # 100 pair tiles: 1.3 waves stay on pairs
    assert p.kernel == B.GEMM_KERNEL_TC2
    rc, p = plan(2048, 2048, 2048)  # K = 2048: pairs
    assert p.kernel == B.GEMM_KERNEL_TC2
    rc, p = plan(8192, 8192, 1024)  # 1024 pair tiles: 13.5 waves stay on pairs
    assert p.kernel == B.GEMM_KERNEL_TC2
    # fewer pair tiles (32): the one-SM rules (here 128 whole tiles of 128 x 128)
    rc, p = plan(1024, 2048, 4096)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_TC
    assert (p.tile_n, p.grid, p.dp_tiles, p.sk_tiles) == (128, 128, 128, 0)
    # skinny shapes swap operands and never pair
    rc, p = plan(64, 65536, 4096)
    assert rc == 0 and p.swap_ab == 1 and p.kernel != B.GEMM_KERNEL_TC2


def test_picker_small_shapes():
    # 512^3: 8 k-blocks per tile is shallow -> whole tiles 64 columns wide, and
    # 64 rows high while those still fit one wave: 64 CTAs instead of 32
    rc, p = plan(512, 512, 512)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_TC
    assert (p.tile_m, p.tile_n, p.tiles_m, p.tiles_n, p.k_iters) == (64, 64, 8, 8, 8)
    assert (p.grid, p.dp_tiles, p.sk_tiles, p.workspace_bytes) == (64, 64, 0, 0)
    # the 8 k-blocks arrive in two copies of 4 per operand: a 12-block ring of 3 groups
    assert (p.k_group, p.stages) == (4, 12)
    # one 128 x 128 output, K-major B: 64 x 32 tiles while they fill under
    # half the SMs (row-major B keeps 64: its boxes are 64 columns wide)
    rc, p = plan(128, 128, 64, bm=1)
    assert (p.kernel, p.tile_m, p.tile_n, p.grid) == (B.GEMM_KERNEL_TC, 64, 32, 8)
    rc, p = plan(128, 128, 64)
    assert (p.tile_m, p.tile_n, p.grid) == (64, 64, 4)
    # 64-row tiles would not fit one wave: 128-row tiles
    rc, p = plan(1024, 1024, 768)  # 12 k-blocks: still narrow whole tiles
    assert (p.kernel, p.tile_m, p.tile_n, p.grid) == (B.GEMM_KERNEL_TC, 128, 64, 128)
    # 16 k-blocks: 32 tiles 64 columns wide in clusters of 4 (4 k-blocks each)
    # cost less per CTA than 16 tiles of 128 in clusters of 8: fewer operand
    # bytes (192 x 4 vs 256 x 2 rows of k-blocks) and far fewer partial bytes
    rc, p = plan(512, 512, 1024)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_SPLITC
    assert (p.tile_n, p.tiles_m, p.tiles_n, p.k_iters) == (64, 4, 8, 16)
    assert (p.cluster_split, p.grid, p.sk_tiles, p.workspace_bytes) == (4, 128, 32, 0)
    # 64-wide tiles in pairs exchange fewer partial bytes than 128-wide ones
    # in clusters of 4 (measured 9.7 vs 10.1 us)
    rc, p = plan(512, 1024, 2048)
    assert (p.kernel, p.tile_n, p.cluster_split, p.grid) == (B.GEMM_KERNEL_SPLITC, 64, 2, 128)
    # the cost rule keeps 128-wide tiles where they load far less per CTA
    rc, p = plan(1024, 1024, 2048)
    assert (p.kernel, p.tile_n, p.cluster_split, p.grid) == (B.GEMM_KERNEL_SPLITC, 128, 2, 128)
    # deep K: 16 tiles in clusters of 8
    rc, p = plan(512, 512, 8192)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_SPLITC
    assert (p.cluster_split, p.grid) == (8, 128)
    # 80 tiles: clusters of 2 would need 160 CTAs -> whole tiles, one per CTA
    rc, p = plan(1280, 1024, 4096)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_TC
    assert (p.tile_n, p.dp_tiles, p.grid, p.cluster_split) == (128, 80, 80, 0)
    # deep K with 48 tiles and no cluster capacity assumed away: clusters of 2
    rc, p = plan(768, 1024, 8192)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_SPLITC and p.cluster_split == 2


@pytest.mark.parametrize("bn,iters", [(256, 11), (128, 8), (64, 6), (32, 4), (16, 2)])
def test_split_granularity_per_tile_width(bn, iters):
    """The fewest k-blocks a split CTA gets: 4 x partial bytes / k-block bytes."""
    assert iters == -(-4 * 128 * bn * 4 // ((128 + bn) * 64 * 2))


@pytest.mark.parametrize("M,swapped", [(1, 1), (64, 1), (65, 0), (96, 0)])
def test_picker_swap_boundary(M, swapped):
    """Operands swap for skinny M up to 64 only (row-major A, N >= 2M)."""
    rc, p = plan(M, 4096, 4096)
    assert rc == 0 and p.swap_ab == swapped
    rc, p = plan(M, 4096, 4096, 1, 0)  # column-major A: never swapped
    assert rc == 0 and p.swap_ab == 0


def test_picker_m128_keeps_operands():
    """M = 128 fills the MMA's 128 rows: no swap (measured faster than the
    swapped 128-wide tile); 32 tiles of 128 x 128 in clusters of 4."""
    rc, p = plan(128, 4096, 4096)
    assert rc == 0 and p.swap_ab == 0 and p.tile_n == 128
    assert p.kernel == B.GEMM_KERNEL_SPLITC and p.cluster_split == 4
    assert (p.tiles_m, p.tiles_n, p.grid) == (1, 32, 128)


@pytest.mark.parametrize("M,bn", [(1, 16), (16, 16), (64, 64)])
def test_picker_skinny_swaps_operands(M, bn):
    rc, p = plan(M, 4096, 4096)
    assert rc == 0 and p.swap_ab == 1 and p.tile_n == bn
    # 32 tiles: clusters of 4 CTAs (128 CTAs), 16 k-blocks each
    assert p.kernel == B.GEMM_KERNEL_SPLITC and p.cluster_split == 4
    assert (p.tiles_m, p.tiles_n, p.k_iters) == (32, 1, 64)
    assert p.grid == 128 and p.workspace_bytes == 0
    assert (p.a_mn_major, p.b_mn_major) == (1, 0)  # Bᵀ is N-contiguous, A is K-contiguous


def test_picker_part_empty_waves_stay_whole():
    # swapped skinny shape with 314 tiles of 128 x 64 on 152 SMs: whole tiles,
    # persistent (2.07 waves); a k-split of the tail measured slower
    rc, p = plan(64, 128 * 314, 1024)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_TC and p.swap_ab == 1
    assert (p.dp_tiles, p.sk_tiles, p.grid) == (314, 0, SMS)
    assert p.group_m == 16  # 2048 rows of the MMA A side per raster group
    # 80 tiles (at least half the SMs): one whole tile per CTA
    rc, p = plan(128 * 10, 128 * 8, 4096)
    assert (p.kernel, p.dp_tiles, p.sk_tiles, p.grid) == (B.GEMM_KERNEL_TC, 80, 0, 80)


def test_picker_fp32_and_degenerate():
    # 256 tiles of 128 on 2 x 152 resident CTAs: every k-block split evenly
    # over 304 CTAs (a whole-tile launch would leave 48 SMs with one tile)
    rc, p = plan(2048, 2048, 2048, 0, 0, F32, F32)
    assert rc == 0 and p.kernel == B.GEMM_KERNEL_SIMT and p.tile_m == 128
    assert (p.grid, p.dp_tiles, p.sk_tiles, p.k_iters, p.tile_k) == (304, 0, 256, 128, 16)
    assert p.workspace_bytes == 2 * 304 * 128 * 128 * 4 and p.group_m == 16
    # whole waves of resident CTAs stay whole: 608 tiles, 2 waves
    rc, p = plan(128 * 16, 128 * 38, 512, 0, 0, F32, F32)
    assert (p.grid, p.dp_tiles, p.sk_tiles) == (608, 608, 0)
    # 404 tiles = one wave + 100: all split over 304 CTAs
    rc, p = plan(128 * 4, 128 * 101, 512, 0, 0, F32, F32)
    assert (p.grid, p.dp_tiles, p.sk_tiles) == (304, 0, 404)
    # 5 waves + 16: whole tiles
    rc, p = plan(128 * 8, 128 * 192, 64, 0, 0, F32, F32)
    assert (p.grid, p.dp_tiles, p.sk_tiles) == (1536, 1536, 0)
    # shallow K: at least 8 k-blocks per split CTA -> 160 tiles x 2 k-blocks stay whole
    rc, p = plan(128 * 10, 128 * 16, 16, 0, 0, F32, F32)
    assert (p.grid, p.dp_tiles, p.sk_tiles) == (160, 160, 0)
    # fewer 128-tiles than SMs: their k-blocks split over more CTAs (16 tiles x
    # 32 k-blocks in runs of at least 8 -> 64 CTAs)
    rc, p = plan(512, 512, 512, 0, 0, F32, F32)
    assert rc == 0 and (p.tile_m, p.grid, p.dp_tiles, p.sk_tiles) == (128, 64, 0, 16)
    # ... unless even that split runs fewer than 8 CTAs: 64x64 tiles
    rc, p = plan(128, 128, 128, 0, 0, F32, F32)
    assert rc == 0 and (p.tile_m, p.grid, p.sk_tiles) == (64, 4, 0)
    assert plan(64, 64, 64, 0, 0, F32, F16)[0] == B.GEMM_ERR_UNSUPPORTED
    assert plan(10, 10, 0)[1].kernel == B.GEMM_KERNEL_FILL
    assert plan(0, 10, 10)[1].kernel == B.GEMM_KERNEL_NONE
    assert plan(10, 0, 10)[1].kernel == B.GEMM_KERNEL_NONE
    assert plan(-1, 10, 10)[0] == B.GEMM_ERR_INVALID_ARG
    rc, _ = B.gemm_plan_for(8, 8, 8, B.layout(2, 0, F16, F32), SMS)
    assert rc == B.GEMM_ERR_INVALID_ARG


def test_picker_fp16_tma_stride_rule():
    """fp16 leading dimensions that are not a multiple of 8 elements break the
    TMA stride rule: those run on the CUDA-core kernel (fp32 accumulation)."""
    simt = B.GEMM_KERNEL_SIMT
    for args in [(64, 64, 100), (64, 100, 64), (100, 64, 64, 1, 0)]:  # K, N, M not % 8
        rc, p = plan(*args)
        assert rc == 0 and p.kernel == simt and p.tile_m == 64
    rc, p = plan(64, 100, 64, 0, 1)                             # B col-major: ldb = K
    assert rc == 0 and p.kernel != simt
    rc, p = plan(2050, 2048, 2048, 0, 0, F16, F16)              # M is no stride: tensor cores
    assert rc == 0 and p.kernel != simt
    rc, p = plan(2048, 2048, 2050, 0, 0, F16, F16)
    assert rc == 0 and p.kernel == simt and p.sk_tiles == 256 and p.grid == 304


PLANS = [(512, 512, 512, 0, 0, F16), (1, 4096, 4096, 0, 0, F16), (16, 4096, 4096, 0, 0, F16),
         (128, 4096, 4096, 0, 0, F16), (128 * 157, 512, 1024, 0, 0, F16),
         (1280, 5120, 1024, 0, 0, F16), (296, 520, 200, 0, 1, F16), (1000, 1000, 4000, 1, 1, F16),
         (8192, 8192, 8192, 0, 1, F16), (2048, 2048, 2048, 0, 0, F32),
         (128 * 4, 128 * 101, 500, 1, 1, F32), (200, 300, 500, 0, 0, F32)]


@pytest.mark.parametrize("M,N,K,am,bm,idt", PLANS)
def test_work_units_match_oracle_reading(M, N, K, am, bm, idt):
    rc, p = plan(M, N, K, am, bm, idt, F32)
    assert rc == 0
    # the two-SM kernel hands work to CTA pairs
    units = p.grid // 2 if p.kernel == B.GEMM_KERNEL_TC2 else p.grid
    if p.kernel == B.GEMM_KERNEL_SPLITC:
        ref = schedule.cluster_split_units(p.sk_tiles, p.k_iters, p.cluster_split)
    else:
        ref = schedule.streamk_units(p.dp_tiles, p.sk_tiles, p.k_iters, units)
    for c in range(units):
        assert B.gemm_work_units(p, c) == ref[c]
    with pytest.raises(B.GemmError):
        B.gemm_work_units(p, units)
    if p.sk_tiles == 0 or p.kernel == B.GEMM_KERNEL_SPLITC:
        return
    # contributors of each split tile: the CTAs touching it, in k order
    owners = {}
    for c, units in enumerate(ref):
        for tile, k0, _ in units:
            if tile >= p.dp_tiles:
                owners.setdefault(tile - p.dp_tiles, []).append((k0, c))
    for s in range(p.sk_tiles):
        cs = [c for _, c in sorted(owners[s])]
        assert B.gemm_split_contributors(p, s) == (cs[0], cs[-1])
        assert cs == list(range(cs[0], cs[-1] + 1))


def test_simt_staging_strides_follow_storage_align():
    a, b = B.gemm_simt_smem_strides()
    assert a == schedule.storage_align_strides([8, 128], [(32, 4), None])[0]
    assert b == schedule.storage_align_strides([8, 128], [(32, 4), None])[0]


def test_run_entry_points_check_handle_and_sizes(lib):
    """gemm_run and gemm_run_host reject a NULL handle before any CUDA call,
    so this runs without a GPU; the status and destroy calls do the same."""
    lay = B.layout(0, 0, B.GEMM_F16, B.GEMM_F32)
    for fn in (B.gemm_run, B.gemm_run_host):
        assert fn(None, 8, 8, 8, 1, 1, None, 1, lay, None) == B.GEMM_ERR_INVALID_ARG
        assert fn(None, -1, 8, 8, 1, 1, None, 1, lay, None) == B.GEMM_ERR_INVALID_ARG
    assert lib.gemm_status(None, None) == B.GEMM_ERR_INVALID_ARG


def test_drain_limit_has_a_floor():
    """The clean-up waits after an aborted wait (for the copies and MMAs a CTA
    issued to land before it frees TMEM and exits) keep at least one second
    whatever the wait limit, so a limit short enough to abort a launch cannot
    cut the clean-up short; longer limits carry over, and <= 0 means the
    default limit (2 s)."""
    for limit in (1, 1000, 250_000, 999_999_999):
        assert B.gemm_drain_limit_ns(limit) == 1_000_000_000
    assert B.gemm_drain_limit_ns(5_000_000_000) == 5_000_000_000
    assert B.gemm_drain_limit_ns(0) == B.gemm_drain_limit_ns(-1) == 2_000_000_000


def test_alloc_failure_injection_arguments():
    """The allocation-failure injector takes n >= 0 (0 disarms) and needs no
    GPU to be armed or disarmed."""
    assert B.gemm_inject_alloc_failure(-1) == B.GEMM_ERR_INVALID_ARG
    assert B.gemm_inject_alloc_failure(3) == B.GEMM_OK
    assert B.gemm_inject_alloc_failure(0) == B.GEMM_OK


def test_shape_workload_spec():
    from dense_gemm_tmem_gb300 import inputs
    w = inputs.workload("1x4096x4096:rr:hf")
    assert (w.M, w.N, w.K, w.a_major, w.b_major) == (1, 4096, 4096, 0, 0)
    assert (w.in_dtype, w.out_dtype, w.bias) == (inputs.F16, inputs.F32, False)
    w = inputs.workload("300x200x100:cr:ff:bias")
    assert (w.a_major, w.b_major, w.in_dtype, w.out_dtype, w.bias) == (1, 0, "f32", "f32", True)
    p = w.make()
    assert p.A.shape == (100, 300) and p.B.shape == (100, 200) and p.bias.shape == (200,)
    w = inputs.workload("64x64x64")
    assert (w.a_major, w.b_major, w.in_dtype, w.out_dtype) == (0, 1, "f16", "f16")
    assert inputs.workload("gemm512_f16_f32out") is inputs.WORKLOADS["gemm512_f16_f32out"]
    for bad in ("abc", "1x2", "1x2x3:rx", "1x2x3:rr:hq", "1x2x3:rr:hh:foo", "-1x2x3"):
        with pytest.raises(ValueError):
            inputs.workload(bad)


def test_picker_store_path():
    """Row-major output leaves by TMA store only on launches of many waves: 10
    or more output tiles per CTA (per pair on the two-SM kernel) for fp16
    output, 4 or more for fp32; plain stores below, on the 64-row kernel, for
    swapped operands (C written transposed), cluster splits and CUDA cores."""
    cases = [  # (M, N, K, a_major, b_major, out dtype) -> (kernel, tma_store)
        ((8192, 8192, 8192, 0, 1, F16), (B.GEMM_KERNEL_TC2, 1)),    # 1024 tiles on 76 pairs
        ((16384, 16384, 16384, 0, 0, F16), (B.GEMM_KERNEL_TC2, 1)),
        ((4096, 14336, 4096, 0, 1, F16), (B.GEMM_KERNEL_TC2, 1)),   # 896: 11.8 per pair
        ((6144, 6144, 6144, 0, 1, F16), (B.GEMM_KERNEL_TC2, 0)),    # 576: 7.6 per pair
        ((6144, 6144, 6144, 0, 1, F32), (B.GEMM_KERNEL_TC2, 1)),
        ((4096, 4096, 4096, 0, 1, F32), (B.GEMM_KERNEL_TC2, 0)),    # 256: 3.4 per pair
        ((2048, 2048, 2048, 0, 1, F16), (B.GEMM_KERNEL_TC2, 0)),
        ((512, 512, 512, 0, 0, F32), (B.GEMM_KERNEL_TC, 0)),        # 64-row tiles
        ((16, 4096, 4096, 0, 0, F32), (B.GEMM_KERNEL_SPLITC, 0)),   # swapped cluster split
    ]
    for (M, N, K, am, bm, odt), want in cases:
        rc, p = plan(M, N, K, am=am, bm=bm, odt=odt)
        assert rc == 0 and (p.kernel, p.tma_store) == want, (M, N, K, odt, p.as_dict())
    rc, p = plan(2048, 2048, 2048, idt=F32, odt=F32)
    assert rc == 0 and (p.kernel, p.tma_store) == (B.GEMM_KERNEL_SIMT, 0)


def test_picker_k_group():
    """k-blocks per TMA copy on the 64-row kernel: up to 4, whole groups in
    the ring; a K-major operand needs K a multiple of 64 (its 3-D view holds
    whole k-blocks), two MN-major operands do not; other kernels copy one
    k-block at a time."""
    cases = [  # (M, N, K, a_major, b_major) -> (tile_m, k_group)
        ((512, 512, 512, 0, 0), (64, 4)),
        ((512, 512, 128, 0, 0), (64, 2)),
        ((512, 512, 192, 0, 1), (64, 2)),
        ((128, 128, 64, 0, 1), (64, 1)),
        ((512, 512, 200, 0, 0), (64, 1)),    # row-major A is K-major: K % 64 != 0
        ((512, 512, 200, 1, 0), (64, 4)),    # both MN-major: zero fill past K
        ((4096, 4096, 4096, 0, 1), (256, 2)),   # two-SM kernel: 2 per copy
        ((4096, 4096, 4104, 0, 1), (256, 1)),   # K-major operands, K % 64 != 0
        ((4096, 4096, 4104, 1, 0), (256, 2)),   # both MN-major
        ((1024, 1024, 768, 0, 1), (128, 2)),    # one-SM 128-row kernel, 8-slot ring: 2
        ((1024, 1024, 776, 0, 1), (128, 1)),    # K-major, K % 64 != 0
    ]
    for (M, N, K, am, bm), want in cases:
        rc, p = plan(M, N, K, am=am, bm=bm)
        assert rc == 0 and (p.tile_m, p.k_group) == want, (M, N, K, am, bm, p.as_dict())
        assert p.stages % p.k_group == 0
