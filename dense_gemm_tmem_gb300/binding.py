"""ctypes binding of include/gemm.h: the same names, argument marshalling only.

Every computation happens in the CUDA library; if the library is missing this
module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

c_int, c_int32, c_int64, c_uint8, c_void_p = (ctypes.c_int, ctypes.c_int32, ctypes.c_int64,
                                              ctypes.c_uint8, ctypes.c_void_p)

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = -1
GEMM_ERR_UNSUPPORTED = -2
GEMM_ERR_ALLOC = -3
GEMM_ERR_CUDA = -4
GEMM_ERR_DEVICE_TIMEOUT = -5

GEMM_F16, GEMM_F32 = 0, 1
GEMM_ROW_MAJOR, GEMM_COL_MAJOR = 0, 1
(GEMM_KERNEL_TC, GEMM_KERNEL_STREAMK, GEMM_KERNEL_SIMT, GEMM_KERNEL_FILL, GEMM_KERNEL_NONE,
 GEMM_KERNEL_TC2, GEMM_KERNEL_SPLITC) = range(7)
(GEMM_OPT_FORCE_KERNEL, GEMM_OPT_FORCE_TILE_N, GEMM_OPT_FORCE_GRID, GEMM_OPT_WAIT_LIMIT_NS,
 GEMM_OPT_MIN_SPLIT_ITERS, GEMM_OPT_FORCE_SWAP_AB, GEMM_OPT_GROUP_M, GEMM_OPT_PAIR,
 GEMM_OPT_CLUSTER_SPLIT, GEMM_OPT_PDL, GEMM_OPT_PAIR_SPLIT, GEMM_OPT_TMA_STORE,
 GEMM_OPT_BIAS_INIT, GEMM_OPT_DYNAMIC_TILES, GEMM_OPT_STAGES, GEMM_OPT_TILE_M,
 GEMM_OPT_K_GROUP) = range(17)


class gemm_layout_t(ctypes.Structure):
    _fields_ = [("a_major", c_uint8), ("b_major", c_uint8), ("in_dtype", c_uint8),
                ("out_dtype", c_uint8)]


class gemm_plan_t(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in (
        "kernel", "swap_ab", "tile_m", "tile_n", "tile_k", "stages", "grid", "tiles_m",
        "tiles_n", "k_iters", "dp_tiles", "sk_tiles", "a_mn_major", "b_mn_major", "group_m",
        "cluster_split")] + [("workspace_bytes", c_int64), ("k_group", c_int32),
                             ("tma_store", c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemmError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        super().__init__("%s%s" % (what + ": " if what else "", gemm_strerror(code)))


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Loads the CUDA library (building it first if asked and needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path) or not _build.up_to_date():
        if not build_if_missing:
            raise RuntimeError("CUDA library not built: %s" % path)
        _build.build()
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    sig = {
        "gemm_create": (c_int, [P(c_void_p), c_int]),
        "gemm_destroy": (c_int, [c_void_p]),
        "gemm_run": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p,
                             c_void_p, c_void_p, gemm_layout_t, c_void_p]),
        "gemm_run_host": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p,
                                  c_void_p, c_void_p, gemm_layout_t, c_void_p]),
        "gemm_status": (c_int, [c_void_p, c_void_p]),
        "gemm_status_detail": (c_int, [c_void_p]),
        "gemm_set_option": (c_int, [c_void_p, c_int, c_int64]),
        "gemm_query_plan": (c_int, [c_void_p, c_int64, c_int64, c_int64, gemm_layout_t,
                                    P(gemm_plan_t)]),
        "gemm_strerror": (ctypes.c_char_p, [c_int]),
        "gemm_plan_for": (c_int, [c_int64, c_int64, c_int64, gemm_layout_t, c_int,
                                  P(gemm_plan_t)]),
        "gemm_work_units": (c_int, [P(gemm_plan_t), c_int, P(c_int32), c_int]),
        "gemm_split_contributors": (c_int, [P(gemm_plan_t), c_int, P(c_int32), P(c_int32)]),
        "gemm_simt_smem_strides": (c_int, [P(c_int32), P(c_int32)]),
        "gemm_drain_limit_ns": (c_int64, [c_int64]),
        "gemm_inject_alloc_failure": (c_int, [c_int64]),
        "gemm_selftest_wait_timeout": (c_int, [c_void_p, c_int64, c_void_p]),
        "gemm_set_trace": (c_int, [c_void_p, c_void_p, c_int64]),
        "gemm_run_noalloc": (c_int, [c_int64, c_int64, c_int64, c_void_p, c_void_p, c_void_p,
                                     c_void_p, gemm_layout_t, c_void_p, c_void_p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def layout(a_major=0, b_major=0, in_dtype=GEMM_F16, out_dtype=GEMM_F32) -> gemm_layout_t:
    return gemm_layout_t(a_major, b_major, in_dtype, out_dtype)


# ---- the C-ABI, one wrapper per function --------------------------------------
def gemm_strerror(code: int) -> str:
    return load().gemm_strerror(int(code)).decode()


def gemm_create(device: int = 0) -> int:
    h = c_void_p()
    rc = load().gemm_create(ctypes.byref(h), int(device))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_create")
    return h.value


def gemm_destroy(h) -> int:
    return load().gemm_destroy(c_void_p(h))


def gemm_run(h, M, N, K, A_ptr, B_ptr, bias_ptr, C_ptr, lay: gemm_layout_t, stream_ptr) -> int:
    return load().gemm_run(c_void_p(h), int(M), int(N), int(K), c_void_p(A_ptr),
                           c_void_p(B_ptr), c_void_p(bias_ptr), c_void_p(C_ptr), lay,
                           c_void_p(stream_ptr))


def gemm_run_host(h, M, N, K, A_ptr, B_ptr, bias_ptr, C_ptr, lay: gemm_layout_t,
                  stream_ptr) -> int:
    return load().gemm_run_host(c_void_p(h), int(M), int(N), int(K), c_void_p(A_ptr),
                                c_void_p(B_ptr), c_void_p(bias_ptr), c_void_p(C_ptr), lay,
                                c_void_p(stream_ptr))


def gemm_status(h, stream_ptr) -> int:
    return load().gemm_status(c_void_p(h), c_void_p(stream_ptr))


def gemm_status_detail(h) -> int:
    return load().gemm_status_detail(c_void_p(h))


def gemm_set_option(h, option: int, value: int) -> int:
    return load().gemm_set_option(c_void_p(h), int(option), int(value))


def gemm_query_plan(h, M, N, K, lay: gemm_layout_t):
    p = gemm_plan_t()
    rc = load().gemm_query_plan(c_void_p(h), int(M), int(N), int(K), lay, ctypes.byref(p))
    return rc, p


def gemm_plan_for(M, N, K, lay: gemm_layout_t, num_sms: int):
    p = gemm_plan_t()
    rc = load().gemm_plan_for(int(M), int(N), int(K), lay, int(num_sms), ctypes.byref(p))
    return rc, p


def gemm_work_units(plan: gemm_plan_t, cta: int):
    n = load().gemm_work_units(ctypes.byref(plan), int(cta), None, 0)
    if n < 0:
        raise GemmError(n, "gemm_work_units")
    buf = (c_int32 * (3 * max(n, 1)))()
    n2 = load().gemm_work_units(ctypes.byref(plan), int(cta), buf, n)
    assert n2 == n
    return [(buf[3 * i], buf[3 * i + 1], buf[3 * i + 2]) for i in range(n)]


def gemm_split_contributors(plan: gemm_plan_t, sk_tile: int):
    f, l = c_int32(), c_int32()
    rc = load().gemm_split_contributors(ctypes.byref(plan), int(sk_tile), ctypes.byref(f),
                                        ctypes.byref(l))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_split_contributors")
    return f.value, l.value


def gemm_simt_smem_strides():
    a, b = c_int32(), c_int32()
    rc = load().gemm_simt_smem_strides(ctypes.byref(a), ctypes.byref(b))
    if rc != GEMM_OK:
        raise GemmError(rc, "gemm_simt_smem_strides")
    return a.value, b.value


def gemm_inject_alloc_failure(n: int) -> int:
    return load().gemm_inject_alloc_failure(int(n))


def gemm_drain_limit_ns(wait_limit_ns: int) -> int:
    return load().gemm_drain_limit_ns(int(wait_limit_ns))


def gemm_selftest_wait_timeout(h, limit_ns: int, stream_ptr) -> int:
    return load().gemm_selftest_wait_timeout(c_void_p(h), int(limit_ns), c_void_p(stream_ptr))


def gemm_run_noalloc(M, N, K, A_ptr, B_ptr, bias_ptr, C_ptr, lay: gemm_layout_t, stream_ptr,
                     status_ptr=None) -> int:
    """The allocation-free entry point (no handle; scratch compiled into the
    library).  Pointers are device addresses on the current device."""
    return load().gemm_run_noalloc(int(M), int(N), int(K), c_void_p(A_ptr), c_void_p(B_ptr),
                                   c_void_p(bias_ptr), c_void_p(C_ptr), lay,
                                   c_void_p(stream_ptr), c_void_p(status_ptr))


def gemm_set_trace(h, dev_buf_ptr, ctas: int) -> int:
    """Points the handle's tensor-core launches at a device buffer of
    ctas x 8 uint64 phase stamps (None / 0 turns tracing off)."""
    return load().gemm_set_trace(c_void_p(h), c_void_p(dev_buf_ptr), int(ctas))


TRACE_PHASES = ("start", "first_load", "first_data", "mma_done", "last_accum", "end")
TRACE_SLOTS = 12  # per CTA: the phases above, units, cluster done, entry, exit, cluster steps
TRACE_UNITS, TRACE_CLUSTER_DONE, TRACE_ENTRY, TRACE_EXIT = 6, 7, 8, 9
TRACE_CLUSTER_PARKED, TRACE_CLUSTER_REDUCED = 10, 11
