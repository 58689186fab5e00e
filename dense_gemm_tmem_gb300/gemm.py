"""Torch-facing wrapper over the C-ABI: tensors -> pointers, sizes, layout and
the current CUDA stream.  PyTorch supplies device memory and streams only."""
from __future__ import annotations

import torch

from . import binding as B

_DT = {torch.float16: B.GEMM_F16, torch.float32: B.GEMM_F32}
ROW, COL = B.GEMM_ROW_MAJOR, B.GEMM_COL_MAJOR


def problem_dims(A: torch.Tensor, Bm: torch.Tensor, a_major: int, b_major: int):
    """(M, N, K) from storage tensors: A is (M, K) row-major or (K, M)
    column-major; B is (K, N) row-major or (N, K) column-major."""
    if A.dim() != 2 or Bm.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = (A.shape[0], A.shape[1]) if a_major == ROW else (A.shape[1], A.shape[0])
    Kb, N = (Bm.shape[0], Bm.shape[1]) if b_major == ROW else (Bm.shape[1], Bm.shape[0])
    if K != Kb:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, Kb))
    return int(M), int(N), int(K)


_LAYOUTS = {}  # (a_major, b_major, in, out) -> gemm_layout_t, built once


def _layout(a_major, b_major, in_code, out_code):
    key = (a_major, b_major, in_code, out_code)
    lay = _LAYOUTS.get(key)
    if lay is None:
        lay = _LAYOUTS[key] = B.layout(a_major, b_major, in_code, out_code)
    return lay


class Gemm:
    """One library handle on one CUDA device."""

    def __init__(self, device=0):
        dev = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        if dev.index is None:
            dev = torch.device("cuda", 0)
        self.device = dev
        self.handle = B.gemm_create(dev.index)
        self._run = B.load().gemm_run  # argument types set once by the binding

    def close(self):
        if getattr(self, "handle", None):
            torch.cuda.synchronize(self.device)
            B.gemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            if getattr(self, "handle", None):
                B.gemm_destroy(self.handle)
                self.handle = None
        except Exception:
            pass

    def _stream(self, stream):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return s.cuda_stream

    def layout(self, A, Bm, C, a_major, b_major):
        return _layout(a_major, b_major, _DT[A.dtype], _DT[C.dtype])

    def run(self, A, Bm, C, bias=None, a_major=ROW, b_major=ROW, stream=None) -> None:
        """Enqueues C = A·B (+bias) into the preallocated row-major C."""
        M, N, K = problem_dims(A, Bm, a_major, b_major)
        idx = self.device.index
        for t in (A, Bm, C) + ((bias,) if bias is not None else ()):
            if t.get_device() != idx:
                raise ValueError("tensor on %s, handle on %s" % (t.device, self.device))
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")
        in_code, out_code = _DT.get(A.dtype), _DT.get(C.dtype)
        if A.dtype != Bm.dtype or in_code is None or out_code is None:
            raise TypeError("A, B: both float16 or both float32; C: float16 or float32")
        if C.dim() != 2 or C.shape[0] != M or C.shape[1] != N:
            raise ValueError("C has shape %s, expected (%d, %d)" % (tuple(C.shape), M, N))
        if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (N,)):
            raise ValueError("bias must be float32 of shape (N,)")
        rc = self._run(self.handle, M, N, K, A.data_ptr(), Bm.data_ptr(),
                       bias.data_ptr() if bias is not None else None, C.data_ptr(),
                       _layout(a_major, b_major, in_code, out_code), self._stream(stream))
        if rc != B.GEMM_OK:
            raise B.GemmError(rc, "gemm_run")

    def run_host(self, A, Bm, C, bias=None, a_major=ROW, b_major=ROW, stream=None) -> None:
        """Enqueues C = A·B (+bias) on host (CPU) tensors through gemm_run_host:
        copies in, the GEMM and the copy out all on the stream.  Pinned tensors
        (`.pin_memory()`) make the copies asynchronous; C is ready once the
        stream has reached this point (e.g. after `status()`), and every
        tensor passed must stay alive until then."""
        M, N, K = problem_dims(A, Bm, a_major, b_major)
        for t in (A, Bm, C) + ((bias,) if bias is not None else ()):
            if t.device.type != "cpu":
                raise ValueError("run_host takes host tensors; got one on %s" % t.device)
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")
        in_code, out_code = _DT.get(A.dtype), _DT.get(C.dtype)
        if A.dtype != Bm.dtype or in_code is None or out_code is None:
            raise TypeError("A, B: both float16 or both float32; C: float16 or float32")
        if C.dim() != 2 or C.shape[0] != M or C.shape[1] != N:
            raise ValueError("C has shape %s, expected (%d, %d)" % (tuple(C.shape), M, N))
        if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (N,)):
            raise ValueError("bias must be float32 of shape (N,)")
        rc = B.gemm_run_host(self.handle, M, N, K, A.data_ptr(), Bm.data_ptr(),
                             bias.data_ptr() if bias is not None else None, C.data_ptr(),
                             _layout(a_major, b_major, in_code, out_code), self._stream(stream))
        if rc != B.GEMM_OK:
            raise B.GemmError(rc, "gemm_run_host")

    def __call__(self, A, Bm, bias=None, a_major=ROW, b_major=ROW, out_dtype=torch.float32,
                 stream=None) -> torch.Tensor:
        M, N, _ = problem_dims(A, Bm, a_major, b_major)
        C = torch.empty((M, N), dtype=out_dtype, device=self.device)
        self.run(A, Bm, C, bias, a_major, b_major, stream)
        return C

    def status(self, stream=None) -> None:
        """Synchronises the stream and raises if a device-side wait expired."""
        rc = B.gemm_status(self.handle, self._stream(stream))
        if rc != B.GEMM_OK:
            raise B.GemmError(rc, "gemm_status (detail %d)" % B.gemm_status_detail(self.handle))

    def set_option(self, option: int, value: int) -> None:
        rc = B.gemm_set_option(self.handle, option, value)
        if rc != B.GEMM_OK:
            raise B.GemmError(rc, "gemm_set_option")

    def plan(self, M, N, K, a_major=ROW, b_major=ROW, in_dtype=B.GEMM_F16,
             out_dtype=B.GEMM_F32) -> dict:
        rc, p = B.gemm_query_plan(self.handle, M, N, K,
                                  B.layout(a_major, b_major, in_dtype, out_dtype))
        if rc != B.GEMM_OK:
            raise B.GemmError(rc, "gemm_query_plan")
        return p.as_dict()
