"""CPU oracle of the fused gated group-RMSNorm -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and it shares no code
with them.

The arithmetic lives in ``ggrn_oracle.cpp`` (plain single-threaded C++, f32 as
the pages fix it).  This module only compiles it with g++ and marshals
arguments through ctypes.

Pinned by ``tests/test_oracle_pins.py``: hand-worked fixtures under
``tests/golden/``, closed forms, library special cases (torch dtype
conversions, ``torch.nn.functional.rms_norm`` and ``silu``), brute force in
double precision and invariants; ``tests/test_oracle_mutants.py`` checks that
plausible mistakes planted in a copy of the source fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ggrn_oracle.cpp")
HDR = os.path.join(HERE, "ggrn_oracle.h")
LIB_PATH = os.path.join(HERE, "libggrn_oracle.so")

F32, F16, BF16 = 0, 1, 2
MAMBA2, ONNX = 0, 1
DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
            "-Wall", "-Wextra"]


def compile_oracle(src: str, out_path: str, include_dir: str = HERE) -> str:
    """Compile one oracle source file into a shared library at ``out_path``."""
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.run(["g++", *CXXFLAGS, "-I", include_dir, "-o", tmp, src], check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``libggrn_oracle.so`` next to its source if it is missing or stale."""
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    return compile_oracle(SRC, LIB_PATH)


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"oracle returned status {status}")
        self.status = status


def _row_stride(t: torch.Tensor, width: int) -> int:
    if t.dim() != 2 or (t.shape[0] > 0 and t.stride(1) != 1):
        raise ValueError("oracle inputs are 2-D with unit inner stride")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), width)


class Oracle:
    """ctypes wrapper of one compiled oracle library."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        i64, vp, f, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        args = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f, ci, ci]
        for name in ("ggrn_oracle_forward", "ggrn_oracle_forward_f64"):
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ci
        L.ggrn_oracle_forward_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                             f, ci, ci]
        L.ggrn_oracle_forward_ex.restype = ci
        L.ggrn_oracle_forward_pre.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                              i64, f, ci, ci]
        L.ggrn_oracle_forward_pre.restype = ci
        L.ggrn_oracle_encode.argtypes = [vp, vp, i64, ci]
        L.ggrn_oracle_encode.restype = None
        L.ggrn_oracle_decode.argtypes = [vp, vp, i64, ci]
        L.ggrn_oracle_decode.restype = None
        self.lib = L
        self.path = path

    def forward(self, y: torch.Tensor, gate: torch.Tensor, w: torch.Tensor, *, group_size: int,
                eps: float, mode: int = MAMBA2, out: torch.Tensor | None = None,
                want_t: bool = False, precision: str = "f32"):
        """Run the oracle on host tensors.

        ``y``/``gate``: 2-D CPU tensors of T, unit inner stride, any row stride.
        ``w``: f32 [width] (MAMBA2) or T [group_size] (ONNX).
        Returns ``out`` (contiguous unless given) and, with ``want_t``, the
        intermediate cast_T(gated*nf) (MAMBA2).  ``precision="f64"`` runs the
        double-precision twin.
        """
        for t in (y, gate, w):
            assert t.device.type == "cpu"
        rows, width = y.shape
        if out is None:
            out = torch.empty((rows, width), dtype=y.dtype)
        t_out = torch.empty((rows, width), dtype=y.dtype) if want_t else None
        w = w.contiguous()
        common = (rows, width, group_size, _row_stride(y, width), _row_stride(gate, width),
                  _row_stride(out, width), float(eps), DTYPE_CODE[y.dtype], mode)
        if precision == "f64":
            assert not want_t
            st = self.lib.ggrn_oracle_forward_f64(y.data_ptr(), gate.data_ptr(), w.data_ptr(),
                                                  out.data_ptr(), *common)
        else:
            st = self.lib.ggrn_oracle_forward_ex(
                y.data_ptr(), gate.data_ptr(), w.data_ptr(), out.data_ptr(),
                t_out.data_ptr() if t_out is not None else None, *common)
        if st != 0:
            raise OracleError(st)
        return (out, t_out) if want_t else out

    def forward_detail(self, y: torch.Tensor, gate: torch.Tensor, w: torch.Tensor, *,
                       group_size: int, eps: float, mode: int = MAMBA2):
        """Run the oracle and also return what the comparison rules need.

        Returns ``(out, t, pre)``: ``out`` as ``forward``; ``t`` the MAMBA2
        intermediate cast_T(gated*nf) (None in ONNX mode); ``pre`` f32
        [rows, width], each element's value just before its rounding to T
        (MAMBA2: gated*nf; ONNX: the product the store rounds).
        """
        for t in (y, gate, w):
            assert t.device.type == "cpu"
        rows, width = y.shape
        out = torch.empty((rows, width), dtype=y.dtype)
        t_out = torch.empty((rows, width), dtype=y.dtype) if mode == MAMBA2 else None
        pre = torch.empty((rows, width), dtype=torch.float32)
        w = w.contiguous()
        st = self.lib.ggrn_oracle_forward_pre(
            y.data_ptr(), gate.data_ptr(), w.data_ptr(), out.data_ptr(),
            t_out.data_ptr() if t_out is not None else None, pre.data_ptr(), rows, width,
            group_size, _row_stride(y, width), _row_stride(gate, width), width, float(eps),
            DTYPE_CODE[y.dtype], mode)
        if st != 0:
            raise OracleError(st)
        return out, t_out, pre

    def status(self, y_ptr, gate_ptr, w_ptr, out_ptr, rows, width, group_size, ys, gs_, os_,
               eps, dtype, mode) -> int:
        """Raw call returning the status code (argument-validation tests)."""
        return self.lib.ggrn_oracle_forward(y_ptr, gate_ptr, w_ptr, out_ptr, rows, width,
                                            group_size, ys, gs_, os_, eps, dtype, mode)

    def encode(self, x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
        """f32 -> T with the oracle's own codec."""
        x = x.to(torch.float32).contiguous()
        out = torch.empty(x.shape, dtype=dtype)
        self.lib.ggrn_oracle_encode(x.data_ptr(), out.data_ptr(), x.numel(), DTYPE_CODE[dtype])
        return out

    def decode(self, x: torch.Tensor) -> torch.Tensor:
        """T -> f32 with the oracle's own codec."""
        x = x.contiguous()
        out = torch.empty(x.shape, dtype=torch.float32)
        self.lib.ggrn_oracle_decode(x.data_ptr(), out.data_ptr(), x.numel(), DTYPE_CODE[x.dtype])
        return out


_lock = threading.Lock()
_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from ``ggrn_oracle.cpp`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def forward(*args, **kwargs):
    return default().forward(*args, **kwargs)
