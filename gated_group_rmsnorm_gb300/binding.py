"""ctypes binding of ``libggrn.so`` (the C ABI declared in ``include/ggrn.h``).

Argument marshalling only: every step of the operation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the current
stream.  There is no fallback: if the library is missing or a call fails, an
exception says so.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

# ggrn_status
(OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_OVERLAP, ERR_CUDA, ERR_UNSUPPORTED, ERR_ARG,
 ERR_LIMIT) = range(10)
# ggrn_dtype / ggrn_mode / ggrn_path
F32, F16, BF16 = 0, 1, 2
MAMBA2, ONNX = 0, 1
PATH_AUTO, PATH_TEAM, PATH_WIDE, PATH_STRADDLE, PATH_SCALAR, PATH_STREAM, PATH_WIDE_CLUSTER = \
    range(7)
PATH_NAMES = {PATH_AUTO: "auto", PATH_TEAM: "team", PATH_WIDE: "wide",
              PATH_STRADDLE: "straddle", PATH_SCALAR: "scalar", PATH_STREAM: "stream",
              PATH_WIDE_CLUSTER: "wide_cluster"}
DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
MODE_CODE = {"mamba2": MAMBA2, "onnx": ONNX, MAMBA2: MAMBA2, ONNX: ONNX}

# The exported symbols, as include/ggrn.h declares them.
EXPORTS = ("ggrn_forward", "ggrn_forward_path", "ggrn_plan", "ggrn_graph_create",
           "ggrn_graph_launch", "ggrn_graph_destroy", "ggrn_status_string", "ggrn_version",
           "ggrn_fault_status", "ggrn_last_cuda_error", "ggrn_forward_noalloc",
           "ggrn_forward_inproj", "ggrn_forward_host", "ggrn_forward_inproj_host",
           "ggrn_host_workspace_bytes", "ggrn_selftest_wait_timeout", "ggrn_norm_outproj",
           "ggrn_norm_outproj_workspace_bytes")


class GgrnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        msg = status_string(status) if _lib is not None else f"status {status}"
        if status == ERR_CUDA and _lib is not None:
            msg += f" [{_lib.ggrn_last_cuda_error().decode()}]"
        super().__init__(f"{what}: {msg} (status {status})" if what else f"{msg} (status {status})")
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("team_lanes", ctypes.c_int32),
                ("vec_per_lane", ctypes.c_int32), ("elems_per_vec", ctypes.c_int32),
                ("grid_blocks", ctypes.c_int64), ("block_threads", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("items", ctypes.c_int64)]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["path_name"] = PATH_NAMES.get(self.path, "?")
        return d


class Call(ctypes.Structure):
    _fields_ = [("y", ctypes.c_void_p), ("gate", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("rows", ctypes.c_int64), ("width", ctypes.c_int64),
                ("group_size", ctypes.c_int64), ("y_row_stride", ctypes.c_int64),
                ("gate_row_stride", ctypes.c_int64), ("out_row_stride", ctypes.c_int64),
                ("eps", ctypes.c_float), ("dtype", ctypes.c_int32), ("mode", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load ``libggrn.so`` (building it first if it is missing and allowed)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"{path} is not built; run gated_group_rmsnorm_gb300.build")
            _build.build()
        L = ctypes.CDLL(path)
        i64, vp, f, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        L.ggrn_forward.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f, ci, ci, vp]
        L.ggrn_forward.restype = ci
        L.ggrn_selftest_wait_timeout.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, vp]
        L.ggrn_selftest_wait_timeout.restype = ci
        L.ggrn_forward_host.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f, ci, ci,
                                        vp, i64, vp]
        L.ggrn_forward_host.restype = ci
        L.ggrn_forward_inproj_host.argtypes = [vp, i64, i64, i64, vp, vp, i64, i64, i64, i64, f,
                                               ci, ci, vp, i64, vp]
        L.ggrn_forward_inproj_host.restype = ci
        L.ggrn_norm_outproj.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f, vp,
                                        i64, vp, vp]
        L.ggrn_norm_outproj.restype = ci
        L.ggrn_norm_outproj_workspace_bytes.argtypes = [i64, i64, i64]
        L.ggrn_norm_outproj_workspace_bytes.restype = i64
        L.ggrn_host_workspace_bytes.argtypes = [i64, i64, ci]
        L.ggrn_host_workspace_bytes.restype = i64
        L.ggrn_forward_inproj.argtypes = [vp, i64, i64, i64, vp, vp, i64, i64, i64, i64, f, ci, ci,
                                          vp]
        L.ggrn_forward_inproj.restype = ci
        L.ggrn_forward_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f, ci,
                                           ci, vp]
        L.ggrn_forward_noalloc.restype = ci
        L.ggrn_forward_path.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f, ci, ci,
                                        ci, vp]
        L.ggrn_forward_path.restype = ci
        L.ggrn_plan.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ci, ci, ci,
                                ctypes.POINTER(PlanInfo)]
        L.ggrn_plan.restype = ci
        L.ggrn_graph_create.argtypes = [ctypes.POINTER(Call), ctypes.c_int32,
                                        ctypes.POINTER(ctypes.c_void_p)]
        L.ggrn_graph_create.restype = ci
        L.ggrn_graph_launch.argtypes = [vp, vp]
        L.ggrn_graph_launch.restype = ci
        L.ggrn_graph_destroy.argtypes = [vp]
        L.ggrn_graph_destroy.restype = ci
        L.ggrn_status_string.argtypes = [ci]
        L.ggrn_status_string.restype = ctypes.c_char_p
        L.ggrn_version.argtypes = []
        L.ggrn_version.restype = ci
        L.ggrn_fault_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ci]
        L.ggrn_fault_status.restype = ci
        L.ggrn_last_cuda_error.argtypes = []
        L.ggrn_last_cuda_error.restype = ctypes.c_char_p
        _lib = L
        return L


def status_string(status: int) -> str:
    return load().ggrn_status_string(status).decode()


def fault_status(clear: bool = False) -> int:
    """The device status word (nonzero: a streaming kernel's bounded wait ran out)."""
    flags = ctypes.c_uint32(0)
    st = load().ggrn_fault_status(ctypes.byref(flags), 1 if clear else 0)
    if st != OK:
        raise GgrnError(st, "ggrn_fault_status")
    return flags.value


# ---------------------------------------------------------------------------
# Raw C-ABI calls (same names as the C functions).
# ---------------------------------------------------------------------------
def ggrn_forward(y, gate, w, out, rows, width, group_size, y_row_stride, gate_row_stride,
                 out_row_stride, eps, dtype, mode, stream) -> int:
    return load().ggrn_forward(y, gate, w, out, rows, width, group_size, y_row_stride,
                               gate_row_stride, out_row_stride, eps, dtype, mode, stream)


def ggrn_forward_inproj(inproj, inproj_row_stride, y_col, gate_col, w, out, out_row_stride, rows,
                        width, group_size, eps, dtype, mode, stream) -> int:
    return load().ggrn_forward_inproj(inproj, inproj_row_stride, y_col, gate_col, w, out,
                                      out_row_stride, rows, width, group_size, eps, dtype, mode,
                                      stream)


def ggrn_forward_host(y, gate, w, out, rows, width, group_size, y_row_stride, gate_row_stride,
                      out_row_stride, eps, dtype, mode, workspace, workspace_bytes, stream) -> int:
    return load().ggrn_forward_host(y, gate, w, out, rows, width, group_size, y_row_stride,
                                    gate_row_stride, out_row_stride, eps, dtype, mode, workspace,
                                    workspace_bytes, stream)


def ggrn_forward_inproj_host(inproj, inproj_row_stride, y_col, gate_col, w, out, out_row_stride,
                             rows, width, group_size, eps, dtype, mode, workspace,
                             workspace_bytes, stream) -> int:
    return load().ggrn_forward_inproj_host(inproj, inproj_row_stride, y_col, gate_col, w, out,
                                           out_row_stride, rows, width, group_size, eps, dtype,
                                           mode, workspace, workspace_bytes, stream)


def ggrn_forward_noalloc(y, gate, w, out, rows, width, group_size, y_row_stride,
                         gate_row_stride, out_row_stride, eps, dtype, mode, stream) -> int:
    """The allocation-free streaming entry point (include/ggrn.h documents when to use it)."""
    return load().ggrn_forward_noalloc(y, gate, w, out, rows, width, group_size, y_row_stride,
                                       gate_row_stride, out_row_stride, eps, dtype, mode, stream)


def ggrn_forward_path(y, gate, w, out, rows, width, group_size, y_row_stride, gate_row_stride,
                      out_row_stride, eps, dtype, mode, path, stream) -> int:
    return load().ggrn_forward_path(y, gate, w, out, rows, width, group_size, y_row_stride,
                                    gate_row_stride, out_row_stride, eps, dtype, mode, path,
                                    stream)


def ggrn_plan(y, gate, w, out, rows, width, group_size, y_row_stride, gate_row_stride,
              out_row_stride, dtype, mode, path=PATH_AUTO):
    info = PlanInfo()
    st = load().ggrn_plan(y, gate, w, out, rows, width, group_size, y_row_stride,
                          gate_row_stride, out_row_stride, dtype, mode, path, ctypes.byref(info))
    return st, info


# ---------------------------------------------------------------------------
# Tensor-level API.
# ---------------------------------------------------------------------------
def _as_rows(t: torch.Tensor, width: int, name: str) -> tuple[int, int]:
    """(rows, row_stride) of a tensor viewed as [rows, width] with unit inner stride."""
    if t.dim() == 0:
        raise ValueError(f"{name} must have rank >= 1")
    if t.shape[-1] != width:
        raise ValueError(f"{name}: last dimension {t.shape[-1]} != width {width}")
    if t.numel() == 0:
        return 0, width
    if t.stride(-1) != 1:
        raise ValueError(f"{name} needs unit stride on its last dimension")
    if t.dim() == 1:
        return 1, width
    lead = t.shape[:-1]
    rows = 1
    for s in lead:
        rows *= s
    # leading axes must fold into one uniformly strided row axis
    stride = t.stride(-2)
    expect = stride
    for d in range(t.dim() - 2, -1, -1):
        if t.shape[d] != 1 and t.stride(d) != expect:
            raise ValueError(f"{name}: leading axes do not fold into one row axis")
        expect *= t.shape[d]
    return rows, (stride if rows > 1 else width)


def _stream_handle(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def plan(y: torch.Tensor, gate: torch.Tensor, w: torch.Tensor, *, group_size: int,
         mode="mamba2", out: torch.Tensor | None = None, path: int = PATH_AUTO) -> dict:
    """The launch ``forward`` would make (host only)."""
    width = y.shape[-1]
    rows, ys = _as_rows(y, width, "y")
    _, gts = _as_rows(gate, width, "gate")
    os_ = width
    optr = 0
    if out is not None:
        _, os_ = _as_rows(out, width, "out")
        optr = out.data_ptr()
    st, info = ggrn_plan(y.data_ptr(), gate.data_ptr(), w.data_ptr(), optr, rows, width,
                         group_size, ys, gts, os_, DTYPE_CODE[y.dtype], MODE_CODE[mode], path)
    if st != OK:
        raise GgrnError(st, "ggrn_plan")
    return info.as_dict()


def forward(y: torch.Tensor, gate: torch.Tensor, w: torch.Tensor, *, group_size: int,
            eps: float, mode="mamba2", out: torch.Tensor | None = None,
            path: int = PATH_AUTO) -> torch.Tensor:
    """Fused gated group-RMSNorm on CUDA tensors, enqueued on the current stream.

    ``y``, ``gate``: [..., width] tensors of T (f32, f16, bf16; ONNX: f32, f16)
    whose leading axes fold into rows (row-strided views allowed).
    ``w``: MAMBA2 -> f32 [width]; ONNX -> T scale with ``group_size`` elements
    (any of the shapes (C), (1, C), (C, 1)).
    ``out``: optional output (same shape as y; allocated like y when omitted).
    """
    if not y.is_cuda:
        raise ValueError("forward runs on CUDA tensors only (no CPU path)")
    m = MODE_CODE[mode]
    width = y.shape[-1]
    if gate.shape != y.shape:
        raise ValueError("gate must have the shape of y")
    if gate.dtype != y.dtype:
        raise ValueError("gate must have the dtype of y")
    w = _weight(w, m, width, group_size, y.dtype)
    if out is None:
        out = torch.empty(y.shape, dtype=y.dtype, device=y.device)
    elif out.shape != y.shape or out.dtype != y.dtype:
        raise ValueError("out must have the shape and dtype of y")
    rows, ys = _as_rows(y, width, "y")
    _, gts = _as_rows(gate, width, "gate")
    _, os_ = _as_rows(out, width, "out")
    if y.dtype not in DTYPE_CODE:
        raise ValueError(f"unsupported dtype {y.dtype}")
    st = ggrn_forward_path(y.data_ptr(), gate.data_ptr(), w.data_ptr(), out.data_ptr(), rows,
                           width, group_size, ys, gts, os_, float(eps), DTYPE_CODE[y.dtype], m,
                           path, _stream_handle(y.device))
    if st != OK:
        raise GgrnError(st, "ggrn_forward")
    return out


def _weight(w: torch.Tensor, m: int, width: int, group_size: int, dtype) -> torch.Tensor:
    if m == MAMBA2 and (w.dtype != torch.float32 or w.numel() != width):
        raise ValueError("MAMBA2 weight is float32 with `width` elements")
    if m == ONNX:
        if w.dtype != dtype or w.numel() != group_size:
            raise ValueError("ONNX scale has the dtype of X and group_size elements")
        w = w.reshape(-1)
    return w if w.is_contiguous() else w.contiguous()


def forward_inproj(inproj: torch.Tensor, w: torch.Tensor, *, width: int, y_col: int,
                   gate_col: int, group_size: int, eps: float, mode="mamba2",
                   out: torch.Tensor | None = None) -> torch.Tensor:
    """The operation on y = inproj[..., y_col:y_col+width] and gate =
    inproj[..., gate_col:gate_col+width], read in place from the packed
    output of a fused input projection (``ggrn_forward_inproj``).

    ``inproj``: [..., inproj_width] tensor of T with unit inner stride whose
    leading axes fold into rows.  ``out``: optional [..., width] output
    (allocated contiguous when omitted).
    """
    if not inproj.is_cuda:
        raise ValueError("forward_inproj runs on CUDA tensors only (no CPU path)")
    m = MODE_CODE[mode]
    if inproj.dtype not in DTYPE_CODE:
        raise ValueError(f"unsupported dtype {inproj.dtype}")
    ipw = inproj.shape[-1]
    rows, ips = _as_rows(inproj, ipw, "inproj")
    w = _weight(w, m, width, group_size, inproj.dtype)
    shape = tuple(inproj.shape[:-1]) + (width,)
    if out is None:
        out = torch.empty(shape, dtype=inproj.dtype, device=inproj.device)
    elif tuple(out.shape) != shape or out.dtype != inproj.dtype:
        raise ValueError("out must have the leading shape of inproj, width columns and its dtype")
    _, os_ = _as_rows(out, width, "out")
    st = ggrn_forward_inproj(inproj.data_ptr(), ips, y_col, gate_col, w.data_ptr(), out.data_ptr(),
                             os_, rows, width, group_size, float(eps), DTYPE_CODE[inproj.dtype], m,
                             _stream_handle(inproj.device))
    if st != OK:
        raise GgrnError(st, "ggrn_forward_inproj")
    return out


def host_workspace(rows: int, width: int, dtype, device) -> torch.Tensor:
    """A device workspace of the size ggrn_forward_host wants for full chunks."""
    n = load().ggrn_host_workspace_bytes(rows, width, DTYPE_CODE[dtype])
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device)


def forward_host(y: torch.Tensor, gate: torch.Tensor, w: torch.Tensor, *, group_size: int,
                 eps: float, mode="mamba2", out: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None) -> torch.Tensor:
    """The operation on CPU tensors (``ggrn_forward_host``), enqueued on the
    current stream of ``w``'s device.  Pinned y, gate and out are read and
    written in place by the kernel over the host link; other host memory is
    staged through a device workspace with the copies overlapped.

    ``y``, ``gate``: CPU [..., width] tensors.  ``w``: the weight / scale on
    the GPU.  ``out``: optional CPU output (allocated pinned when omitted).
    ``workspace``: optional device uint8 tensor for the copy route
    (``host_workspace`` when omitted and needed).  The result is complete
    when the stream reaches this point (synchronise before reading it).
    """
    if y.is_cuda or gate.is_cuda:
        raise ValueError("forward_host takes y and gate in host memory")
    if not w.is_cuda:
        raise ValueError("the weight lives on the GPU")
    m = MODE_CODE[mode]
    width = y.shape[-1]
    if gate.shape != y.shape or gate.dtype != y.dtype:
        raise ValueError("gate must have the shape and dtype of y")
    if y.dtype not in DTYPE_CODE:
        raise ValueError(f"unsupported dtype {y.dtype}")
    w = _weight(w, m, width, group_size, y.dtype)
    if out is None:
        out = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    elif out.is_cuda or out.shape != y.shape or out.dtype != y.dtype:
        raise ValueError("out must be a host tensor with the shape and dtype of y")
    rows, ys = _as_rows(y, width, "y")
    _, gts = _as_rows(gate, width, "gate")
    _, os_ = _as_rows(out, width, "out")
    if workspace is None and not (y.is_pinned() and gate.is_pinned() and out.is_pinned()):
        workspace = host_workspace(rows, width, y.dtype, w.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    packed = _packed_pair(y, gate, rows, width, ys, gts)
    with torch.cuda.device(w.device):
        if packed is not None:
            # y and gate are column ranges of one tensor's rows: declared as
            # one packed matrix (the copy route may then move both at once)
            base, ycol, gcol = packed
            st = ggrn_forward_inproj_host(base, ys, ycol, gcol, w.data_ptr(), out.data_ptr(),
                                          os_, rows, width, group_size, float(eps),
                                          DTYPE_CODE[y.dtype], m, ws_ptr, ws_bytes,
                                          _stream_handle(w.device))
        else:
            st = ggrn_forward_host(y.data_ptr(), gate.data_ptr(), w.data_ptr(), out.data_ptr(),
                                   rows, width, group_size, ys, gts, os_, float(eps),
                                   DTYPE_CODE[y.dtype], m, ws_ptr, ws_bytes,
                                   _stream_handle(w.device))
    if st != OK:
        raise GgrnError(st, "ggrn_forward_host")
    return out


def ggrn_norm_outproj(y, gate, w, w_out, z, rows, width, group_size, y_row_stride,
                      gate_row_stride, d_model, eps, workspace, workspace_bytes, a_out,
                      stream) -> int:
    return load().ggrn_norm_outproj(y, gate, w, w_out, z, rows, width, group_size, y_row_stride,
                                    gate_row_stride, d_model, eps, workspace, workspace_bytes,
                                    a_out, stream)


def norm_outproj(y: torch.Tensor, gate: torch.Tensor, w: torch.Tensor, w_out: torch.Tensor, *,
                 group_size: int, eps: float, out: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None,
                 a_out: torch.Tensor | None = None) -> torch.Tensor:
    """The Mamba-2 norm fused into the out_proj GEMM (``ggrn_norm_outproj``):
    ``out = norm(y, gate, w) @ w_out.T`` in bf16 with f32 sums, the norm's
    output never written unless ``a_out`` (a [rows, width] bf16 tensor) is
    given.  ``y``, ``gate``: bf16 CUDA [..., width] (row-strided views
    allowed); ``w``: f32 [width]; ``w_out``: bf16 [d_model, width]
    contiguous.  Enqueued on the current stream."""
    if not (y.is_cuda and gate.is_cuda and w.is_cuda and w_out.is_cuda):
        raise ValueError("norm_outproj takes CUDA tensors")
    if y.dtype != torch.bfloat16 or gate.dtype != torch.bfloat16 or w_out.dtype != torch.bfloat16:
        raise ValueError("norm_outproj takes bf16 y, gate and w_out")
    width = y.shape[-1]
    rows, ys = _as_rows(y, width, "y")
    _, gts = _as_rows(gate, width, "gate")
    w = w.reshape(width).to(torch.float32).contiguous()
    if w_out.dim() != 2 or w_out.shape[1] != width or not w_out.is_contiguous():
        raise ValueError("w_out must be a contiguous [d_model, width] tensor")
    d_model = w_out.shape[0]
    if out is None:
        out = torch.empty(y.shape[:-1] + (d_model,), dtype=torch.bfloat16, device=y.device)
    if workspace is None:
        nbytes = load().ggrn_norm_outproj_workspace_bytes(rows, width, group_size)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=y.device)
    st = ggrn_norm_outproj(y.data_ptr(), gate.data_ptr(), w.data_ptr(), w_out.data_ptr(),
                           out.data_ptr(), rows, width, group_size, ys, gts, d_model, float(eps),
                           workspace.data_ptr(), workspace.numel(),
                           a_out.data_ptr() if a_out is not None else None,
                           _stream_handle(y.device))
    if st != OK:
        raise GgrnError(st, "ggrn_norm_outproj")
    return out


def _packed_pair(y, gate, rows, width, ys, gts):
    """(base pointer, y column, gate column) when y and gate are two column
    ranges of the same rows of one tensor's storage, which holds every row
    from the earlier range's first column to the later range's last one;
    else None."""
    if rows < 2 or ys != gts:
        return None
    if y.untyped_storage().data_ptr() != gate.untyped_storage().data_ptr():
        return None
    es = y.element_size()
    yp, gp = y.data_ptr(), gate.data_ptr()
    base = min(yp, gp)
    ycol, gcol = (yp - base) // es, (gp - base) // es
    if (yp - base) % es or (gp - base) % es or max(ycol, gcol) + width > ys:
        return None
    st0 = y.untyped_storage().data_ptr()
    end = base + ((rows - 1) * ys + max(ycol, gcol) + width) * es
    if base < st0 or end > st0 + y.untyped_storage().nbytes():
        return None
    return base, ycol, gcol


class DecodeGraph:
    """A chain of calls captured once into a CUDA graph and replayed with one launch.

    ``calls``: list of dicts with the tensors and arguments of ``forward``
    (``y``, ``gate``, ``w``, ``out``, ``group_size``, ``eps``, ``mode``).  The
    tensors are baked into the graph: keep them alive and refill them in
    place between replays.  A chain of one call is launched directly on each
    replay (a graph of one small kernel costs more to launch than the kernel).
    """

    def __init__(self, calls: list[dict]):
        arr = (Call * len(calls))()
        self._keep = []
        for i, c in enumerate(calls):
            y, gate, w, out = c["y"], c["gate"], c["w"], c["out"]
            width = y.shape[-1]
            rows, ys = _as_rows(y, width, "y")
            _, gts = _as_rows(gate, width, "gate")
            _, os_ = _as_rows(out, width, "out")
            arr[i] = Call(y.data_ptr(), gate.data_ptr(), w.data_ptr(), out.data_ptr(), rows, width,
                          c["group_size"], ys, gts, os_, float(c["eps"]), DTYPE_CODE[y.dtype],
                          MODE_CODE[c.get("mode", "mamba2")])
            self._keep.extend([y, gate, w, out])
        self._handle = ctypes.c_void_p()
        st = load().ggrn_graph_create(arr, len(calls), ctypes.byref(self._handle))
        if st != OK:
            raise GgrnError(st, "ggrn_graph_create")
        self.device = calls[0]["y"].device

    def replay(self, stream: torch.cuda.Stream | None = None) -> None:
        s = stream.cuda_stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        st = load().ggrn_graph_launch(self._handle, ctypes.c_void_p(s))
        if st != OK:
            raise GgrnError(st, "ggrn_graph_launch")

    def close(self) -> None:
        if self._handle:
            load().ggrn_graph_destroy(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
