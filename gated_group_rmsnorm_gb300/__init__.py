"""GB300 (sm_103a) fused gated group-RMSNorm.

The operation ("gated_group_rmsnorm" Mojo module page, math block; and
"com.microsoft.GatedRMSNorm" README, Description): for every row and every
contiguous group of ``group_size`` columns,

  mamba2: out = cast(w[col] * cast(y*silu(gate) * rsqrt(mean((y*silu(gate))^2) + eps)))
  onnx:   out = cast(x * rsqrt(mean(x^2) + eps) * scale[j] * silu(gate))

computed by hand-written CUDA kernels behind a C ABI (``include/ggrn.h``,
``libggrn.so``).  This package is the thin Python binding.
"""
from .binding import (BF16, DTYPE_CODE, F16, F32, MAMBA2, ONNX, PATH_AUTO, PATH_NAMES,
                      PATH_SCALAR, PATH_STRADDLE, PATH_STREAM, PATH_TEAM, PATH_WIDE,
                      PATH_WIDE_CLUSTER, DecodeGraph,
                      GgrnError, fault_status, forward, forward_host, forward_inproj,
                      ggrn_forward, ggrn_forward_host, ggrn_forward_inproj,
                      ggrn_forward_inproj_host, ggrn_forward_noalloc, ggrn_forward_path,
                      ggrn_norm_outproj, norm_outproj, ggrn_plan, host_workspace, library_path, load, plan,
                      status_string)

__all__ = ["forward", "forward_host", "forward_inproj", "plan", "DecodeGraph", "GgrnError",
           "ggrn_forward", "ggrn_forward_host", "ggrn_forward_inproj", "ggrn_forward_inproj_host",
           "ggrn_forward_noalloc", "ggrn_norm_outproj", "norm_outproj",
           "ggrn_forward_path", "ggrn_plan", "host_workspace", "load",
           "library_path", "status_string", "MAMBA2", "ONNX", "F32", "F16", "BF16", "PATH_AUTO", "PATH_TEAM", "PATH_WIDE", "PATH_STRADDLE", "PATH_SCALAR",
           "PATH_STREAM", "PATH_WIDE_CLUSTER", "PATH_NAMES", "DTYPE_CODE", "fault_status"]
