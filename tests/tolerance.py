"""Comparison rules for the fused gated group-RMSNorm.

Floating-point bar (set by the workload statement of this library): every
16-bit output element within 1 ulp of T of the oracle's f32-accumulated
result, cast-boundary flips from a different summation order allowed; f32
outputs within 1e-5 relative.

The Mamba-2 semantics cast twice (t = cast_T(gated*nf), then
out = cast_T(w*t)).  A different summation order moves m2 by an f32 ulp or so;
when gated*nf then sits next to a T rounding midpoint, t flips by one T ulp,
and the second rounding can turn that into 2 ulps of out.  The flip-aware rule
accepts an element when it is within 1 ulp of the oracle's out, OR within 1
ulp of cast_T(w * t') with t' a T-neighbour of the oracle's t.  The ONNX
semantics round once, so 1 ulp is the whole rule there.
"""
from __future__ import annotations

import torch

F32_RTOL = 1e-5
F32_ATOL = 1e-30


def ordinal(t: torch.Tensor) -> torch.Tensor:
    """Monotone integer image of a float tensor; +0 and -0 both map to 0."""
    t = t.contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        u = t.view(torch.int16).to(torch.int64) & 0xFFFF
        mag = u & 0x7FFF
        neg = (u & 0x8000) != 0
    elif t.dtype == torch.float32:
        u = t.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
        mag = u & 0x7FFFFFFF
        neg = (u & 0x80000000) != 0
    else:
        raise TypeError(t.dtype)
    return torch.where(neg, -mag, mag)


def from_ordinal(o: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    if dtype in (torch.bfloat16, torch.float16):
        bits = torch.where(o < 0, (-o) | 0x8000, o).to(torch.int32)
        bits = torch.where(bits >= 0x8000, bits - 0x10000, bits).to(torch.int16)
        return bits.view(dtype)
    bits = torch.where(o < 0, (-o) | 0x80000000, o)
    bits = torch.where(bits >= 0x80000000, bits - 0x100000000, bits).to(torch.int32)
    return bits.view(torch.float32)


def ulp_dist(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    """|ordinal(a) - ordinal(b)|; NaN vs NaN counts 0, NaN vs number a large value."""
    assert a.dtype == b.dtype and a.shape == b.shape
    d = (ordinal(a) - ordinal(b)).abs()
    an, bn = torch.isnan(a.float()), torch.isnan(b.float())
    d = torch.where(an & bn, torch.zeros_like(d), d)
    d = torch.where(an ^ bn, torch.full_like(d, 1 << 40), d)
    return d


def neighbours(t: torch.Tensor):
    o = ordinal(t)
    return from_ordinal(o + 1, t.dtype), from_ordinal(o - 1, t.dtype)


def mamba2_accept(got: torch.Tensor, ref: torch.Tensor, ref_t: torch.Tensor,
                  w_cols: torch.Tensor) -> torch.Tensor:
    """Per-element acceptance (bool tensor) for 16-bit T under Mamba-2 semantics.

    ``w_cols``: f32 weight broadcast to ``ref``'s shape (w[col] per element).
    """
    ok = ulp_dist(got, ref) <= 1
    for tn in neighbours(ref_t):
        alt = (w_cols.float() * tn.float()).to(ref.dtype)
        ok |= ulp_dist(got, alt) <= 1
    return ok


def f32_accept(got: torch.Tensor, ref: torch.Tensor, rtol: float = F32_RTOL,
               atol: float = F32_ATOL) -> torch.Tensor:
    g, r = got.double(), ref.double()
    ok = (g - r).abs() <= rtol * r.abs() + atol
    both_nan = torch.isnan(g) & torch.isnan(r)
    same_inf = torch.isinf(g) & torch.isinf(r) & (torch.sign(g) == torch.sign(r))
    return ok | both_nan | same_inf


def check(got: torch.Tensor, ref: torch.Tensor, *, mode: int, ref_t: torch.Tensor | None = None,
          w_cols: torch.Tensor | None = None) -> dict:
    """Apply the rule for ``mode`` (0 Mamba-2, 1 ONNX); return a summary dict.

    The summary has ``ok`` (all accepted), ``bad`` (rejected count),
    ``over1`` (raw count of elements more than 1 ulp from the oracle's out),
    ``max_ulp`` and ``n``.
    """
    got = got.cpu()
    ref = ref.cpu()
    if ref.dtype == torch.float32:
        acc = f32_accept(got, ref)
        over1 = int((~acc).sum())
        max_ulp = int(ulp_dist(got, ref).max()) if ref.numel() else 0
    else:
        d = ulp_dist(got, ref)
        over1 = int((d > 1).sum())
        max_ulp = int(d.max()) if ref.numel() else 0
        if mode == 0:
            assert ref_t is not None and w_cols is not None
            acc = mamba2_accept(got, ref, ref_t.cpu(), w_cols.cpu())
        else:
            acc = d <= 1
    bad = int((~acc).sum())
    return {"ok": bad == 0, "bad": bad, "over1": over1, "max_ulp": max_ulp, "n": ref.numel()}


def weight_cols(w: torch.Tensor, rows: int, width: int) -> torch.Tensor:
    """Mamba-2 weight (f32, length width) broadcast to [rows, width]."""
    return w.float().reshape(1, width).expand(rows, width)
