"""Comparison rules for the fused gated group-RMSNorm.

Floating-point bar (set by the workload statement of this library): every
16-bit output element within 1 ulp of T of the oracle's f32-accumulated
result, cast-boundary flips from a different summation order allowed; f32
outputs within 1e-5 relative.

What a correct GPU result can differ in.  The GPU sums the squares of a group
in another order than the oracle's sequential sum, and computes silu and the
reciprocal square root with the hardware's approximate instructions, so its
value of each element just before a rounding to T (``pre``: gated*nf for the
Mamba-2 intermediate cast, the full product for the ONNX store) differs from
the oracle's by a small relative amount.  Every other step is the same IEEE
operation on both sides (the f32 product w*t of the Mamba-2 epilogue, the
round-to-nearest-even casts).  So an output element can differ from the
oracle's only through a *flip*: ``pre`` lies so close to a rounding midpoint
of T that the two sides round it to neighbouring T values.

  * Mamba-2 ("gated_group_rmsnorm" page, math block): t = cast_T(gated*nf)
    flips to its neighbour t' on the side of the nearer midpoint, and then
    out = cast_T(w*t') exactly (one f32 multiply, one rounding), which can be
    2 ulps from the oracle's out.
  * ONNX ("com.microsoft.GatedRMSNorm" README, Description): one rounding, so
    the flipped output is the oracle's out's neighbour on that side.

A flip is *explained* when the element equals that flipped value bit for bit
AND the oracle's ``pre`` lies within ``tau * |pre|`` of the midpoint, where
tau bounds the relative difference of the two sides' ``pre``.  With u = 2^-24
(half an f32 ulp, relative), n the group size and b the gate values:

  Mamba-2  tau_j = (n + |b_j| + max_k |b_k| + 48) u   (k over the group)
  ONNX     tau_j = (n + |b_j| + 48) u

from: any two orders of a sum of n non-negative terms differ by at most
2(n-1)u relative, halved by the square root; silu's base-2 exponential takes
an argument rounded by u relative, an absolute error of |b|u in the exponent
(|b| counted up to 89, beyond which both sides saturate exactly), plus a few
u for the approximate exponential and reciprocal; a few u for the divide, the
eps add, the approximate rsqrt (budgeted 8u) and the products.

Rules applied (``check``):
  ``ok``           the stated bar: each element within 1 ulp of the oracle's,
                   or an explained Mamba-2 flip (which may be 2 ulps away);
  ``unexplained``  elements that differ from the oracle's and are not an
                   explained flip -- zero for a correct kernel, asserted by
                   ``assert_parity``;
  ``over1``        elements more than 1 ulp away (all of them explained
                   flips); ``flips`` and ``over1`` are bounded (below).

The rates.  A flip needs ``pre`` within the two sides' actual difference of
a midpoint; that difference grows like the square root of the group size
(rounding errors of a sum add up like a random walk) plus a few u, and the
midpoints sit one T ulp apart (2^-8 relative for bf16, 2^-11 for fp16, at
the least), so the expected share of flipped elements is about
(sqrt(n) + 8) u / ulp_T.  That is the bound (``flip_bound``), plus a floor of
four elements; at most 35 % of the bound may be more than 1 ulp away.  On
GB300 every full-size workload came in 4 to 18 times below it (flips per
element: 960-wide bf16 groups 3.3e-5, 5120-wide 1.2e-4, 100-wide 1.5e-5,
128-wide fp16 1.3e-4; >1 ulp: 7 to 14 % of the flips).
"""
from __future__ import annotations

import torch

F32_RTOL = 1e-5
F32_ATOL = 1e-30
U = 2.0 ** -24
TAU_CONST = 48.0
SILU_ARG_CAP = 89.0
ULP_REL = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
OVER1_SHARE = 0.35


def flip_bound(n_elems: int, group_size: int, dtype: torch.dtype) -> float:
    """Most flips a correct kernel may show over ``n_elems`` elements."""
    if dtype not in ULP_REL:
        return 0.0
    return (group_size ** 0.5 + 8.0) * U / ULP_REL[dtype] * n_elems + 4.0


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


def flip_target(t: torch.Tensor, pre: torch.Tensor, tau: torch.Tensor):
    """For each element: the T neighbour t' of ``t`` on the side of ``pre``
    (the value the other side's rounding gives if it flips), and whether
    ``pre`` lies within ``tau * |pre|`` of the midpoint between t and t'."""
    p = pre.double()
    tv = t.double()
    up, down = neighbours(t)
    toward_up = p >= tv
    tn = torch.where(toward_up, up, down)
    tnv = tn.double()
    # a neighbour past the largest finite value: the midpoint is half a
    # spacing beyond t, the spacing of t's own binade
    other = torch.where(toward_up, down, up).double()
    spacing = torch.where(torch.isfinite(tnv), (tnv - tv).abs(), (tv - other).abs())
    mid = tv + torch.where(toward_up, 0.5, -0.5) * spacing
    near = (p - mid).abs() <= tau * p.abs()
    near &= torch.isfinite(p) & torch.isfinite(tv)
    return tn, near


def mamba2_accept(got: torch.Tensor, ref: torch.Tensor, ref_t: torch.Tensor,
                  w_cols: torch.Tensor, pre: torch.Tensor, tau: torch.Tensor):
    """Per-element (accepted, explained flip) for 16-bit T under Mamba-2
    semantics.  ``w_cols``: f32 weight broadcast to ``ref``'s shape."""
    tn, near = flip_target(ref_t, pre, tau)
    alt = (w_cols.float() * tn.float()).to(ref.dtype)
    flip = near & (ulp_dist(got, alt) == 0)
    return (ulp_dist(got, ref) <= 1) | flip, flip


def onnx_flip(got: torch.Tensor, ref: torch.Tensor, pre: torch.Tensor,
              tau: torch.Tensor) -> torch.Tensor:
    """Explained flips of the single ONNX rounding."""
    tn, near = flip_target(ref, pre, tau)
    return near & (ulp_dist(got, tn) == 0)


def mamba2_flip_mask(ref_t: torch.Tensor, pre: torch.Tensor, gate: torch.Tensor,
                     group_size: int) -> torch.Tensor:
    """Elements whose Mamba-2 intermediate t may flip on a correct kernel
    (``pre`` within tau of a rounding midpoint, tau as in ``check``): the only
    elements of a correct kernel's output that may differ from the oracle's."""
    rows, width = ref_t.shape
    b = gate.double().abs().clamp(max=SILU_ARG_CAP)
    b = torch.where(torch.isnan(b), torch.full_like(b, SILU_ARG_CAP), b)
    bmax = b.reshape(rows, width // group_size, group_size).amax(-1, keepdim=True)
    tau = ((group_size + TAU_CONST) + b +
           bmax.expand(rows, width // group_size, group_size).reshape(rows, width)) * U
    _, near = flip_target(ref_t, pre, tau)
    return near


def f32_accept(got: torch.Tensor, ref: torch.Tensor, rtol: float = F32_RTOL,
               atol: float = F32_ATOL) -> torch.Tensor:
    g, r = got.double(), ref.double()
    ok = (g - r).abs() <= rtol * r.abs() + atol
    both_nan = torch.isnan(g) & torch.isnan(r)
    same_inf = torch.isinf(g) & torch.isinf(r) & (torch.sign(g) == torch.sign(r))
    return ok | both_nan | same_inf


def check(got: torch.Tensor, ref: torch.Tensor, *, mode: int, ref_t: torch.Tensor | None = None,
          w_cols: torch.Tensor | None = None, pre: torch.Tensor | None = None,
          gate: torch.Tensor | None = None, group_size: int | None = None) -> dict:
    """Apply the rules for ``mode`` (0 Mamba-2, 1 ONNX); return a summary dict
    with ``ok``, ``bad`` (rejected by the stated bar), ``unexplained``,
    ``flips``, ``over1``, ``max_ulp``, ``same`` (equal by value) and ``n``.

    16-bit T needs the oracle's ``pre`` and the ``gate`` values (for tau) and
    ``group_size``; Mamba-2 also ``ref_t`` and ``w_cols``.  The rules are
    evaluated on the elements whose bits differ (equal bits are equal values).
    """
    got = got.cpu()
    ref = ref.cpu()
    n = ref.numel()
    if ref.dtype == torch.float32:
        acc = f32_accept(got, ref)
        bad = int((~acc).sum())
        d = ulp_dist(got, ref)
        return {"ok": bad == 0, "bad": bad, "unexplained": bad, "flips": 0, "over1": bad,
                "max_ulp": int(d.max()) if n else 0, "same": int((d == 0).sum()), "n": n,
                "flip_bound": 0.0}
    assert pre is not None and gate is not None and group_size is not None
    assert got.shape == ref.shape and ref.dim() == 2
    rows, width = ref.shape
    idx = torch.nonzero((got.contiguous().view(torch.int16) != ref.contiguous().view(torch.int16))
                        .view(-1)).view(-1)
    fb = flip_bound(n, group_size, ref.dtype)
    if idx.numel() == 0:
        return {"ok": True, "bad": 0, "unexplained": 0, "flips": 0, "over1": 0, "max_ulp": 0,
                "same": n, "n": n, "flip_bound": fb}
    g1, r1 = got.reshape(-1)[idx], ref.reshape(-1)[idx]
    d = ulp_dist(g1, r1)
    # tau of the differing elements: their own gate value and (Mamba-2) the
    # largest |gate| of their group
    b = gate.cpu().double().abs().clamp(max=SILU_ARG_CAP)
    b = torch.where(torch.isnan(b), torch.full_like(b, SILU_ARG_CAP), b)
    tau = (group_size + TAU_CONST) + b.reshape(-1)[idx]
    if mode == 0:
        bmax = b.reshape(rows * (width // group_size), group_size).amax(-1)
        tau = tau + bmax[idx // group_size]
    tau = tau * U
    p1 = pre.cpu().reshape(-1)[idx]
    if mode == 0:
        assert ref_t is not None and w_cols is not None
        t1 = ref_t.cpu().reshape(-1)[idx]
        wc = w_cols.cpu().reshape(-1)[idx] if w_cols.is_contiguous() else \
            w_cols.cpu().contiguous().reshape(-1)[idx]
        acc, flip = mamba2_accept(g1, r1, t1, wc, p1, tau)
    else:
        flip = onnx_flip(g1, r1, p1, tau)
        acc = d <= 1
    differ = d != 0   # bits differ but values may be equal (+0 / -0, two NaNs)
    bad = int((~acc).sum())
    return {"ok": bad == 0, "bad": bad,
            "unexplained": int((differ & ~flip).sum()),
            "flips": int((differ & flip).sum()),
            "over1": int((d > 1).sum()),
            "max_ulp": int(d.max()),
            "same": n - int(differ.sum()), "n": n, "flip_bound": fb}


def merge(results: list[dict]) -> dict:
    """Sum the counts of several ``check`` summaries (blocks of one output)."""
    out = {"ok": all(r["ok"] for r in results)}
    for k in ("bad", "unexplained", "flips", "over1", "same", "n"):
        out[k] = sum(r[k] for r in results)
    # one bound over all the blocks (the floor counted once)
    out["flip_bound"] = sum(max(r["flip_bound"] - 4.0, 0.0) for r in results) + 4.0
    out["max_ulp"] = max((r["max_ulp"] for r in results), default=0)
    return out


def parity_ok(res: dict) -> bool:
    """The stated bar, no unexplained difference, flips within ``flip_bound``
    and at most ``OVER1_SHARE`` of that bound more than 1 ulp away."""
    fb = res["flip_bound"]
    return (res["ok"] and res["unexplained"] == 0 and res["flips"] <= fb
            and res["over1"] <= OVER1_SHARE * fb)


def assert_parity(res: dict, what="") -> None:
    assert parity_ok(res), (what, res)


def weight_cols(w: torch.Tensor, rows: int, width: int) -> torch.Tensor:
    """Mamba-2 weight (f32, length width) broadcast to [rows, width]."""
    return w.float().reshape(1, width).expand(rows, width)
