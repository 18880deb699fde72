"""Pins of the CPU oracle to facts outside the oracle itself.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with the fact.  ``tests/test_oracle_pins.py`` runs every pin
against the real oracle; ``tests/test_oracle_mutants.py`` runs them against
copies of the oracle with planted mistakes and requires each copy to fail at
least one pin.

What pins what (definitions: "gated_group_rmsnorm" Mojo module page, math
block; "com.microsoft.GatedRMSNorm" README, Description and Type constraints):
  golden       hand-worked values with derivations (tests/golden/*.txt)
  codec        T <-> f32 conversion vs torch's RNE conversions, every 16-bit
               pattern and edge values
  rms_norm     large-gate limit: silu(32) = 32 exactly, so Mamba-2 with
               gate = 32 is a plain group RMSNorm of y (library special case,
               torch.nn.functional.rms_norm in f64), weight indexed by column;
               ONNX with gate = 32 is 32 * rms_norm(X) * scale[j]
  silu         ONNX, C = 1, X = 1, scale = 1, eps = 0 reduces to silu(gate)
               (torch.nn.functional.silu in f64)
  brute        double-precision twin on every tiny shape (the flip-aware rule)
  invariants   group independence, power-of-two scale invariance (eps = 0),
               zero gate, permutation within a group, ONNX gate separability,
               strided views equal contiguous copies
"""
from __future__ import annotations

import torch

import ggrn_inputs
from tests import golden_cases
from tests.tolerance import check, f32_accept, ulp_dist, weight_cols

MAMBA2, ONNX = 0, 1
DTYPES = (torch.bfloat16, torch.float16, torch.float32)


def _val_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Equal by value (-0 == +0), NaN == NaN."""
    a, b = a.double(), b.double()
    return bool(((a == b) | (torch.isnan(a) & torch.isnan(b))).all())


# --------------------------------------------------------------------------
def pin_golden(orc) -> None:
    cases = golden_cases.load_all()
    assert len(cases) >= 10
    for c in cases:
        out = orc.forward(c.y, c.gate, c.w, group_size=c.group_size, eps=c.eps, mode=c.mode)
        assert _val_equal(out, c.expect), (
            f"{c.source}:{c.name}: got {out.double().tolist()} expected {c.expect.double().tolist()}")


# --------------------------------------------------------------------------
def _special_f32() -> torch.Tensor:
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e30, -1e30,
            float("inf"), float("-inf"), 2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001,
            2.0 ** -26, 3.0 * 2.0 ** -26, 2.0 ** -15 * 1.5, 1e-40, -1e-40, 3.3895e38, 3.39e38,
            3.4e38, 5.9604645e-08, 6.1035156e-05, 1.00048828125, 1.000732421875, 1.0009765625]
    return torch.tensor(vals, dtype=torch.float32)


def _tie_f32(dtype: torch.dtype, n: int, gen: torch.Generator) -> torch.Tensor:
    """f32 values exactly halfway between two T values (exercise ties-to-even)."""
    if dtype == torch.bfloat16:
        hi = torch.randint(0, 0x7F7F, (n,), generator=gen, dtype=torch.int64)
        bits = (hi << 16) | 0x8000
    else:  # fp16 normal range: exponent 1..30 -> f32 exponent 113..142; 13 dropped bits
        e = torch.randint(113, 143, (n,), generator=gen, dtype=torch.int64)
        m = torch.randint(0, 1 << 10, (n,), generator=gen, dtype=torch.int64)
        bits = (e << 23) | (m << 13) | 0x1000
    sign = torch.randint(0, 2, (n,), generator=gen, dtype=torch.int64) << 31
    bits = bits | sign
    bits = torch.where(bits >= 2 ** 31, bits - 2 ** 32, bits).to(torch.int32)
    return bits.view(torch.float32)


def pin_codec(orc) -> None:
    gen = torch.Generator().manual_seed(1234)
    for dtype in (torch.bfloat16, torch.float16):
        # decode: all 65536 patterns
        pats = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(dtype)
        got = orc.decode(pats)
        ref = pats.float()
        nan_ok = torch.isnan(got) == torch.isnan(ref)
        assert bool(nan_ok.all()), f"{dtype}: decode NaN mismatch"
        fin = ~torch.isnan(ref)
        assert torch.equal(got[fin].view(torch.int32), ref[fin].view(torch.int32)), f"{dtype}: decode"
        # encode: random magnitudes, ties, specials
        xs = [torch.randn(20000, generator=gen) * (10.0 ** torch.randint(-9, 6, (20000,), generator=gen)),
              _tie_f32(dtype, 20000, gen), _special_f32(),
              (torch.rand(5000, generator=gen) * 2 ** -13) * torch.sign(torch.randn(5000, generator=gen))]
        x = torch.cat(xs)
        got = orc.encode(x, dtype)
        ref = x.to(dtype)
        gn, rn = torch.isnan(got.float()), torch.isnan(ref.float())
        assert bool((gn == rn).all()), f"{dtype}: encode NaN"
        gb = got.view(torch.int16)[~rn]
        rb = ref.view(torch.int16)[~rn]
        bad = (gb != rb).nonzero()
        assert bad.numel() == 0, (
            f"{dtype}: encode differs from torch at {x[~rn][bad[:5, 0]].tolist()}")
        # NaN stays NaN and quiet
        nan_in = torch.tensor([float("nan"), -float("nan")])
        assert bool(torch.isnan(orc.encode(nan_in, dtype).float()).all())


# --------------------------------------------------------------------------
def pin_rms_norm(orc) -> None:
    """Large-gate limit: silu(32) == 32 in f32, so the gate is a constant factor."""
    F = torch.nn.functional
    gen = torch.Generator().manual_seed(7)
    for (rows, width, gs) in ((3, 12, 4), (2, 21, 7), (4, 64, 64), (2, 40, 1), (5, 30, 10)):
        groups = width // gs
        y = torch.randn(rows, width, generator=gen, dtype=torch.float32)
        gate = torch.full((rows, width), 32.0)
        w = 1.0 + 0.1 * torch.randn(width, generator=gen)
        for eps in (0.0, 1e-2):
            # Mamba-2, T = f32: out = w[col] * rms_norm(32 y, eps)[col]
            #                        = w[col] * rms_norm(y, eps/1024)[col]
            out = orc.forward(y, gate, w, group_size=gs, eps=eps, mode=MAMBA2)
            ref = F.rms_norm(y.double().view(rows, groups, gs), (gs,), eps=eps / 1024.0)
            ref = (ref * w.double().view(groups, gs)).view(rows, width)
            assert bool(f32_accept(out, ref.float(), rtol=2e-6).all()), f"mamba2 rms {rows}x{width}/{gs}"
            # ONNX, T = f32: Y = 32 * rms_norm(X, eps)[j] * scale[j]
            scale = 1.0 + 0.1 * torch.randn(gs, generator=gen)
            out = orc.forward(y, gate, scale, group_size=gs, eps=eps, mode=ONNX)
            ref = F.rms_norm(y.double().view(rows, groups, gs), (gs,), weight=scale.double(),
                             eps=eps) * 32.0
            assert bool(f32_accept(out, ref.view(rows, width).float(), rtol=2e-6).all()), \
                f"onnx rms {rows}x{width}/{gs}"


def pin_silu(orc) -> None:
    """ONNX, C = 1, X = 1, scale = 1, eps = 0: Y = 1 * 1 * 1 * silu(gate)."""
    F = torch.nn.functional
    g = torch.cat([torch.linspace(-30, 30, 601), torch.tensor([0.0, 0.5, -0.5, 1e-3, -1e-3, 87.0, -87.0,
                                                               -100.0, 17.0, 16.0])]).float()
    n = g.numel()
    x = torch.ones(n, 1)
    out = orc.forward(x, g.view(n, 1), torch.ones(1), group_size=1, eps=0.0, mode=ONNX).view(-1)
    ref = F.silu(g.double())
    # f32 silu: exp (< 1 ulp), add, divide: a few f32 ulps of relative error
    assert bool(f32_accept(out, ref.float(), rtol=4 * 2.0 ** -23, atol=1e-37).all()), "silu"
    # Mamba-2 route: y = [1, 1], gate = [g, 32], eps = 0:
    #   out0 = silu(g) / sqrt((silu(g)^2 + 1024) / 2)
    y = torch.ones(n, 2)
    gate = torch.stack([g, torch.full_like(g, 32.0)], dim=1)
    out = orc.forward(y, gate, torch.ones(2), group_size=2, eps=0.0, mode=MAMBA2)
    s = F.silu(g.double())
    ref0 = s / torch.sqrt((s * s + 1024.0) / 2.0)
    assert bool(f32_accept(out[:, 0], ref0.float(), rtol=8 * 2.0 ** -23, atol=1e-37).all()), "silu m2"


# --------------------------------------------------------------------------
def pin_brute(orc) -> None:
    """Double-precision twin vs the f32 oracle on every tiny shape."""
    seed = 0
    for dtype in DTYPES:
        for mode in (MAMBA2, ONNX):
            if mode == ONNX and dtype == torch.bfloat16:
                continue
            for gs in range(1, 10):
                for ngroups in (1, 2, 3):
                    for rows in (1, 3):
                        seed += 1
                        inp = ggrn_inputs.random_case(rows, gs * ngroups, gs, dtype, mode, seed,
                                                      std=1.0 + (seed % 3))
                        eps = 1e-5
                        out, t, pre = orc.forward_detail(inp.y, inp.gate, inp.w, group_size=gs,
                                                         eps=eps, mode=mode)
                        twin = orc.forward(inp.y, inp.gate, inp.w, group_size=gs, eps=eps,
                                           mode=mode, precision="f64")
                        # the twin against the f32 oracle: within 1 ulp, or a flip of the
                        # intermediate the f32 arithmetic explains
                        res = check(twin, out, mode=mode, ref_t=t, pre=pre, gate=inp.gate,
                                    group_size=gs,
                                    w_cols=weight_cols(inp.w, rows, gs * ngroups) if mode == 0 else None)
                        assert res["ok"], f"brute {dtype} mode={mode} gs={gs} g={ngroups} rows={rows}: {res}"


# --------------------------------------------------------------------------
def _case(dtype, mode, rows=3, width=24, gs=8, seed=5, std=1.0):
    return ggrn_inputs.random_case(rows, width, gs, dtype, mode, seed, std=std)


def pin_group_independence(orc) -> None:
    for dtype in DTYPES:
        for mode in (MAMBA2, ONNX):
            if mode == ONNX and dtype == torch.bfloat16:
                continue
            inp = _case(dtype, mode)
            base = orc.forward(inp.y, inp.gate, inp.w, group_size=8, eps=1e-5, mode=mode)
            y2, g2 = inp.y.clone(), inp.gate.clone()
            y2[1, 8:16] = -3.0 * y2[1, 8:16]
            g2[1, 8:16] = g2[1, 8:16] + 1.5
            pert = orc.forward(y2, g2, inp.w, group_size=8, eps=1e-5, mode=mode)
            keep = torch.ones(3, 24, dtype=torch.bool)
            keep[1, 8:16] = False
            assert torch.equal(pert[keep].view(-1).float(), base[keep].view(-1).float()), "independence"
            assert not torch.equal(pert[1, 8:16].float(), base[1, 8:16].float())


def pin_scale_invariance(orc) -> None:
    for dtype in DTYPES:
        for mode in (MAMBA2, ONNX):
            if mode == ONNX and dtype == torch.bfloat16:
                continue
            inp = _case(dtype, mode, seed=11)
            base = orc.forward(inp.y, inp.gate, inp.w, group_size=8, eps=0.0, mode=mode)
            for c in (4.0, 0.125):
                out = orc.forward(inp.y * c, inp.gate, inp.w, group_size=8, eps=0.0, mode=mode)
                assert torch.equal(out.float(), base.float()), f"scale {c} {dtype} mode={mode}"


def pin_zero_gate(orc) -> None:
    for dtype in DTYPES:
        inp = _case(dtype, MAMBA2, seed=13)
        out = orc.forward(inp.y, torch.zeros_like(inp.gate), inp.w, group_size=8, eps=1e-5,
                          mode=MAMBA2)
        assert bool((out.float() == 0).all()), "zero gate mamba2"
        if dtype != torch.bfloat16:
            inp = _case(dtype, ONNX, seed=13)
            out = orc.forward(inp.y, torch.zeros_like(inp.gate), inp.w, group_size=8, eps=1e-5,
                              mode=ONNX)
            assert bool((out.float() == 0).all()), "zero gate onnx"


def pin_permutation(orc) -> None:
    gen = torch.Generator().manual_seed(3)
    for dtype in DTYPES:
        for mode in (MAMBA2, ONNX):
            if mode == ONNX and dtype == torch.bfloat16:
                continue
            rows, width, gs = 4, 32, 16
            inp = _case(dtype, mode, rows=rows, width=width, gs=gs, seed=17)
            perm = torch.cat([torch.randperm(gs, generator=gen) + k * gs for k in range(width // gs)])
            base, t, pre = orc.forward_detail(inp.y, inp.gate, inp.w, group_size=gs, eps=1e-5,
                                              mode=mode)
            if mode == MAMBA2:
                wp = inp.w[perm]
            else:
                # scale is indexed by j, shared by the groups: permute within one period
                perm = perm.clone()
                perm[gs:] = perm[:gs] + gs
                wp = inp.w[perm[:gs]]
            out = orc.forward(inp.y[:, perm].contiguous(), inp.gate[:, perm].contiguous(), wp,
                              group_size=gs, eps=1e-5, mode=mode)
            res = check(out, base[:, perm].contiguous(), mode=mode,
                        ref_t=t[:, perm].contiguous() if t is not None else None,
                        pre=pre[:, perm].contiguous(), gate=inp.gate[:, perm].contiguous(),
                        group_size=gs,
                        w_cols=weight_cols(wp, rows, width) if mode == 0 else None)
            assert res["ok"], f"permutation {dtype} mode={mode}: {res}"


def pin_onnx_gate_separability(orc) -> None:
    """ONNX normalises X and applies the gate afterwards: a gate value moves only its element."""
    for dtype in (torch.float16, torch.float32):
        inp = _case(dtype, ONNX, seed=19)
        base = orc.forward(inp.y, inp.gate, inp.w, group_size=8, eps=1e-6, mode=ONNX)
        g2 = inp.gate.clone()
        g2[2, 13] = g2[2, 13] + 2.0
        out = orc.forward(inp.y, g2, inp.w, group_size=8, eps=1e-6, mode=ONNX)
        diff = (out.float() != base.float())
        assert bool(diff[2, 13]) and int(diff.sum()) == 1, "onnx gate separability"
    # The same perturbation under Mamba-2 semantics moves the whole group.
    inp = _case(torch.float32, MAMBA2, seed=19)
    base = orc.forward(inp.y, inp.gate, inp.w, group_size=8, eps=1e-6, mode=MAMBA2)
    g2 = inp.gate.clone()
    g2[2, 13] = g2[2, 13] + 2.0
    out = orc.forward(inp.y, g2, inp.w, group_size=8, eps=1e-6, mode=MAMBA2)
    assert int((out != base)[2, 8:16].sum()) == 8


def pin_strided(orc) -> None:
    """Row-strided views (split of a packed in-proj buffer) give the contiguous result."""
    gen = torch.Generator().manual_seed(23)
    for dtype in DTYPES:
        rows, width, gs, packed_w = 5, 20, 10, 52
        packed = torch.randn(rows, packed_w, generator=gen).to(dtype)
        other = torch.randn(rows, 29, generator=gen).to(dtype)
        w = 1.0 + 0.1 * torch.randn(width, generator=gen)
        # y and gate from the same packed buffer (same stride), then from two
        # buffers with different row strides
        for y, gate in ((packed[:, :width], packed[:, width:2 * width]),
                        (packed[:, 7:7 + width], other[:, 4:4 + width])):
            for mode in (MAMBA2, ONNX):
                if mode == ONNX and dtype == torch.bfloat16:
                    continue
                wm = w if mode == MAMBA2 else w[:gs].to(dtype)
                out_big = torch.zeros(rows, 33, dtype=dtype)
                out_view = out_big[:, 3:3 + width]
                orc.forward(y, gate, wm, group_size=gs, eps=1e-5, mode=mode, out=out_view)
                ref = orc.forward(y.contiguous(), gate.contiguous(), wm, group_size=gs, eps=1e-5,
                                  mode=mode)
                assert torch.equal(out_view.float(), ref.float()), "strided"
                assert bool((out_big[:, :3].float() == 0).all())
                assert bool((out_big[:, 3 + width:].float() == 0).all())


def pin_validation(orc) -> None:
    """Argument errors: the contract rejects what it cannot compute."""
    y = torch.zeros(2, 8)
    p = y.data_ptr()
    ok = orc.status(p, p, p, p, 2, 8, 4, 8, 8, 8, 1e-5, 0, MAMBA2)
    assert ok == 0
    assert orc.status(p, p, p, p, 2, 8, 3, 8, 8, 8, 1e-5, 0, MAMBA2) == 2   # width % gs
    assert orc.status(p, p, p, p, 2, 8, 0, 8, 8, 8, 1e-5, 0, MAMBA2) == 2   # gs = 0
    assert orc.status(p, p, p, p, -1, 8, 4, 8, 8, 8, 1e-5, 0, MAMBA2) == 2  # rows < 0
    assert orc.status(p, p, p, p, 2, 8, 4, 7, 8, 8, 1e-5, 0, MAMBA2) == 2   # stride < width
    assert orc.status(None, p, p, p, 2, 8, 4, 8, 8, 8, 1e-5, 0, MAMBA2) == 1
    assert orc.status(p, p, p, p, 2, 8, 4, 8, 8, 8, 1e-5, 2, ONNX) == 4     # onnx + bf16
    assert orc.status(p, p, p, p, 2, 8, 4, 8, 8, 8, 1e-5, 7, MAMBA2) == 4   # unknown dtype
    assert orc.status(None, None, None, None, 0, 8, 4, 8, 8, 8, 1e-5, 0, MAMBA2) == 0  # empty


ALL_PINS = [pin_golden, pin_codec, pin_rms_norm, pin_silu, pin_brute, pin_group_independence,
            pin_scale_invariance, pin_zero_gate, pin_permutation, pin_onnx_gate_separability,
            pin_strided, pin_validation]
