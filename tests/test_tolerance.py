"""The comparison rules of tests/tolerance.py, on the CPU.

A rule that accepts too much hides kernel errors, one that accepts too little
fails correct kernels.  So: planted errors that no flip explains must be
caught (a 2-ulp and a 1-ulp deviation, a "flip" far from a rounding
midpoint), and a model of a correct kernel that sums each group's squares in
another order (32 lanes, each summing every 32nd square, then a butterfly,
as the GPU's warp-wide teams do) must pass every rule, flips included.
"""
import torch

import ggrn_inputs
import oracle
from tests.tolerance import assert_parity, check, neighbours, ulp_dist, weight_cols

MAMBA2, ONNX = 0, 1


def _detail(wl, rows, seed=0):
    w = wl.with_rows(rows)
    inp = ggrn_inputs.make_inputs(w, seed=seed)
    y, g = inp.y.contiguous(), inp.gate.contiguous()
    out, t, pre = oracle.default().forward_detail(y, g, inp.w, group_size=w.group_size,
                                                  eps=w.eps, mode=w.mode)
    return w, ggrn_inputs.Inputs(y=y, gate=g, w=inp.w), out, t, pre


def _check(w, inp, got, out, t, pre):
    return check(got, out, mode=w.mode, ref_t=t, pre=pre, gate=inp.gate,
                 group_size=w.group_size,
                 w_cols=weight_cols(inp.w, w.rows, w.width) if w.mode == MAMBA2 else None)


def _reordered(w, inp):
    """A correct implementation with another summation order (f32 throughout,
    the same roundings as the definition otherwise)."""
    rows, gs = w.rows, w.group_size
    yf, gf = inp.y.float(), inp.gate.float()
    silu = gf / (1.0 + torch.exp(-gf))
    a = (yf * silu) if w.mode == MAMBA2 else yf
    a3 = a.view(rows, -1, gs)
    sq = a3 * a3
    lanes = 32
    sq = torch.nn.functional.pad(sq, (0, (-gs) % lanes))
    part = torch.zeros(rows, sq.shape[1], lanes)
    for k in range(sq.shape[2] // lanes):
        part = part + sq[:, :, k * lanes:(k + 1) * lanes]
    while part.shape[-1] > 1:
        h = part.shape[-1] // 2
        part = part[..., :h] + part[..., h:]
    nf = torch.rsqrt(((part[..., 0] / gs) + w.eps).double()).float().unsqueeze(-1)
    if w.mode == MAMBA2:
        t = (a3 * nf).to(w.dtype).float()
        return (inp.w.view(1, -1, gs) * t).to(w.dtype).view(rows, -1)
    r = ((a3 * nf) * inp.w.float().view(1, 1, gs)) * silu.view(rows, -1, gs)
    return r.to(w.dtype).view(rows, -1)


def test_reordered_sum_passes_with_flips():
    flips = 0
    for name, rows in (("mamba2_prefill", 256), ("wide_single_group", 192),
                       ("strided_odd_span", 1024), ("gdn_onnx", 1024)):
        w, inp, out, t, pre = _detail(ggrn_inputs.WORKLOADS[name], rows)
        res = _check(w, inp, _reordered(w, inp), out, t, pre)
        assert_parity(res, name)
        flips += res["flips"]
    assert flips > 0  # the rule was exercised


def test_planted_errors_are_caught():
    w, inp, out, t, pre = _detail(ggrn_inputs.WORKLOADS["mamba2_prefill"], 16)
    ordo = out.view(torch.int16).clone()
    # an element whose intermediate sits far from every rounding midpoint
    tv, pv = t.double(), pre.double()
    up, down = neighbours(t)
    spacing = (up.double() - tv).abs()
    far = ((pv - tv).abs() < 0.1 * spacing) & (out.double().abs() > 0.5)
    idx = int(torch.nonzero(far.view(-1))[0])
    for delta, name in ((2, "2-ulp"), (1, "1-ulp")):
        bad = ordo.clone()
        bad.view(-1)[idx] += delta
        res = _check(w, inp, bad.view(torch.bfloat16), out, t, pre)
        assert res["unexplained"] == 1, (name, res)
        if delta == 2:
            assert not res["ok"], res
    # the value a flip of the intermediate would give, at an element whose
    # intermediate is nowhere near a midpoint: not explained
    tn = up.view(-1)[idx:idx + 1].float()
    alt = (inp.w.view(1, -1).expand(16, -1).reshape(-1)[idx] * tn).to(torch.bfloat16)
    if int(ulp_dist(alt, out.view(-1)[idx:idx + 1])) != 0:
        bad = out.clone()
        bad.view(-1)[idx] = alt[0]
        res = _check(w, inp, bad, out, t, pre)
        assert res["unexplained"] == 1, res


def test_genuine_flip_is_explained():
    """An intermediate moved across its nearest midpoint by a relative amount
    within tau, and the output recomputed from it: an explained flip."""
    w, inp, out, t, pre = _detail(ggrn_inputs.WORKLOADS["mamba2_prefill"], 64)
    tv, pv = t.double(), pre.double()
    up, down = neighbours(t)
    toward_up = pv >= tv
    tn = torch.where(toward_up, up, down)
    mid = (tv + tn.double()) / 2
    rel = ((pv - mid).abs() / pv.abs()).view(-1)
    wc = weight_cols(inp.w, w.rows, w.width)
    alt = (wc * tn.float()).to(torch.bfloat16)
    cand = (rel < 64 * 2.0 ** -24) & (ulp_dist(alt, out).view(-1) > 0)
    assert bool(cand.any()), "no element near a midpoint in this sample"
    idx = int(torch.nonzero(cand)[0])
    got = out.clone()
    got.view(-1)[idx] = alt.view(-1)[idx]
    res = _check(w, inp, got, out, t, pre)
    assert res["flips"] == 1 and res["unexplained"] == 0 and res["ok"], res


def test_onnx_single_rounding():
    w, inp, out, t, pre = _detail(ggrn_inputs.WORKLOADS["gdn_onnx"], 8)
    assert t is None
    res = _check(w, inp, out.clone(), out, t, pre)
    assert res["same"] == res["n"] and res["unexplained"] == 0
    bad = out.view(torch.int16).clone()
    bad.view(-1)[5] += 1
    res = _check(w, inp, bad.view(torch.float16), out, t, pre)
    # one ulp off: within the stated bar, but no flip explains it unless the
    # product sat at a midpoint
    assert res["ok"] and res["unexplained"] + res["flips"] == 1
