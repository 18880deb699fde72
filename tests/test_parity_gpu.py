"""Parity of the CUDA path with the CPU oracle, element by element, on the same
seeded bytes (GPU).

Bar: 16-bit outputs within 1 ulp of the oracle's f32-accumulated result, the
Mamba-2 intermediate-cast flip allowed (tests/tolerance.py); f32 outputs
within 1e-5 relative.
"""
import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
from tests import gpu_util
from tests.tolerance import assert_parity, parity_ok, ulp_dist

pytestmark = pytest.mark.gpu

MAMBA2, ONNX = 0, 1
WL = ggrn_inputs.WORKLOADS
PATHS = (g.PATH_AUTO, g.PATH_TEAM, g.PATH_WIDE, g.PATH_STRADDLE, g.PATH_SCALAR, g.PATH_STREAM,
         g.PATH_WIDE_CLUSTER)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.load()
    yield
    torch.cuda.synchronize()


def _run(inp_dev, wl, path=g.PATH_AUTO, out=None):
    return g.forward(inp_dev.y, inp_dev.gate, inp_dev.w, group_size=wl.group_size, eps=wl.eps,
                     mode=wl.mode, path=path, out=out)


# Small row counts of each workload: full width, every group, the same recipe.
SMALL_ROWS = {"mamba2_decode": 1, "mamba2_prefill": 67, "wide_single_group": 33, "gdn_onnx": 45,
              "strided_odd_span": 71}


@pytest.mark.parametrize("name", sorted(WL))
def test_workload_small(name):
    wl = WL[name].with_rows(SMALL_ROWS[name])
    host = ggrn_inputs.make_inputs(wl)
    dev = gpu_util.to_device(host)
    out = _run(dev, wl)
    torch.cuda.synchronize()
    res = gpu_util.compare(out, host, wl.group_size, wl.eps, wl.mode)
    assert res["ok"], res


@pytest.mark.parametrize("name", sorted(WL))
def test_workload_full_size_all_rows(name):
    """Full size, the launch the benchmark times: every row against the oracle
    (the streaming kernels' claimed schedule decides which CTA writes which
    rows), and two calls give the same bits."""
    wl = WL[name]
    dev = ggrn_inputs.make_inputs(wl, device="cuda")
    out = _run(dev, wl)
    out2 = _run(dev, wl)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16) if out.dtype != torch.float32 else out,
                       out2.view(torch.int16) if out2.dtype != torch.float32 else out2), \
        "two calls on the same input differ"
    host = gpu_util.to_host(dev)
    got = out.cpu()
    del out2
    res = gpu_util.compare_all_rows(got, host, wl.group_size, wl.eps, wl.mode)
    print(f"{name} all {wl.rows} rows:", res)
    assert_parity(res, name)


# group sizes: below, at and above the vector width, the warp width, the
# register tile limits; odd spans; 72, 80, 112 (16-bit) put 4-lane streaming
# teams on items 1, 2 and 6 shared-memory slots apart (each team map)
GS_LIST = [1, 2, 3, 4, 6, 7, 8, 9, 10, 12, 16, 24, 31, 32, 33, 40, 50, 64, 72, 80, 100, 112, 126,
           127, 128, 129, 200, 250, 256,
           264, 960, 1000, 1024, 1032, 2048, 4096, 5120, 5121, 8200]


def _combos():
    for dtype in (torch.bfloat16, torch.float16, torch.float32):
        for mode in (MAMBA2, ONNX):
            if mode == ONNX and dtype == torch.bfloat16:
                continue
            yield dtype, mode


@pytest.mark.parametrize("dtype,mode", list(_combos()),
                         ids=lambda v: str(v).replace("torch.", ""))
def test_sweep_every_path(dtype, mode):
    """Every kernel family on every shape it accepts, against the oracle."""
    seed = 0
    failures = []
    covered = {p: 0 for p in PATHS}
    for gs in GS_LIST:
        for rows, ngroups in ((1, 1), (3, 3), (5, 2), (2, 8)):
            if gs * ngroups * rows > 400000:
                continue
            seed += 1
            inp = ggrn_inputs.random_case(rows, gs * ngroups, gs, dtype, mode, seed,
                                          std=1.0 + seed % 2)
            wl = ggrn_inputs.Workload("sweep", rows, gs * ngroups, gs, dtype, mode, 1e-5)
            dev = gpu_util.to_device(inp)
            for path in PATHS:
                try:
                    out = _run(dev, wl, path=path)
                except g.GgrnError as e:
                    assert e.status in (7, 3), (gs, rows, path, str(e))
                    continue
                torch.cuda.synchronize()
                covered[path] += 1
                res = gpu_util.compare(out, inp, gs, 1e-5, mode, strict=False)
                if not parity_ok(res):
                    failures.append((gs, rows, ngroups, g.PATH_NAMES[path], res))
    assert not failures, failures[:10]
    for p in PATHS:
        assert covered[p] > 0, f"path {g.PATH_NAMES[p]} never ran"


@pytest.mark.parametrize("dtype,mode", list(_combos()),
                         ids=lambda v: str(v).replace("torch.", ""))
def test_lone_wide_groups(dtype, mode):
    """A batch-1 step of a norm with one wide group (and a row of two):
    automatic selection takes a cluster of CTAs per group (from 256 vectors);
    every element against the oracle."""
    cases = [(1, 7680, 7680), (1, 5120, 5120), (1, 2048, 2048), (1, 8200, 8200),
             (2, 10240, 5120), (1, 8192, 8192)]
    for rows, width, gs in cases:
        inp = ggrn_inputs.random_case(rows, width, gs, dtype, mode, seed=width + rows,
                                      std=1.5)
        dev = gpu_util.to_device(inp)
        wl = ggrn_inputs.Workload("lone", rows, width, gs, dtype, mode, 1e-5)
        plan = g.plan(dev.y, dev.gate, dev.w, group_size=gs, mode=mode)
        out = _run(dev, wl)
        torch.cuda.synchronize()
        gpu_util.compare(out, inp, gs, 1e-5, mode)
        nvec = gs * (2 if dtype != torch.float32 else 4) // 16
        if 256 <= nvec <= 1024:
            assert plan["path"] == g.PATH_WIDE_CLUSTER, (rows, width, gs, plan)


def test_strided_views_and_canaries():
    """Views split from packed buffers, different row strides for y, gate and
    out, and sentinel-filled padding that must stay untouched."""
    gen = torch.Generator().manual_seed(5)
    for dtype in (torch.bfloat16, torch.float16, torch.float32):
        for (width, gs, pw_y, pw_g, pw_o, off_o) in ((4800, 100, 9664, 9664, 4864, 16),
                                                     (960, 960, 2048, 1024, 1000, 24),
                                                     (1024, 128, 2056, 3072, 1032, 8),
                                                     (300, 100, 611, 301, 305, 1)):
            rows = 19
            packed = torch.randn(rows, pw_y, generator=gen).to(dtype)
            other = torch.randn(rows, pw_g, generator=gen).to(dtype)
            y_h = packed[:, :width]
            g_h = other[:, pw_g - width:] if pw_g >= 2 * width else other[:, :width]
            w_h = 1.0 + 0.1 * torch.randn(width, generator=gen)
            y_d = packed.cuda()[:, :width]
            g_d = (other.cuda()[:, pw_g - width:] if pw_g >= 2 * width else other.cuda()[:, :width])
            sentinel = torch.full((rows, pw_o), -1280.0, dtype=dtype).cuda()  # exact in bf16/f16/f32
            out_v = sentinel[:, off_o:off_o + width]
            g.forward(y_d, g_d, w_h.cuda(), group_size=gs, eps=1e-5, out=out_v)
            torch.cuda.synchronize()
            host = ggrn_inputs.Inputs(y=y_h.contiguous(), gate=g_h.contiguous(), w=w_h)
            res = gpu_util.compare(out_v, host, gs, 1e-5, MAMBA2)
            assert res["ok"], (dtype, width, gs, res)
            pad = sentinel.clone()
            pad[:, off_o:off_o + width] = -1280.0
            assert bool((pad.float() == -1280.0).all()), f"write outside out: {dtype} {width}/{gs}"


def test_misaligned_pointer_takes_scalar_path():
    for dtype in (torch.bfloat16, torch.float32):
        base = torch.randn(9, 1 + 5 * 640, device="cuda").to(dtype)
        y = base[:, 1:1 + 1280]
        gate = base[:, 1 + 1280:1 + 2560]
        w = torch.rand(1280, device="cuda") + 0.5
        assert g.plan(y, gate, w, group_size=640)["path"] == g.PATH_SCALAR
        out = g.forward(y, gate, w, group_size=640, eps=1e-5)
        torch.cuda.synchronize()
        host = ggrn_inputs.Inputs(y=y.cpu().contiguous(), gate=gate.cpu().contiguous(),
                                           w=w.cpu())
        res = gpu_util.compare(out, host, 640, 1e-5, MAMBA2)
        assert res["ok"], res


def test_extreme_values():
    """Saturated and overflowing silu, infinities and NaN: same as the oracle
    (NaN where the oracle has NaN)."""
    vals = [0.0, 1.0, -1.0, 8.0, -8.0, 20.0, -20.0, 87.5, -87.5, 88.0, -88.0, 88.5, -88.5, -89.0,
            -100.0, 100.0, 1e4, -1e4]
    for dtype in (torch.bfloat16, torch.float16, torch.float32):
        gs = 8
        gate = torch.tensor(vals + [0.5] * (-len(vals) % gs), dtype=torch.float32)
        n = gate.numel()
        y = torch.linspace(-2, 2, n)
        gate = gate.to(dtype).view(1, n)
        y = y.to(dtype).view(1, n)
        for mode in (MAMBA2, ONNX):
            if mode == ONNX and dtype == torch.bfloat16:
                continue
            w = (torch.rand(n) + 0.5) if mode == MAMBA2 else (torch.rand(gs) + 0.5).to(dtype)
            host = ggrn_inputs.Inputs(y=y, gate=gate, w=w)
            for path in (g.PATH_AUTO, g.PATH_SCALAR):
                out = g.forward(y.cuda(), gate.cuda(), w.cuda(), group_size=gs, eps=1e-5,
                                mode=mode, path=path)
                torch.cuda.synchronize()
                res = gpu_util.compare(out, host, gs, 1e-5, mode)
                assert res["ok"], (dtype, mode, path, res)


def test_nan_reaches_only_its_group():
    for mode, dtype in ((MAMBA2, torch.bfloat16), (ONNX, torch.float16)):
        inp = ggrn_inputs.random_case(4, 256, 64, dtype, mode, 3)
        y = inp.y.clone()
        y[2, 70] = float("nan")
        out = g.forward(y.cuda(), inp.gate.cuda(), inp.w.cuda(), group_size=64, eps=1e-5,
                        mode=mode).cpu().float()
        nan = torch.isnan(out)
        assert bool(nan[2, 64:128].all()) and int(nan.sum()) == 64
        gate = inp.gate.clone()
        gate[1, 3] = float("nan")
        out = g.forward(inp.y.cuda(), gate.cuda(), inp.w.cuda(), group_size=64, eps=1e-5,
                        mode=mode).cpu().float()
        nan = torch.isnan(out)
        if mode == MAMBA2:
            assert bool(nan[1, 0:64].all()) and int(nan.sum()) == 64   # gate enters m2
        else:
            assert bool(nan[1, 3]) and int(nan.sum()) == 1             # gate applied after


def test_zero_eps_zero_group_matches_oracle():
    y = torch.zeros(2, 16, dtype=torch.bfloat16)
    y[1] = 1.0
    gate = torch.ones(2, 16, dtype=torch.bfloat16)
    w = torch.ones(16)
    out = g.forward(y.cuda(), gate.cuda(), w.cuda(), group_size=8, eps=0.0).cpu()
    host = ggrn_inputs.Inputs(y=y, gate=gate, w=w)
    res = gpu_util.compare(out, host, 8, 0.0, MAMBA2)
    assert res["ok"], res
    assert bool(torch.isnan(out[0].float()).all())


def test_rows_zero_and_leading_axes():
    e = torch.empty(0, 128, dtype=torch.float16, device="cuda")
    s = torch.ones(128, dtype=torch.float16, device="cuda")
    assert g.forward(e, e, s, group_size=128, eps=1e-6, mode="onnx").shape == (0, 128)
    # ONNX: X of rank 3 folds its leading axes; scale as (C), (1, C), (C, 1)
    inp = ggrn_inputs.random_case(6 * 5, 4 * 32, 32, torch.float16, ONNX, 8)
    x3 = inp.y.view(6, 5, 128).cuda()
    g3 = inp.gate.view(6, 5, 128).cuda()
    outs = [g.forward(x3, g3, sc.cuda(), group_size=32, eps=1e-6, mode="onnx")
            for sc in (inp.w, inp.w.view(1, 32), inp.w.view(32, 1))]
    torch.cuda.synchronize()
    for o in outs:
        assert o.shape == (6, 5, 128)
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    res = gpu_util.compare(outs[0].view(30, 128), inp, 32, 1e-6, ONNX)
    assert res["ok"], res


def test_overlap_is_rejected():
    y = torch.randn(4, 64, device="cuda").to(torch.bfloat16)
    with pytest.raises(g.GgrnError) as ei:
        g.forward(y, y.clone(), torch.ones(64, device="cuda"), group_size=64, eps=1e-5, out=y)
    assert ei.value.status == 5


def test_deterministic_bits():
    for name in ("mamba2_prefill", "strided_odd_span", "gdn_onnx", "wide_single_group"):
        wl = WL[name].with_rows(40)
        dev = gpu_util.to_device(ggrn_inputs.make_inputs(wl))
        a = _run(dev, wl)
        b = _run(dev, wl)
        torch.cuda.synchronize()
        assert ulp_dist(a.cpu(), b.cpu()).max() == 0


# Row counts for the streaming family: several units per CTA on some CTAs, a
# ragged last wave, and (flat layouts) a partial last unit.
STREAM_ROWS = {"mamba2_prefill": 1031, "gdn_onnx": 1023, "strided_odd_span": 777}


@pytest.mark.parametrize("name", sorted(STREAM_ROWS))
def test_stream_family(name):
    """The bulk-copy streaming family, forced, against the oracle; and the
    device status word stays clear (no bounded wait ran out)."""
    g.fault_status(clear=True)
    wl = WL[name].with_rows(STREAM_ROWS[name])
    host = ggrn_inputs.make_inputs(wl)
    dev = gpu_util.to_device(host)
    assert g.plan(dev.y, dev.gate, dev.w, group_size=wl.group_size,
                  mode=wl.mode, path=g.PATH_STREAM)["path"] == g.PATH_STREAM
    out = _run(dev, wl, path=g.PATH_STREAM)
    out2 = _run(dev, wl, path=g.PATH_STREAM)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    res = gpu_util.compare(out, host, wl.group_size, wl.eps, wl.mode)
    assert res["ok"], res
    assert g.fault_status() == 0


def test_stream_flat_partial_unit_and_strided_out():
    """Flat rows whose group count leaves a partial last unit; then the same
    data with a strided output (units stay inside a row)."""
    for dtype, mode, gs in ((torch.bfloat16, MAMBA2, 64), (torch.float16, ONNX, 256),
                            (torch.float32, MAMBA2, 128), (torch.bfloat16, MAMBA2, 100)):
        rows, width = 613, gs * 6
        inp = ggrn_inputs.random_case(rows, width, gs, dtype, mode, 31)
        dev = gpu_util.to_device(inp)
        out = g.forward(dev.y, dev.gate, dev.w, group_size=gs, eps=1e-5, mode=mode,
                        path=g.PATH_STREAM)
        torch.cuda.synchronize()
        res = gpu_util.compare(out, inp, gs, 1e-5, mode)
        assert res["ok"], (dtype, gs, res)
        big = torch.zeros(rows, width + 64, dtype=dtype, device="cuda")
        ov = big[:, 32:32 + width]
        g.forward(dev.y, dev.gate, dev.w, group_size=gs, eps=1e-5, mode=mode, out=ov,
                  path=g.PATH_STREAM)
        torch.cuda.synchronize()
        assert torch.equal(ov.cpu().view(torch.int16) if dtype != torch.float32 else ov.cpu(),
                           out.cpu().view(torch.int16) if dtype != torch.float32 else out.cpu())
        assert bool((big[:, :32] == 0).all()) and bool((big[:, 32 + width:] == 0).all())
    assert g.fault_status() == 0
