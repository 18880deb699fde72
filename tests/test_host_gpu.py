"""ggrn_forward_host: host-resident y, gate and out (GPU).  Pinned buffers
are read and written in place by one kernel over the host link; pageable
ones go through the workspace with the copies overlapped.  On both routes
every output row must arrive, match the oracle, and match the
device-resident call within the parity tolerance (the routes and the chunks
may take another kernel family than the whole device call)."""
import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
from gated_group_rmsnorm_gb300 import binding
from tests import gpu_util
from tests.tolerance import ulp_dist

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.load()


def _host_case(name, rows, pinned=True, seed=0):
    wl = ggrn_inputs.WORKLOADS[name].with_rows(rows)
    inp = ggrn_inputs.make_inputs(wl, seed=seed)
    if inp.packed is not None:
        packed = inp.packed.pin_memory() if pinned else inp.packed.clone()
        y, gate = packed[:, :wl.width], packed[:, wl.width:2 * wl.width]
    else:
        y = inp.y.pin_memory() if pinned else inp.y.clone()
        gate = inp.gate.pin_memory() if pinned else inp.gate.clone()
    return wl, inp, y, gate


@pytest.mark.parametrize("pinned", [True, False], ids=["in_place", "copies"])
@pytest.mark.parametrize("name,rows", [("mamba2_prefill", 1031), ("gdn_onnx", 2048),
                                       ("strided_odd_span", 777), ("wide_single_group", 300),
                                       ("mamba2_decode", 1)])
def test_matches_oracle_and_device_call(name, rows, pinned):
    wl, inp, y, gate = _host_case(name, rows, pinned=pinned)
    w = inp.w.cuda()
    out = g.forward_host(y, gate, w, group_size=wl.group_size, eps=wl.eps, mode=wl.mode)
    torch.cuda.synchronize()
    assert not out.is_cuda
    res = gpu_util.compare(out, inp, wl.group_size, wl.eps, wl.mode)
    assert res["ok"], res
    dev = g.forward(y.cuda(), gate.cuda(), w, group_size=wl.group_size, eps=wl.eps, mode=wl.mode)
    # the two calls may sum in different orders (other families): in MAMBA2
    # mode a flip of the intermediate cast becomes up to 2 ulp after the
    # weight's rounding, the case the tolerance against the oracle admits
    assert int(ulp_dist(out, dev.cpu()).max()) <= (2 if wl.mode == 0 else 1)


def test_small_workspace_pageable_memory_and_reuse():
    """One row per slot (hundreds of chunks), pageable host memory, and the
    same workspace for two calls in a row."""
    wl, inp, y, gate = _host_case("mamba2_prefill", 200, pinned=False, seed=4)
    w = inp.w.cuda()
    ws = torch.empty(3 * 3 * wl.width * 2 + 2304, dtype=torch.uint8, device="cuda")
    outs = [g.forward_host(y, gate, w, group_size=wl.group_size, eps=wl.eps, workspace=ws)
            for _ in range(2)]
    torch.cuda.synchronize()
    for o in outs:
        res = gpu_util.compare(o, inp, wl.group_size, wl.eps, wl.mode)
        assert res["ok"], res
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_ordered_on_the_callers_stream():
    """Work enqueued on the caller's stream afterwards sees every output row:
    a device copy of the host output, made on a side stream after the call,
    equals the output read after a full synchronisation."""
    wl, inp, y, gate = _host_case("gdn_onnx", 1500, seed=6)
    w = inp.w.cuda()
    side = torch.cuda.Stream()
    out = torch.full(y.shape, -1280.0, dtype=y.dtype).pin_memory()
    back = torch.empty(y.shape, dtype=y.dtype, device="cuda")
    with torch.cuda.stream(side):
        g.forward_host(y, gate, w, group_size=wl.group_size, eps=wl.eps, mode=wl.mode, out=out)
        back.copy_(out, non_blocking=True)   # ordered after the call on `side`
    side.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(back.cpu().view(torch.int16), out.view(torch.int16))
    assert not bool((out == -1280.0).any())


@pytest.mark.parametrize("pinned", [True, False], ids=["in_place", "copies"])
@pytest.mark.parametrize("pw,ycol,gcol", [(9664, 64, 4864),    # joint copy, y not at row start
                                          (9664, 4864, 0),     # joint copy, gate first
                                          (14400, 0, 9600)])   # too much unused: 2-D copies
def test_packed_host_buffers(pw, ycol, gcol, pinned):
    rows, width, gs = 333, 4800, 100
    gen = torch.Generator().manual_seed(pw + ycol)
    packed = torch.randn(rows, pw, generator=gen).to(torch.bfloat16)
    if pinned:
        packed = packed.pin_memory()
    w = 1.0 + 0.1 * torch.randn(width, generator=gen)
    y, gate = packed[:, ycol:ycol + width], packed[:, gcol:gcol + width]
    ws = g.host_workspace(rows, width, torch.bfloat16, "cuda")
    out = g.forward_host(y, gate, w.cuda(), group_size=gs, eps=1e-5, workspace=ws)
    torch.cuda.synchronize()
    host = ggrn_inputs.Inputs(y=y.contiguous(), gate=gate.contiguous(), w=w)
    res = gpu_util.compare(out, host, gs, 1e-5, 0)
    assert res["ok"], res


def test_undeclared_packed_views_copy_separately():
    """Two ranges of one pageable matrix given to ggrn_forward_host as two
    matrices (not declared packed): copied one range at a time, never with
    the bytes between them, and the same bits as the declared route."""
    rows, width, gs = 333, 4800, 100
    gen = torch.Generator().manual_seed(77)
    packed = torch.randn(rows, 9664, generator=gen).to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(width, generator=gen)).cuda()
    y, gate = packed[:, :width], packed[:, width:2 * width]
    ws = g.host_workspace(rows, width, torch.bfloat16, "cuda")
    declared = g.forward_host(y, gate, w, group_size=gs, eps=1e-5, workspace=ws)
    out = torch.empty((rows, width), dtype=torch.bfloat16)
    st = g.ggrn_forward_host(y.data_ptr(), gate.data_ptr(), w.data_ptr(), out.data_ptr(), rows,
                             width, gs, 9664, 9664, width, 1e-5, binding.DTYPE_CODE[y.dtype], 0,
                             ws.data_ptr(), ws.numel(), binding._stream_handle(w.device))
    assert st == binding.OK
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), declared.view(torch.int16))
    host = ggrn_inputs.Inputs(y=y.contiguous(), gate=gate.contiguous(), w=w.cpu())
    gpu_util.compare(out, host, gs, 1e-5, 0)


def test_route_by_host_memory():
    """Pinned y, gate and out are read in place: the workspace is left as it
    was (and may be omitted); pageable ones are staged through it."""
    wl, inp, y, gate = _host_case("mamba2_prefill", 300, seed=8)
    w = inp.w.cuda()
    ws = torch.full((g.host_workspace(300, wl.width, wl.dtype, "cuda").numel(),), 0x5A,
                    dtype=torch.uint8, device="cuda")
    out = g.forward_host(y, gate, w, group_size=wl.group_size, eps=wl.eps, workspace=ws)
    torch.cuda.synchronize()
    assert bool((ws == 0x5A).all()), "pinned buffers went through the workspace"
    assert gpu_util.compare(out, inp, wl.group_size, wl.eps, wl.mode)["ok"]
    out2 = g.forward_host(y, gate, w, group_size=wl.group_size, eps=wl.eps)  # no workspace
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    out3 = g.forward_host(y.clone(), gate.clone(), w, group_size=wl.group_size, eps=wl.eps,
                          out=torch.empty(y.shape, dtype=y.dtype), workspace=ws)
    torch.cuda.synchronize()
    assert not bool((ws == 0x5A).all()), "pageable buffers did not use the workspace"
    assert gpu_util.compare(out3, inp, wl.group_size, wl.eps, wl.mode)["ok"]


@pytest.mark.parametrize("pinned", [True, False], ids=["in_place", "copies"])
def test_misaligned_host_views(pinned):
    """y and gate one element off a 16-byte boundary (element loads only) and
    an odd row stride: still correct on both routes."""
    rows, width, gs = 129, 960, 96
    gen = torch.Generator().manual_seed(21)
    buf = torch.randn(rows, 2 * width + 3, generator=gen).to(torch.bfloat16)
    if pinned:
        buf = buf.pin_memory()
    y, gate = buf[:, 1:1 + width], buf[:, 2 + width:2 + 2 * width]
    w = 1.0 + 0.1 * torch.randn(width, generator=gen)
    out = g.forward_host(y, gate, w.cuda(), group_size=gs, eps=1e-5)
    torch.cuda.synchronize()
    host = ggrn_inputs.Inputs(y=y.contiguous(), gate=gate.contiguous(), w=w)
    res = gpu_util.compare(out, host, gs, 1e-5, 0)
    assert res["ok"], res
