"""ggrn_forward_inproj: y and gate read in place from a packed in-proj output
(GPU).  Results must match the oracle on the same columns, and equal, bit for
bit, ggrn_forward on the equivalent strided views (the same kernels run)."""
import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
from tests import gpu_util
from tests.tolerance import assert_parity

pytestmark = pytest.mark.gpu
MAMBA2, ONNX = 0, 1


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.load()


def _bits(t):
    return t.view(torch.int16) if t.dtype != torch.float32 else t.view(torch.int32)


def _packed(rows, pw, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(rows, pw, generator=gen).to(dtype)


def _weight(width, gs, dtype, mode, seed):
    gen = torch.Generator().manual_seed(seed + 1)
    if mode == MAMBA2:
        return 1.0 + 0.1 * torch.randn(width, generator=gen)
    return (1.0 + 0.05 * torch.randn(gs, generator=gen)).to(dtype)


# (rows, packed width, width, group, y_col, gate_col, dtype, mode): the odd
# span layout of the strided workload, gate before y, offsets that break
# 16-byte alignment, ONNX heads, f32
CASES = [
    (777, 9664, 4800, 100, 0, 4800, torch.bfloat16, MAMBA2),
    (300, 9664, 4800, 100, 4864, 0, torch.bfloat16, MAMBA2),
    (129, 2 * 7680 + 72, 7680, 960, 8, 7688, torch.bfloat16, MAMBA2),
    (65, 2 * 7680 + 72, 7680, 960, 3, 7690, torch.bfloat16, MAMBA2),
    (1, 2 * 7680 + 64, 7680, 960, 0, 7680, torch.bfloat16, MAMBA2),
    (700, 2 * 4096 + 64, 4096, 128, 64, 4160, torch.float16, ONNX),
    (50, 2 * 1024 + 4, 1024, 256, 0, 1028, torch.float32, MAMBA2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[2]}g{c[3]}y{c[4]}g{c[5]}")
def test_matches_oracle_and_views(case):
    rows, pw, width, gs, ycol, gcol, dtype, mode = case
    packed = _packed(rows, pw, dtype, seed=rows)
    w = _weight(width, gs, dtype, mode, seed=rows)
    pd, wd = packed.cuda(), w.cuda()
    out = g.forward_inproj(pd, wd, width=width, y_col=ycol, gate_col=gcol, group_size=gs,
                           eps=1e-5, mode=mode)
    ref = g.forward(pd[:, ycol:ycol + width], pd[:, gcol:gcol + width], wd, group_size=gs,
                    eps=1e-5, mode=mode)
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref))
    host = ggrn_inputs.Inputs(y=packed[:, ycol:ycol + width].contiguous(),
                              gate=packed[:, gcol:gcol + width].contiguous(), w=w)
    res = gpu_util.compare(out, host, gs, 1e-5, mode)
    assert res["ok"], res


def test_leading_axes_and_strided_out():
    """A [2, rows, packed width] buffer folds into rows; a strided output view
    is written in place and nothing beside it."""
    packed = _packed(2 * 200, 9664, torch.bfloat16, seed=5)
    w = _weight(4800, 100, torch.bfloat16, MAMBA2, seed=5)
    pd = packed.cuda().view(2, 200, 9664)
    big = torch.full((2, 200, 4864), -1280.0, dtype=torch.bfloat16, device="cuda")
    view = big[:, :, 32:32 + 4800]
    g.forward_inproj(pd, w.cuda(), width=4800, y_col=0, gate_col=4800, group_size=100, eps=1e-5,
                     out=view)
    ref = g.forward(pd[..., :4800], pd[..., 4800:9600], w.cuda(), group_size=100, eps=1e-5)
    torch.cuda.synchronize()
    assert torch.equal(_bits(view), _bits(ref))
    assert bool((big[..., :32] == -1280.0).all()) and bool((big[..., 4832:] == -1280.0).all())


def test_full_size_strided_workload_all_rows():
    """The strided workload's full packed buffer through the in-proj entry
    point: every row against the oracle, and the same bits as the view path."""
    wl = ggrn_inputs.WORKLOADS["strided_odd_span"]
    dev = ggrn_inputs.make_inputs(wl, device="cuda")
    out = g.forward_inproj(dev.packed, dev.w, width=wl.width, y_col=0, gate_col=wl.width,
                           group_size=wl.group_size, eps=wl.eps)
    ref = g.forward(dev.y, dev.gate, dev.w, group_size=wl.group_size, eps=wl.eps)
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref))
    host = gpu_util.to_host(dev)
    res = gpu_util.compare_all_rows(out.cpu(), host, wl.group_size, wl.eps, wl.mode)
    print("strided_odd_span via forward_inproj, all rows:", res)
    assert_parity(res, "strided_odd_span inproj")
