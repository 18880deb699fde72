"""Tensors past 2^31 elements and 4 GiB (GPU).

Every kernel family addresses rows with 64-bit offsets; a 32-bit product of
row and stride would wrap exactly at the rows checked here.  The inputs are
the workloads' own recipes at row counts that take y, gate (and, for the
packed in-proj layout, the shared buffer) past 2^31 elements; out is filled
with NaN first, so a row no launch wrote shows up, and the oracle checks
rows on both sides of each 2^31-element and 2^31-byte boundary plus the
first, last and random rows.  Needs about 40 GB of device memory."""
import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
from tests import gpu_util

pytestmark = pytest.mark.gpu

# (workload, rows, families forced besides automatic selection)
CASES = [
    ("mamba2_prefill", 300_000, (g.PATH_TEAM, g.PATH_WIDE, g.PATH_SCALAR)),
    ("strided_odd_span", 240_000, (g.PATH_TEAM, g.PATH_STRADDLE, g.PATH_SCALAR)),
    ("gdn_onnx", 600_000, (g.PATH_TEAM, g.PATH_WIDE, g.PATH_SCALAR)),
]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 48 * 2**30:
        pytest.skip("needs about 48 GB of free device memory")
    g.load()
    yield
    torch.cuda.empty_cache()


def _boundary_rows(n, stride_elems, elem_bytes):
    rows = set()
    for limit in (2**31, 2**31 // elem_bytes):  # elements, bytes
        r = limit // stride_elems
        rows.update(x for x in (r - 1, r, r + 1) if 0 <= x < n)
    return rows


@pytest.mark.parametrize("name,rows,paths", CASES, ids=[c[0] for c in CASES])
def test_offsets_past_2_31(name, rows, paths):
    wl = ggrn_inputs.WORKLOADS[name].with_rows(rows)
    dev = ggrn_inputs.make_inputs(wl, device="cuda")
    torch.cuda.synchronize()
    in_stride = dev.y.stride(0)
    assert rows * in_stride > 2**31
    es = dev.y.element_size()
    gen = torch.Generator().manual_seed(7)
    sample = {0, 1, rows - 2, rows - 1}
    sample |= _boundary_rows(rows, in_stride, es)
    sample |= _boundary_rows(rows, wl.width, es)  # out is contiguous
    sample |= set(torch.randint(0, rows, (12,), generator=gen).tolist())
    sample = sorted(sample)
    host = gpu_util.to_host(dev, sample)
    idx = torch.tensor(sample, device="cuda")

    out = torch.empty((rows, wl.width), dtype=wl.dtype, device="cuda")
    assert g.plan(dev.y, dev.gate, dev.w, group_size=wl.group_size, mode=wl.mode,
                  out=out)["path"] == g.PATH_STREAM
    g.fault_status(clear=True)
    for path in (g.PATH_STREAM,) + paths:
        out.fill_(float("nan"))
        g.forward(dev.y, dev.gate, dev.w, group_size=wl.group_size, eps=wl.eps, mode=wl.mode,
                  out=out, path=path)
        torch.cuda.synchronize()
        assert not torch.isnan(out).any(), f"{g.PATH_NAMES[path]}: rows left unwritten"
        res = gpu_util.compare(out.index_select(0, idx).cpu(), host, wl.group_size, wl.eps,
                               wl.mode)
        assert res["ok"], (g.PATH_NAMES[path], res)
    assert g.fault_status() == 0
    del out, dev
