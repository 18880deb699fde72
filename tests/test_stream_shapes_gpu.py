"""The streaming family at the edges of each team shape, against the oracle.

The streaming consumers take some slot ranges as given by the team shapes
the planner picks (4 vectors a lane with 2L < nvec <= 4L; 4 lanes x 7
vectors for pairs of 17..27 vectors): the slots every lane fills, the slots
wholly in the first or the second group of a pair, and the weight area's
slack that slots past an item read.  These cases sit at both ends of every
shape, for each dtype and mode the family serves, in contiguous (flat
units) and row-strided (chunk or row units) layouts, with the family forced.
"""
import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
from tests import gpu_util

pytestmark = pytest.mark.gpu

# group sizes of 16-bit T at the smallest and largest vector count of each
# team shape (8 elements a vector): 1, 2, 4, 8, 16 and 32 lanes of 4
# vectors; pairs of odd half-vector groups (gs = 4 mod 8) on 2..32 lanes and
# on the 4 x 7 layout (17..27 vectors a pair)
GS_16BIT = [32, 40, 64, 72, 128, 136, 256, 264, 512, 520, 1024,
            20, 28, 36, 60, 132, 252, 260, 508,
            68, 76, 84, 92, 100, 108]
# f32 T (4 elements a vector): 4 vectors (one lane) up to 128, and pairs
GS_F32 = [16, 20, 32, 36, 64, 68, 128, 132, 256, 260, 512, 34, 38, 54]


def _cases():
    out = []
    for gs in GS_16BIT:
        for dtype, mode in ((torch.bfloat16, 0), (torch.float16, 0), (torch.float16, 1)):
            out.append((dtype, mode, gs))
    for gs in GS_F32:
        for mode in (0, 1):
            out.append((torch.float32, mode, gs))
    return out


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.load()


def _strided(t, pad):
    if pad == 0:
        return t
    buf = torch.zeros((t.shape[0], t.shape[1] + pad), dtype=t.dtype, device=t.device)
    buf[:, :t.shape[1]] = t
    return buf[:, :t.shape[1]]


@pytest.mark.parametrize("dtype,mode,gs", _cases())
@pytest.mark.parametrize("pad", [0, 64])
def test_stream_shape_edges_match_oracle(dtype, mode, gs, pad):
    width = gs * 12
    rows = max(37, min(700, 400_000 // width))
    host = ggrn_inputs.random_case(rows, width, gs, dtype, mode, seed=gs * 7 + pad + mode)
    y = _strided(host.y.cuda(), pad)
    gate = _strided(host.gate.cuda(), pad)
    w = host.w.cuda()
    try:
        plan = g.plan(y, gate, w, group_size=gs, mode=mode, path=g.PATH_STREAM)
    except g.GgrnError:
        pytest.skip("the streaming family does not take this shape")
    if plan["path"] != g.PATH_STREAM:
        pytest.skip("the streaming family does not take this shape")
    g.fault_status(clear=True)
    out = _strided(torch.full((rows, width), float("nan"), dtype=dtype, device="cuda"), pad)
    g.forward(y, gate, w, group_size=gs, eps=1e-5, mode=mode, out=out, path=g.PATH_STREAM)
    torch.cuda.synchronize()
    res = gpu_util.compare(out, host, gs, 1e-5, mode)
    assert res["ok"], (dtype, mode, gs, pad, plan, res)
    assert g.fault_status() == 0
