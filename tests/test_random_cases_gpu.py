"""Seeded random cases on the GPU: dtype, mode, group size, width, row count
and padded row strides drawn at random, run through automatic selection and
through the streaming family when it accepts the shape, each compared with
the oracle element by element."""
import random

import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
from tests import gpu_util

pytestmark = pytest.mark.gpu

GS_POOL = [4, 8, 12, 16, 24, 40, 64, 72, 80, 96, 100, 112, 128, 200, 256, 384, 960, 1000, 1024,
           2048, 5120]
N_CASES = 60


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.load()


def _case(rnd):
    while True:
        dtype = rnd.choice((torch.float32, torch.float16, torch.bfloat16))
        mode = rnd.choice((0, 1)) if dtype != torch.bfloat16 else 0
        gs = rnd.choice(GS_POOL)
        width = gs * rnd.choice((1, 2, 3, 8, 24, 48))
        rows = rnd.choice((1, 3, 17, 150, 611, 1500, 3001))
        if rows * width <= 6_000_000:
            return dtype, mode, gs, width, rows, rnd.choice((0, 8, 64)), rnd.choice((0, 8, 40))


def _strided(t, pad):
    """The same values in a row-strided view (pad extra elements per row)."""
    if pad == 0:
        return t
    buf = torch.zeros((t.shape[0], t.shape[1] + pad), dtype=t.dtype, device=t.device)
    buf[:, :t.shape[1]] = t
    return buf[:, :t.shape[1]]


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case_matches_oracle(seed):
    rnd = random.Random(seed)
    dtype, mode, gs, width, rows, in_pad, out_pad = _case(rnd)
    host = ggrn_inputs.random_case(rows, width, gs, dtype, mode, seed=seed + 1000,
                                   std=rnd.choice((0.5, 1.0, 3.0)))
    y = _strided(host.y.cuda(), in_pad)
    gate = _strided(host.gate.cuda(), in_pad)
    w = host.w.cuda()
    g.fault_status(clear=True)
    paths = [g.PATH_AUTO]
    try:
        if g.plan(y, gate, w, group_size=gs, mode=mode, path=g.PATH_STREAM)["path"] == g.PATH_STREAM:
            paths.append(g.PATH_STREAM)
    except g.GgrnError:
        pass
    for path in paths:
        out = _strided(torch.full((rows, width), float("nan"), dtype=dtype, device="cuda"),
                       out_pad)
        g.forward(y, gate, w, group_size=gs, eps=1e-5, mode=mode, out=out, path=path)
        torch.cuda.synchronize()
        res = gpu_util.compare(out, host, gs, 1e-5, mode)
        assert res["ok"], (dtype, mode, gs, width, rows, in_pad, out_pad, g.PATH_NAMES[path], res)
    assert g.fault_status() == 0
