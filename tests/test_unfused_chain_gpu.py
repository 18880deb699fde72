"""The unfused PyTorch chain that bench.py times as context computes the same
operation (GPU): it must agree with the oracle within the parity tolerance,
else its timing would describe another operation."""
import pytest
import torch

import bench
import ggrn_inputs
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,rows", [("mamba2_prefill", 64), ("gdn_onnx", 128),
                                       ("strided_odd_span", 96), ("wide_single_group", 16)])
def test_unfused_chain_matches_oracle(name, rows):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = ggrn_inputs.WORKLOADS[name].with_rows(rows)
    host = ggrn_inputs.make_inputs(wl)
    dev = gpu_util.to_device(host)
    out = bench.unfused_chain_fn(wl)(dev)
    torch.cuda.synchronize()
    res = gpu_util.compare(out, host, wl.group_size, wl.eps, wl.mode)
    assert res["ok"], res
