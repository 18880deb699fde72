"""The streaming family's bounded waits (GPU): a launch whose producer issues
nothing makes every consumer wait run out.  The kernel must then end on its
own, report the consumer-wait bit in the device status word, leave the
buffers untouched, and leave the context usable for the next call."""
import ctypes

import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
from gated_group_rmsnorm_gb300 import binding
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.load()


def test_wait_timeout_sets_status_and_context_survives():
    g.fault_status(clear=True)
    wl = ggrn_inputs.WORKLOADS["mamba2_prefill"].with_rows(64)
    host = ggrn_inputs.make_inputs(wl, seed=21)
    dev = gpu_util.to_device(host)
    out = torch.full((wl.rows, wl.width), -1280.0, dtype=wl.dtype, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = g.load().ggrn_selftest_wait_timeout(dev.y.data_ptr(), dev.gate.data_ptr(),
                                             dev.w.data_ptr(), out.data_ptr(), wl.rows, wl.width,
                                             wl.group_size, binding.BF16, stream)
    assert st == binding.OK
    torch.cuda.synchronize()               # the kernel ended by itself
    flags = g.fault_status(clear=True)
    assert flags == 1, flags               # consumer wait ran out; nothing else
    assert bool((out == -1280.0).all())    # nothing written
    # the next call runs normally and is correct
    res = gpu_util.compare(g.forward(dev.y, dev.gate, dev.w, group_size=wl.group_size,
                                     eps=wl.eps, path=g.PATH_STREAM), host, wl.group_size,
                           wl.eps, wl.mode)
    assert res["ok"], res
    assert g.fault_status() == 0
