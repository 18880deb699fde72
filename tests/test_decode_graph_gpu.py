"""Decode graphs: a chain of batch-1 calls captured once and replayed with one
launch gives the same bits as the same calls launched one by one (GPU)."""
import pytest
import torch

import ggrn_inputs
import gated_group_rmsnorm_gb300 as g
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _layer_inputs(n_layers):
    wl = ggrn_inputs.WORKLOADS["mamba2_decode"]
    return [gpu_util.to_device(ggrn_inputs.make_inputs(wl, seed=100 + i)) for i in range(n_layers)]


@pytest.mark.parametrize("n_layers", [1, 21])
def test_graph_replay_matches_eager(n_layers):
    wl = ggrn_inputs.WORKLOADS["mamba2_decode"]
    layers = _layer_inputs(n_layers)
    eager = [g.forward(l.y, l.gate, l.w, group_size=wl.group_size, eps=wl.eps) for l in layers]
    outs = [torch.empty_like(l.y) for l in layers]
    calls = [dict(y=l.y, gate=l.gate, w=l.w, out=o, group_size=wl.group_size, eps=wl.eps)
             for l, o in zip(layers, outs)]
    graph = g.DecodeGraph(calls)
    for _ in range(3):
        for o in outs:
            o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for e, o in zip(eager, outs):
            assert torch.equal(e.view(torch.int16), o.view(torch.int16))
    # refill one input in place: the replay sees the new values
    layers[0].y.mul_(-1)
    graph.replay()
    ref = g.forward(layers[0].y, layers[0].gate, layers[0].w, group_size=wl.group_size, eps=wl.eps)
    torch.cuda.synchronize()
    assert torch.equal(ref.view(torch.int16), outs[0].view(torch.int16))
    host = gpu_util.to_host(layers[0])
    res = gpu_util.compare(outs[0], host, wl.group_size, wl.eps, 0)
    assert res["ok"], res
    graph.close()


def test_graph_rejects_invalid_call():
    wl = ggrn_inputs.WORKLOADS["mamba2_decode"]
    l = _layer_inputs(1)[0]
    with pytest.raises(g.GgrnError):
        g.DecodeGraph([dict(y=l.y, gate=l.gate, w=l.w, out=l.y, group_size=wl.group_size,
                            eps=wl.eps)])
