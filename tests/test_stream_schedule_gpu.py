"""The streaming family's unit schedule (GPU).

Eager launches claim units dynamically from device words; launches recorded
into a CUDA graph keep the static interleaved schedule.  Every unit is the
same computation whichever CTA takes it, so all of these must agree bit for
bit, and the device status word must stay clear."""
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
    g.load()


def _bits(t):
    return t.view(torch.int16) if t.dtype != torch.float32 else t.view(torch.int32)


def _case(name, rows, seed=0):
    wl = ggrn_inputs.WORKLOADS[name].with_rows(rows)
    host = ggrn_inputs.make_inputs(wl, seed=seed)
    return wl, host, gpu_util.to_device(host)


def _fwd(wl, dev, out=None):
    return g.forward(dev.y, dev.gate, dev.w, group_size=wl.group_size, eps=wl.eps, mode=wl.mode,
                     out=out, path=g.PATH_STREAM)


# rows at which automatic selection streams (12, 36 and 8 units per CTA slot
# for these three team layouts), so that the library's own graph API, which
# selects automatically, records STREAM too
@pytest.mark.parametrize("name,rows", [("mamba2_prefill", 4096), ("gdn_onnx", 16800),
                                       ("strided_odd_span", 6400)])
def test_claimed_schedule_matches_oracle_and_graph_replay(name, rows):
    g.fault_status(clear=True)
    wl, host, dev = _case(name, rows)
    assert g.plan(dev.y, dev.gate, dev.w, group_size=wl.group_size, mode=wl.mode)["path"] == \
        g.PATH_STREAM
    eager = _fwd(wl, dev)
    torch.cuda.synchronize()
    res = gpu_util.compare(eager, host, wl.group_size, wl.eps, wl.mode)
    assert res["ok"], res
    # the same call recorded by torch into a CUDA graph (static schedule)
    out = torch.empty_like(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _fwd(wl, dev, out=out)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _fwd(wl, dev, out=out)
    for _ in range(2):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(_bits(out), _bits(eager))
    # the library's own graph API records the static schedule too
    out2 = torch.empty_like(eager)
    dg = g.DecodeGraph([dict(y=dev.y, gate=dev.gate, w=dev.w, out=out2, group_size=wl.group_size,
                             eps=wl.eps, mode=wl.mode)])
    for _ in range(2):
        out2.zero_()
        dg.replay()
        torch.cuda.synchronize()
        assert torch.equal(_bits(out2), _bits(eager))
    dg.close()
    assert g.fault_status() == 0


def test_two_streams_at_once():
    """Launches on two streams overlap on the device; each launch still
    covers all of its units."""
    g.fault_status(clear=True)
    wl_a, _, dev_a = _case("mamba2_prefill", 2048, seed=1)
    wl_b, _, dev_b = _case("gdn_onnx", 4096, seed=2)
    ref_a = _fwd(wl_a, dev_a)
    ref_b = _fwd(wl_b, dev_b)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs_a = [torch.empty_like(ref_a) for _ in range(12)]
    outs_b = [torch.empty_like(ref_b) for _ in range(12)]
    for oa, ob in zip(outs_a, outs_b):
        with torch.cuda.stream(sa):
            _fwd(wl_a, dev_a, out=oa)
        with torch.cuda.stream(sb):
            _fwd(wl_b, dev_b, out=ob)
    torch.cuda.synchronize()
    for oa in outs_a:
        assert torch.equal(_bits(oa), _bits(ref_a))
    for ob in outs_b:
        assert torch.equal(_bits(ob), _bits(ref_b))
    assert g.fault_status() == 0


def test_many_launches_cycle_the_claim_words():
    """More launches than claim words on one stream: the stream keeps one
    word, and each launch replaces the previous launch's epoch in it."""
    g.fault_status(clear=True)
    wl, _, dev = _case("mamba2_prefill", 700, seed=3)
    ref = _fwd(wl, dev)
    outs = [torch.empty_like(ref) for _ in range(4)]
    for i in range(200):
        _fwd(wl, dev, out=outs[i % 4])
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(_bits(o), _bits(ref))
    assert g.fault_status() == 0


def test_more_streams_than_claim_words():
    """Launches on more streams than there are claim words, all in flight at
    once: each running launch gets a word of its own or, when every word is
    held by another stream's running launch, the static schedule; every
    output is the same bits."""
    g.fault_status(clear=True)
    wl, _, dev = _case("mamba2_prefill", 700, seed=4)
    ref = _fwd(wl, dev)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(70)]
    outs = [[torch.empty_like(ref) for _ in range(3)] for _ in streams]
    for k in range(3):
        for st, o in zip(streams, outs):
            with torch.cuda.stream(st):
                _fwd(wl, dev, out=o[k])
    torch.cuda.synchronize()
    for o in outs:
        for x in o:
            assert torch.equal(_bits(x), _bits(ref))
    assert g.fault_status() == 0


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


# Row counts around the point where each CTA slot's first unit becomes a
# short one (a half unit of groups for flat units, one row fewer for row
# units): it applies once the rest still fills a full unit per slot.
#   mamba2_prefill, flat, 1 CTA/SM: 8 of 16 groups first -> from 3 x SMs rows
#   gdn_onnx, flat, 2 CTAs/SM: 24 of 48 groups first -> from 4.5 x SMs rows
#   strided_odd_span, rows, 1 CTA/SM: 4 of 5 rows first -> from 9 x SMs rows
@pytest.mark.parametrize("name,per_sm", [("mamba2_prefill", 3.0), ("gdn_onnx", 4.5),
                                         ("strided_odd_span", 9.0)])
@pytest.mark.parametrize("delta", [-1, 0, 1])
def test_short_first_units_threshold(name, per_sm, delta):
    g.fault_status(clear=True)
    rows = int(per_sm * _sms()) + delta
    wl, host, dev = _case(name, rows, seed=rows)
    pl = g.plan(dev.y, dev.gate, dev.w, group_size=wl.group_size, mode=wl.mode, path=g.PATH_STREAM)
    assert pl["path"] == g.PATH_STREAM
    eager = _fwd(wl, dev)
    torch.cuda.synchronize()
    res = gpu_util.compare(eager, host, wl.group_size, wl.eps, wl.mode)
    assert res["ok"], res
    out = torch.empty_like(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _fwd(wl, dev, out=out)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _fwd(wl, dev, out=out)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(eager))
    assert g.fault_status() == 0
