"""The C-ABI library on the host (no GPU): it loads, exports every symbol the
header declares, validates arguments before enqueuing anything, and selects
kernel families as designed."""
import ctypes
import os
import re

import pytest
import torch

import gated_group_rmsnorm_gb300 as g
from gated_group_rmsnorm_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions(header="ggrn.h"):
    names = set()
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(ggrn_\w+)\s*\(", src, flags=re.M):
        names.add(m.group(1))
    return names


def test_every_header_is_checked():
    assert sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")) == \
        ["ggrn.h", "ggrn_timeline.h"]


def test_profiling_build_exports_its_symbols():
    """The profiling build (libggrn_timeline.so) exports what ggrn_timeline.h
    declares, besides every entry point of ggrn.h."""
    from gated_group_rmsnorm_gb300 import build as gbuild
    tl = ctypes.CDLL(gbuild.build(timeline=True))
    for name in _declared_functions("ggrn_timeline.h") | _declared_functions("ggrn.h"):
        assert hasattr(tl, name), f"{name} not exported by the profiling build"


@pytest.fixture(scope="module")
def lib():
    return g.load()


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared == set(binding.EXPORTS), declared ^ set(binding.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_version_and_status_strings(lib):
    assert lib.ggrn_version() >= 100
    for st in range(10):
        assert g.status_string(st)
    assert g.status_string(99) == "unknown status"


# Fake, 256-byte aligned "device" addresses: validation never dereferences them.
Y, GATE, W, OUT = 0x10000, 0x200000, 0x300000, 0x400000


def _fwd(*, y=Y, gate=GATE, w=W, out=OUT, rows=4, width=16, gs=8, ys=16, gts=16, os_=16,
         dtype=2, mode=0, path=0):
    return g.ggrn_forward_path(y, gate, w, out, rows, width, gs, ys, gts, os_, 1e-5, dtype, mode,
                               path, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(width=16, gs=3), binding.ERR_SHAPE),
    (dict(gs=0), binding.ERR_SHAPE),
    (dict(width=0), binding.ERR_SHAPE),
    (dict(rows=-1), binding.ERR_SHAPE),
    (dict(ys=15), binding.ERR_SHAPE),
    (dict(os_=8), binding.ERR_SHAPE),
    (dict(rows=1 << 62, ys=1 << 40, gts=1 << 40, os_=1 << 40), binding.ERR_SHAPE),
    (dict(y=0), binding.ERR_NULL),
    (dict(out=0), binding.ERR_NULL),
    (dict(w=0), binding.ERR_NULL),
    (dict(dtype=2, mode=1), binding.ERR_DTYPE),
    (dict(dtype=3), binding.ERR_DTYPE),
    (dict(mode=2), binding.ERR_DTYPE),
    (dict(y=Y + 1), binding.ERR_ALIGN),
    (dict(w=W + 2), binding.ERR_ALIGN),
    (dict(out=Y + 8), binding.ERR_OVERLAP),
    (dict(out=GATE - 2), binding.ERR_OVERLAP),
    (dict(out=W), binding.ERR_OVERLAP),
    (dict(path=9), binding.ERR_ARG),
    (dict(path=1, width=24, gs=12, ys=24, gts=24, os_=24), binding.ERR_UNSUPPORTED),  # TEAM: gs % 8
    (dict(path=3, gs=8), binding.ERR_UNSUPPORTED),              # STRADDLE needs gs % 8 != 0
    (dict(path=1, y=Y + 2), binding.ERR_ALIGN),                 # vector path, unaligned pointer
    (dict(path=2, ys=20, gts=20, os_=20), binding.ERR_ALIGN),    # vector path, unaligned stride
])
def test_validation_rejects_before_launch(kwargs, status):
    assert _fwd(**kwargs) == status


def test_rows_zero_is_a_no_op():
    assert _fwd(rows=0, y=0, gate=0, w=0, out=0) == binding.OK


def test_graph_create_rejects_bad_calls(lib):
    handle = ctypes.c_void_p()
    assert lib.ggrn_graph_create(None, 1, ctypes.byref(handle)) == binding.ERR_ARG
    calls = (binding.Call * 1)()
    calls[0] = binding.Call(Y, GATE, W, OUT, 4, 16, 3, 16, 16, 16, 1e-5, 2, 0)
    assert lib.ggrn_graph_create(calls, 1, ctypes.byref(handle)) == binding.ERR_SHAPE
    assert lib.ggrn_graph_destroy(None) == binding.OK


def _plan(rows, width, gs, dtype, mode=0, ys=None, off=0, path=0):
    es = 4 if dtype == 0 else 2
    # far-apart fake addresses; out = NULL (not allocated yet) is allowed here
    st, info = g.ggrn_plan((1 << 40) + off * es, (2 << 40) + off * es, 3 << 40, 0, rows, width,
                           gs, ys or width, ys or width, width, dtype, mode, path)
    assert st == binding.OK, g.status_string(st)
    return info


def test_plan_selects_families():
    # Mamba-2 prefill 4096x7680, group 960: streamed, one row (8 groups) per
    # unit after a first unit of half a row for each of the 304 CTA slots,
    # one warp per group (32 lanes x 4 vectors of 16 bytes), 8 consumer warps
    # + 1 producer warp, two CTAs on each of 152 SMs claiming units
    p = _plan(4096, 7680, 960, 2)
    assert (p.path, p.team_lanes, p.vec_per_lane, p.items, p.block_threads) == \
        (g.PATH_STREAM, 32, 4, 304 + (4096 * 8 - 304 * 4) // 8, 9 * 32)
    assert p.grid_blocks == 304
    # the same shape on the register-resident family: one warp per group
    p = _plan(4096, 7680, 960, 2, path=g.PATH_TEAM)
    assert (p.path, p.team_lanes, p.vec_per_lane, p.items) == (g.PATH_TEAM, 32, 4, 32768)
    # gated-DeltaNet per-head, C=128 fp16 (16 vectors): 4-lane teams with 4
    # vectors each, 8 groups per warp; 6 consumer warps, units of 48 groups
    # of the contiguous rows (the last one partial) after a first unit of 24
    # for each of the 304 CTA slots, 2 CTAs per SM
    p = _plan(32768, 4096, 128, 1, mode=1)
    assert (p.path, p.team_lanes, p.vec_per_lane, p.items, p.block_threads, p.grid_blocks) == \
        (g.PATH_STREAM, 4, 4, 304 + -(-(32768 * 32 - 304 * 24) // 48), 7 * 32, 304)
    p = _plan(32768, 4096, 128, 1, mode=1, path=g.PATH_TEAM)
    assert (p.path, p.team_lanes, p.vec_per_lane) == (g.PATH_TEAM, 4, 4)
    # wide single group of 5120 (640 vectors): one 160-thread CTA per group
    p = _plan(16384, 5120, 5120, 2)
    assert (p.path, p.block_threads, p.vec_per_lane, p.grid_blocks) == (g.PATH_WIDE, 160, 4, 16384)
    # fewer rows of it: more threads per group (1 or 2 vectors each)
    p = _plan(256, 5120, 5120, 2)
    assert (p.path, p.block_threads, p.vec_per_lane) == (g.PATH_WIDE, 640, 1)
    p = _plan(512, 5120, 5120, 2)
    assert (p.path, p.block_threads, p.vec_per_lane) == (g.PATH_WIDE, 320, 2)
    p = _plan(500, 2048, 2048, 2)
    assert (p.path, p.block_threads, p.vec_per_lane) == (g.PATH_WIDE, 128, 2)
    # odd span 100 (200 bytes, an odd number of 8-byte halves) at row stride
    # 9664: streamed in pairs of groups (25 whole 16-byte vectors) by teams of
    # 4 lanes x 7 vectors; units of 2 whole rows (6 consumer warps x 8 teams
    # x 2 groups = 96 groups) after a first unit of 1 row for each of the
    # 304 CTA slots, two CTAs per SM
    p = _plan(65536, 4800, 100, 2, ys=9664)
    assert (p.path, p.team_lanes, p.vec_per_lane, p.items, p.block_threads, p.grid_blocks) == \
        (g.PATH_STREAM, 4, 7, 304 + -(-(65536 - 304 * 1) // 2), 7 * 32, 304)
    # register-resident teams of 8 lanes x 4 vectors, 24 pairs per row
    p = _plan(65536, 4800, 100, 2, ys=9664, path=g.PATH_TEAM)
    assert (p.path, p.team_lanes, p.vec_per_lane, p.items) == (g.PATH_TEAM, 8, 4, 24 * 65536)
    # the straddle family: one warp per chunk of 5 periods (lcm(100, 8) = 200
    # elements = 25 vectors) in 128 slots, 5 chunks per row
    p = _plan(65536, 4800, 100, 2, ys=9664, path=g.PATH_STRADDLE)
    assert (p.path, p.block_threads, p.vec_per_lane, p.items) == (g.PATH_STRADDLE, 256, 4, 5 * 65536)
    # a group of 12 bf16 (24 bytes): 8-byte shared-memory vectors are not
    # chosen automatically; forced streaming pairs the groups (3 vectors per
    # pair is below 4, so it is refused)
    assert _plan(4096, 48 * 12, 12, 2).path != g.PATH_STREAM
    # a width that is not a multiple of the vector goes to the scalar path
    assert _plan(4, 300, 100, 2).path == g.PATH_SCALAR
    # decode (one row, 8 groups): a CTA of 128 threads per group, one 16-byte
    # vector per thread
    p = _plan(1, 7680, 960, 2)
    assert (p.path, p.block_threads, p.vec_per_lane, p.grid_blocks) == (g.PATH_WIDE, 128, 1, 8)
    # still few groups (16 rows x 8 = 128 <= 152 SMs); then TEAM
    assert _plan(16, 7680, 960, 2).path == g.PATH_WIDE
    assert _plan(64, 7680, 960, 2).path == g.PATH_TEAM
    # tiny groups and misaligned views fall back to element loads
    assert _plan(8, 12, 3, 2).path == g.PATH_SCALAR
    assert _plan(8, 960, 960, 2, off=1).path == g.PATH_SCALAR
    assert _plan(8, 960, 960, 2, ys=961).path == g.PATH_SCALAR
    # f32: 4 elements per vector; with few groups one vector per thread
    p = _plan(256, 128, 128, 0)
    assert (p.path, p.elems_per_vec, p.team_lanes, p.vec_per_lane) == (g.PATH_TEAM, 4, 8, 4)
    p = _plan(8, 128, 128, 0)
    assert (p.path, p.elems_per_vec, p.block_threads, p.vec_per_lane) == (g.PATH_WIDE, 4, 32, 1)
    # a few wide groups (256..1024 vectors): a cluster of up to 8 CTAs of up
    # to 128 threads per group; the decode shape's 960-wide groups stay one
    # CTA each
    p = _plan(1, 7680, 7680, 2)
    assert (p.path, p.block_threads, p.grid_blocks) == (g.PATH_WIDE_CLUSTER, 128, 8)
    p = _plan(2, 8192, 8192, 2)
    assert (p.path, p.block_threads, p.grid_blocks) == (g.PATH_WIDE_CLUSTER, 128, 16)
    assert _plan(1, 5120, 5120, 2).path == g.PATH_WIDE_CLUSTER
    assert _plan(2, 1 << 16, 1 << 16, 2).path == g.PATH_SCALAR   # beyond 1024 vectors
    assert _plan(1, 7680, 960, 2).path == g.PATH_WIDE
    assert _plan(1, 1024, 1024, 2).path == g.PATH_WIDE        # below 256 vectors
    # too many groups for every cluster to be resident at once: the one-CTA path
    assert _plan(64, 5120, 5120, 2).path != g.PATH_WIDE_CLUSTER
    # a group too wide for registers even across a cluster goes to the
    # scalar two-pass path
    assert _plan(2, 1 << 17, 1 << 17, 2).path == g.PATH_SCALAR
    # rows == 0 still plans, with nothing to launch
    assert _plan(0, 7680, 960, 2).grid_blocks == 0


def test_binding_rejects_cpu_tensors():
    y = torch.zeros(2, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        g.forward(y, y, torch.ones(8), group_size=4, eps=1e-5)


def test_noalloc_rejects_before_touching_the_device():
    """The allocation-free entry point validates and plans on the host: bad
    arguments, shapes its kernel family cannot stream, and calls beyond its
    counter's limit return before any allocation or launch."""
    def call(**kw):
        args = dict(y=Y, gate=GATE, w=W, out=OUT, rows=4, width=64, gs=32, ys=64, gts=64, os_=64,
                    dtype=2, mode=0)
        args.update(kw)
        return g.ggrn_forward_noalloc(args["y"], args["gate"], args["w"], args["out"],
                                      args["rows"], args["width"], args["gs"], args["ys"],
                                      args["gts"], args["os_"], 1e-5, args["dtype"],
                                      args["mode"], None)
    assert call(rows=0, y=0, gate=0, w=0, out=0) == binding.OK
    assert call(y=0) == binding.ERR_NULL
    assert call(gs=3) == binding.ERR_SHAPE
    assert call(y=Y + 2) == binding.ERR_ALIGN            # 2-byte aligned: no 16-byte vectors
    assert call(width=64 * 12, gs=12, ys=64 * 12, gts=64 * 12, os_=64 * 12) == \
        binding.ERR_UNSUPPORTED                          # 24-byte groups: not streamed
    # 2^38 rows of one 32-wide group, 256 groups per unit: 2^30 units is the
    # limit, 2^31 is beyond it (fake, far-apart addresses; nothing is read)
    big = dict(y=1 << 46, gate=2 << 46, w=3 << 46, out=4 << 46, width=32, ys=32, gts=32, os_=32)
    assert call(rows=1 << 39, **big) == binding.ERR_LIMIT


def _stream_units(rows, width, gs, dtype=2, mode=0):
    st, info = g.ggrn_plan(1 << 46, 2 << 46, 3 << 46, 4 << 46, rows, width, gs, width, width,
                           width, dtype, mode, g.PATH_STREAM)
    assert st == binding.OK
    return info.items


def test_noalloc_limit_boundary():
    """A call of exactly GGRN_NOALLOC_MAX_UNITS streamed units passes the
    limit check, one more unit does not.  Without a device the call that
    passes then stops at its first CUDA call (the scratch address lookup);
    with one it would launch on the fake addresses, so it is not run there."""
    if torch.cuda.is_available():
        pytest.skip("would launch a kernel on fake addresses")
    limit = 1 << 30
    width = gs = 32
    lo, hi = 1, 1 << 40          # rows with at most / more than `limit` units
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _stream_units(mid, width, gs) <= limit:
            lo = mid
        else:
            hi = mid
    assert _stream_units(lo, width, gs) == limit, "no row count gives exactly the limit"
    assert _stream_units(hi, width, gs) == limit + 1

    def call(rows):
        return g.ggrn_forward_noalloc(1 << 46, 2 << 46, 3 << 46, 4 << 46, rows, width, gs, width,
                                      width, width, 1e-5, 2, 0, None)
    assert call(hi) == binding.ERR_LIMIT
    assert call(lo) == binding.ERR_CUDA     # past the check: no device to look the scratch up on


def test_inproj_validation():
    """The packed in-proj entry point checks its column ranges on the host."""
    P = 0x1000000  # fake packed buffer; nothing is read

    def call(**kw):
        a = dict(inproj=P, stride=96, ycol=0, gcol=32, w=W, out=OUT, os_=32, rows=4, width=32,
                 gs=8, dtype=2, mode=0)
        a.update(kw)
        return g.ggrn_forward_inproj(a["inproj"], a["stride"], a["ycol"], a["gcol"], a["w"],
                                     a["out"], a["os_"], a["rows"], a["width"], a["gs"], 1e-5,
                                     a["dtype"], a["mode"], None)
    assert call(rows=0, inproj=0) == binding.OK
    assert call(inproj=0) == binding.ERR_NULL
    assert call(ycol=-1) == binding.ERR_SHAPE
    assert call(ycol=65) == binding.ERR_SHAPE            # y columns leave the row
    assert call(gcol=80) == binding.ERR_SHAPE            # gate columns leave the row
    assert call(stride=48) == binding.ERR_SHAPE          # 32 + 32 > 48
    assert call(gs=5) == binding.ERR_SHAPE               # width % group_size
    assert call(dtype=7) == binding.ERR_DTYPE
    assert call(out=P + 2 * 40) == binding.ERR_OVERLAP   # out inside the gate columns
    assert call(w=0) == binding.ERR_NULL


def test_host_pipeline_rejects_before_enqueueing():
    """ggrn_forward_host checks the host matrices and the workspace first."""
    H_Y, H_G, H_O = 0x10000000, 0x20000000, 0x30000000  # fake host addresses

    def call(**kw):
        a = dict(y=H_Y, gate=H_G, w=W, out=H_O, rows=4, width=64, gs=32, ws=0x40000000,
                 wsb=1 << 20, dtype=2)
        a.update(kw)
        return g.ggrn_forward_host(a["y"], a["gate"], a["w"], a["out"], a["rows"], a["width"],
                                   a["gs"], a["width"], a["width"], a["width"], 1e-5, a["dtype"], 0,
                                   a["ws"], a["wsb"], None)
    assert call(rows=0, y=0, gate=0, out=0, ws=0) == binding.OK
    assert call(y=0) == binding.ERR_NULL
    assert call(gs=5) == binding.ERR_SHAPE
    assert call(out=H_Y + 64) == binding.ERR_OVERLAP
    assert call(ws=0) == binding.ERR_NULL
    assert call(ws=0x40000008) == binding.ERR_ALIGN
    assert call(wsb=1000) == binding.ERR_ARG       # not one row per slot
    lib = g.load()
    need = lib.ggrn_host_workspace_bytes(4096, 7680, 2)
    assert need == 3 * 3 * (-(-min(4096, (32 << 20) // (2 * 7680 * 2)) * 7680 * 2 // 256) * 256)
    assert lib.ggrn_host_workspace_bytes(0, 7680, 2) == 0


def test_stream_short_first_units():
    """A short first unit per CTA slot once the rest fills a full unit per
    slot: units = slots + ceil((n - slots * head) / unit)."""
    # prefill (flat, 304 slots, head 4 of 8 groups, 8 groups a row)
    for rows, units in ((455, 455), (456, 304 + 304), (457, 304 + -(-(457 * 8 - 1216) // 8))):
        assert _plan(rows, 7680, 960, 2, path=g.PATH_STREAM).items == units, rows
    # odd span (rows of 48 groups, 304 slots, head 1 of 2 rows)
    for rows, units in ((911, 456), (912, 304 + 304), (913, 304 + 305)):
        assert _plan(rows, 4800, 100, 2, ys=9664, path=g.PATH_STREAM).items == units, rows
    # chunk units (part of a row each) keep one size
    p = _plan(4096, 3 * 4096, 4096 // 4, 2, ys=4 * 4096, path=g.PATH_STREAM)
    assert p.items % 4096 == 0


def test_stream_two_cta_shapes_and_fallback():
    """32-lane teams and 4 x 7 pairs run two CTAs of 8 (6) consumer warps per
    SM; where two do not fit (wide rows, whose staged f32 weight is large)
    the planner takes the one-CTA warp counts instead of leaving the SM with
    6-8 consumer warps."""
    p = _plan(16384, 7680, 960, 2, path=g.PATH_STREAM)
    assert (p.block_threads, p.grid_blocks) == (9 * 32, 2 * 152)
    p = _plan(16384, 16320, 960, 2, path=g.PATH_STREAM)
    assert (p.block_threads, p.grid_blocks) == (17 * 32, 152)
    p = _plan(65536, 4800, 100, 2, ys=9664, path=g.PATH_STREAM)
    assert (p.block_threads, p.grid_blocks) == (7 * 32, 2 * 152)
    # 120 groups a row: one-row units; two CTAs of 8 warps would not fit,
    # one CTA takes 15 consumer warps (two rows a unit)
    p = _plan(16384, 12000, 100, 2, ys=12064, path=g.PATH_STREAM)
    assert (p.block_threads, p.grid_blocks) == (16 * 32, 152)


def test_stream_threshold_by_team_layout():
    """Automatic selection streams from 6 units per CTA slot for 32-lane
    teams, 36 for teams of at most 4 lanes and 3 for paired 4 x 7 teams."""
    # prefill: 1-row units, 304 slots -> from 6 * 304 units (1824 rows;
    # counted before the short first units are cut)
    assert _plan(1823, 7680, 960, 2).path != g.PATH_STREAM
    assert _plan(1824, 7680, 960, 2).path == g.PATH_STREAM
    # 128-wide fp16 heads: units of 48 of the 32 heads a row, 304 slots ->
    # from 36 * 304 units (16415 rows)
    assert _plan(16413, 4096, 128, 1, mode=1).path == g.PATH_TEAM
    assert _plan(16416, 4096, 128, 1, mode=1).path == g.PATH_STREAM
    # odd span: 2-row units, 304 slots -> from 3 * 304 units (1823 rows)
    assert _plan(1822, 4800, 100, 2, ys=9664).path == g.PATH_TEAM
    assert _plan(1823, 4800, 100, 2, ys=9664).path == g.PATH_STREAM


def test_plans_respect_launch_limits():
    """A seeded sweep of shapes, strides, dtypes, modes and forced families:
    every plan the host accepts is a launch the device accepts (block and
    shared-memory limits, the streaming kernels' warp bounds, a nonempty
    grid), and a refusal is one of the documented statuses."""
    import random
    rnd = random.Random(1234)
    gs_pool = [1, 3, 4, 8, 12, 16, 24, 40, 64, 72, 80, 96, 100, 112, 128, 200, 256, 384, 960,
               1000, 1024, 2048, 4096, 5120, 7680, 8200]
    allowed = {binding.ERR_UNSUPPORTED, binding.ERR_ALIGN}
    checked = 0
    for _ in range(1500):
        dtype = rnd.choice((0, 1, 2))
        mode = rnd.choice((0, 1)) if dtype != 2 else 0
        gs = rnd.choice(gs_pool)
        width = gs * rnd.choice((1, 2, 3, 8, 32, 48))
        if width > 1 << 16:
            continue
        rows = rnd.choice((1, 2, 7, 64, 1000, 4096, 20000, 70000))
        ys = width + rnd.choice((0, 0, 8, 64))
        path = rnd.choice((0, 0, 1, 2, 3, 4, 5, 6))
        st, info = g.ggrn_plan(1 << 40, 2 << 40, 3 << 40, 0, rows, width, gs, ys, ys, width, dtype,
                               mode, path)
        if st != binding.OK:
            assert path != 0 and st in allowed, (st, rows, width, gs, ys, dtype, mode, path)
            continue
        checked += 1
        case = (rows, width, gs, ys, dtype, mode, path, info.as_dict())
        assert info.grid_blocks >= 1 and info.items >= 1, case
        assert 32 <= info.block_threads <= 1024 and info.block_threads % 32 == 0, case
        assert 0 <= info.smem_bytes <= 227 * 1024, case
        if info.path == g.PATH_STREAM:
            bound = 16 if info.vec_per_lane == 7 else 17   # consumer warps + producer
            assert info.block_threads <= bound * 32, case
            assert info.smem_bytes > 0, case
            # the team shapes whose slot ranges the streaming consumers take
            # as given (slots every lane fills; slots wholly in one group of
            # a pair): 4 vectors a lane with 2L < nvec <= 4L, or 4 lanes x 7
            # vectors with 17 <= nvec <= 27; pairs have an odd vector count
            se = info.elems_per_vec
            q = 1 if gs % se == 0 else 2
            nvec = q * gs // se
            lanes, vpl = info.team_lanes, info.vec_per_lane
            if q == 2:
                assert nvec % 2 == 1, case
            if vpl == 7:
                assert lanes == 4 and 17 <= nvec <= 27, case
            else:
                assert vpl == 4 and 2 * lanes < nvec <= 4 * lanes, case
        if info.path == g.PATH_WIDE_CLUSTER:
            # whole clusters of 2..8 CTAs, one per group
            ctas = info.grid_blocks // info.items
            assert 2 <= ctas <= 8 and ctas * info.items == info.grid_blocks, case
        if path == 0:
            assert info.path in (g.PATH_TEAM, g.PATH_WIDE, g.PATH_STRADDLE, g.PATH_SCALAR,
                                 g.PATH_STREAM, g.PATH_WIDE_CLUSTER), case
            if info.path == g.PATH_WIDE_CLUSTER:
                assert info.grid_blocks <= 152, case   # every cluster resident at once
    assert checked > 500
