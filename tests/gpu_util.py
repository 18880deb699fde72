"""Helpers shared by the GPU parity tests: move seeded inputs to the device
(keeping their strides), run the CUDA path through the binding, run the
oracle on the same bytes, and compare with the rules of tests/tolerance.py."""
from __future__ import annotations

import torch

import ggrn_inputs
import oracle
from tests.tolerance import assert_parity, check, merge, weight_cols

MAMBA2, ONNX = 0, 1


def to_device(inp: ggrn_inputs.Inputs, device="cuda") -> ggrn_inputs.Inputs:
    """Copy inputs to the device; views of a packed buffer stay views of its copy."""
    if inp.packed is not None:
        packed = inp.packed.to(device)
        width = inp.y.shape[1]
        y_off = inp.y.storage_offset() - inp.packed.storage_offset()
        g_off = inp.gate.storage_offset() - inp.packed.storage_offset()
        pw = inp.packed.shape[1]
        assert y_off < pw and g_off < pw
        y = packed[:, y_off:y_off + width]
        gate = packed[:, g_off:g_off + width]
        return ggrn_inputs.Inputs(y=y, gate=gate, w=inp.w.to(device), packed=packed)
    return ggrn_inputs.Inputs(y=inp.y.to(device), gate=inp.gate.to(device), w=inp.w.to(device))


def to_host(inp: ggrn_inputs.Inputs, rows=None) -> ggrn_inputs.Inputs:
    """Host copy of the inputs, optionally of selected rows only (contiguous)."""
    if rows is None:
        if inp.packed is not None:
            return to_device(inp, "cpu")
        return ggrn_inputs.Inputs(y=inp.y.cpu(), gate=inp.gate.cpu(), w=inp.w.cpu())
    idx = torch.as_tensor(rows, device=inp.y.device)
    return ggrn_inputs.Inputs(y=inp.y.index_select(0, idx).cpu(),
                              gate=inp.gate.index_select(0, idx).cpu(), w=inp.w.cpu())


def oracle_ref(inp_host: ggrn_inputs.Inputs, group_size: int, eps: float, mode: int):
    """(out, t, pre) from the oracle; t is None in ONNX mode."""
    return oracle.default().forward_detail(inp_host.y, inp_host.gate, inp_host.w,
                                           group_size=group_size, eps=eps, mode=mode)


def compare(got: torch.Tensor, inp_host: ggrn_inputs.Inputs, group_size: int, eps: float,
            mode: int, strict: bool = True) -> dict:
    """Compare ``got`` with the oracle on ``inp_host``; with ``strict`` (the
    default) assert the parity rules of tests/tolerance.py (``assert_parity``)."""
    ref, t, pre = oracle_ref(inp_host, group_size, eps, mode)
    rows, width = ref.shape
    w_cols = weight_cols(inp_host.w, rows, width) if mode == MAMBA2 else None
    res = check(got.cpu().reshape(rows, width), ref, mode=mode, ref_t=t, w_cols=w_cols, pre=pre,
                gate=inp_host.gate, group_size=group_size)
    if strict:
        assert_parity(res)
    return res


def compare_all_rows(got: torch.Tensor, inp_host: ggrn_inputs.Inputs, group_size: int,
                     eps: float, mode: int, block_rows: int = 1024, workers: int = 0) -> dict:
    """Every row of ``got`` (host tensor) against the oracle; returns the
    summary (not asserted).  The oracle runs over blocks of rows on all host
    cores (its C call releases the interpreter lock), then the rules are
    applied to larger blocks with torch's own threads."""
    import concurrent.futures
    import os
    rows, width = got.shape
    if workers <= 0:
        workers = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 8
    dtype = inp_host.y.dtype
    ref = torch.empty((rows, width), dtype=dtype)
    t = torch.empty((rows, width), dtype=dtype) if mode == MAMBA2 else None
    pre = torch.empty((rows, width), dtype=torch.float32)
    orc = oracle.default()

    def one(r0):
        sl = slice(r0, min(rows, r0 + block_rows))
        o, tt, pp = orc.forward_detail(inp_host.y[sl], inp_host.gate[sl], inp_host.w,
                                       group_size=group_size, eps=eps, mode=mode)
        ref[sl] = o
        pre[sl] = pp
        if t is not None:
            t[sl] = tt

    starts = list(range(0, rows, block_rows))
    with concurrent.futures.ThreadPoolExecutor(max(1, min(workers, len(starts)))) as ex:
        list(ex.map(one, starts))
    results = []
    step = max(1, (1 << 24) // width)  # about 16 M elements per check
    for r0 in range(0, rows, step):
        sl = slice(r0, min(rows, r0 + step))
        n = sl.stop - sl.start
        w_cols = weight_cols(inp_host.w, n, width) if mode == MAMBA2 else None
        results.append(check(got[sl], ref[sl], mode=mode, ref_t=t[sl] if t is not None else None,
                             w_cols=w_cols, pre=pre[sl], gate=inp_host.gate[sl],
                             group_size=group_size))
    return merge(results)
