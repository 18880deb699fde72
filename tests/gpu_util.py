"""Helpers shared by the GPU parity tests: move seeded inputs to the device
(keeping their strides), run the CUDA path through the binding, run the
oracle on the same bytes, and compare with the rules of tests/tolerance.py."""
from __future__ import annotations

import torch

import ggrn_inputs
import oracle
from tests.tolerance import check, weight_cols

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
    """(out, t) from the oracle; t is None in ONNX mode."""
    if mode == MAMBA2:
        return oracle.forward(inp_host.y, inp_host.gate, inp_host.w, group_size=group_size,
                              eps=eps, mode=mode, want_t=True)
    return oracle.forward(inp_host.y, inp_host.gate, inp_host.w, group_size=group_size, eps=eps,
                          mode=mode), None


def compare(got: torch.Tensor, inp_host: ggrn_inputs.Inputs, group_size: int, eps: float,
            mode: int) -> dict:
    ref, t = oracle_ref(inp_host, group_size, eps, mode)
    rows, width = ref.shape
    w_cols = weight_cols(inp_host.w, rows, width) if mode == MAMBA2 else None
    return check(got.cpu().reshape(rows, width), ref, mode=mode, ref_t=t, w_cols=w_cols)
