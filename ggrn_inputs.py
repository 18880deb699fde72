"""Seeded synthetic inputs for the fused gated group-RMSNorm.

This module is the only code shared by the oracle side and the CUDA side.  It
draws random tensors and nothing else: it holds none of the method's
arithmetic.  Both sides receive the very same bytes (the CUDA side after a
host-to-device copy, or the oracle side after a device-to-host copy when the
draw runs on the GPU).

Recipe (every workload): a ``torch.Generator`` seeded with ``seed`` (0 unless
given) draws, in this order and in f32,
  1. y       (or, for the strided workload, the whole packed in-proj buffer),
  2. gate    (not drawn separately for the strided workload),
  3. the weight,
  4. the saturation mask ``rand < frac`` (prefill only) and
  5. its signs ``rand < 0.5`` -> gate = +-8,
then casts y, gate (and the ONNX scale) to T with round-to-nearest-even.

Workloads (shapes of the Nemotron-H Mamba-2 mixer, d_inner 7680 in 8 groups,
and of a gated-DeltaNet per-head output norm):
  mamba2_decode       rows=1,     width=7680, group 960, bf16, y,gate ~N(0,1),
                      w ~ 1+0.1 N(0,1), eps 1e-5
  mamba2_prefill      rows=4096,  width=7680, group 960, bf16, as above, and 1%
                      of gate entries set to +-8 (silu saturation)
  wide_single_group   rows=16384, width=5120, group 5120, bf16, y,gate ~N(0,2)
                      (std 2), w ~ U(0.5, 1.5), eps 1e-5
  gdn_onnx            rows=32768, H=32 heads x C=128 (width 4096), fp16, ONNX
                      semantics, X,gate ~N(0,1), scale ~ 1+0.05 N(0,1) (fp16),
                      eps 1e-6
  strided_odd_span    rows=65536, width=4800, group 100, bf16; y and gate are
                      the column slices [0,4800) and [4800,9600) of a packed
                      [rows, 9664] buffer ~N(0,1) (row stride 9664); w ~
                      1+0.1 N(0,1); out contiguous
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

MAMBA2, ONNX = 0, 1


@dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    width: int
    group_size: int
    dtype: torch.dtype
    mode: int
    eps: float
    std: float = 1.0                # std of y and gate
    weight: str = "normal"          # "normal": 1 + wstd*N(0,1); "uniform": U(0.5, 1.5)
    wstd: float = 0.1
    sat_frac: float = 0.0           # fraction of gate entries set to +-8
    packed_width: int = 0           # >0: y, gate are slices of a packed [rows, packed_width] buffer
    seed: int = 0
    notes: dict = field(default_factory=dict, compare=False)

    @property
    def groups(self) -> int:
        return self.width // self.group_size

    def with_rows(self, rows: int) -> "Workload":
        return replace(self, rows=rows)

    def algorithmic_bytes(self) -> int:
        """y + gate read once, out written once, the weight read once."""
        es = torch.tensor([], dtype=self.dtype).element_size()
        per_row = 3 * self.width * es
        wbytes = (self.width * 4) if self.mode == MAMBA2 else (self.group_size * es)
        return self.rows * per_row + wbytes


WORKLOADS = {
    "mamba2_decode": Workload("mamba2_decode", 1, 7680, 960, torch.bfloat16, MAMBA2, 1e-5),
    "mamba2_prefill": Workload("mamba2_prefill", 4096, 7680, 960, torch.bfloat16, MAMBA2, 1e-5,
                               sat_frac=0.01),
    "wide_single_group": Workload("wide_single_group", 16384, 5120, 5120, torch.bfloat16, MAMBA2,
                                  1e-5, std=2.0, weight="uniform"),
    "gdn_onnx": Workload("gdn_onnx", 32768, 4096, 128, torch.float16, ONNX, 1e-6, wstd=0.05),
    "strided_odd_span": Workload("strided_odd_span", 65536, 4800, 100, torch.bfloat16, MAMBA2,
                                 1e-5, packed_width=9664),
}


@dataclass
class Inputs:
    y: torch.Tensor          # [rows, width] T (possibly a strided view)
    gate: torch.Tensor       # [rows, width] T (possibly a strided view)
    w: torch.Tensor          # f32 [width] (MAMBA2) or T [group_size] (ONNX)
    packed: torch.Tensor | None = None   # the packed buffer the views come from


def make_inputs(wl: Workload, device: str | torch.device = "cpu", seed: int | None = None) -> Inputs:
    """Draw the inputs of ``wl`` on ``device`` following the recipe above."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed if seed is None else seed)
    rows, width = wl.rows, wl.width
    f32 = dict(dtype=torch.float32, device=device, generator=g)

    packed = None
    if wl.packed_width:
        pk = torch.randn((rows, wl.packed_width), **f32) * wl.std
        packed = pk.to(wl.dtype)
        del pk
        y = packed[:, :width]
        gate = packed[:, width:2 * width]
    else:
        y32 = torch.randn((rows, width), **f32) * wl.std
        gate32 = torch.randn((rows, width), **f32) * wl.std
        y = None
        gate = None

    wlen = width if wl.mode == MAMBA2 else wl.group_size
    if wl.weight == "uniform":
        w32 = 0.5 + torch.rand((wlen,), **f32)
    else:
        w32 = 1.0 + wl.wstd * torch.randn((wlen,), **f32)
    w = w32 if wl.mode == MAMBA2 else w32.to(wl.dtype)

    if not wl.packed_width:
        if wl.sat_frac > 0:
            mask = torch.rand((rows, width), **f32) < wl.sat_frac
            sign = torch.rand((rows, width), **f32) < 0.5
            sat = torch.where(sign, torch.full_like(gate32, 8.0), torch.full_like(gate32, -8.0))
            gate32 = torch.where(mask, sat, gate32)
            del mask, sign, sat
        y = y32.to(wl.dtype)
        gate = gate32.to(wl.dtype)
        del y32, gate32
    return Inputs(y=y, gate=gate, w=w, packed=packed)


def random_case(rows: int, width: int, group_size: int, dtype: torch.dtype, mode: int,
                seed: int, std: float = 1.0, device: str = "cpu") -> Inputs:
    """Small contiguous case for parity sweeps: y, gate ~ std*N(0,1), w ~ 1+0.1N."""
    wl = Workload(f"case_{rows}x{width}_g{group_size}", rows, width, group_size, dtype, mode,
                  1e-5, std=std, seed=seed)
    return make_inputs(wl, device=device)


def make_outproj_weight(d_model: int, width: int, device: str | torch.device = "cpu",
                        seed: int = 0) -> torch.Tensor:
    """The out_proj weight that follows the norm (a Linear layer's
    [d_model, width] matrix): N(0, 1/width) f32 draws from a generator seeded
    with ``seed``, cast to bf16 with round-to-nearest-even."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.randn((d_model, width), dtype=torch.float32, device=device, generator=g)
    return (w * (1.0 / width ** 0.5)).to(torch.bfloat16)
