"""Reader for the hand-worked fixtures under ``tests/golden/``.

Each file holds blocks ``case NAME`` ... ``end`` of ``key value...`` lines;
``#`` starts a comment.  Keys: mode (mamba2|onnx), dtype (bf16|f16|f32), rows,
width, group_size, eps, y, gate, w, expect.
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import torch

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
_MODE = {"mamba2": 0, "onnx": 1}


@dataclass
class GoldenCase:
    name: str
    source: str
    mode: int
    dtype: torch.dtype
    rows: int
    width: int
    group_size: int
    eps: float
    y: torch.Tensor
    gate: torch.Tensor
    w: torch.Tensor
    expect: torch.Tensor


def _parse_file(path: str) -> list[GoldenCase]:
    cases, cur = [], None
    with open(path) as fh:
        for raw in fh:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
            elif key == "end":
                cases.append(_finish(cur, os.path.basename(path)))
                cur = None
            else:
                cur[key] = vals
    assert cur is None, f"unterminated case in {path}"
    return cases


def _finish(d: dict, source: str) -> GoldenCase:
    dtype = _DT[d["dtype"][0]]
    mode = _MODE[d["mode"][0]]
    rows, width, gs = int(d["rows"][0]), int(d["width"][0]), int(d["group_size"][0])

    def vec(key, dt):
        return torch.tensor([float(v) for v in d[key]], dtype=torch.float64).to(dt)

    y = vec("y", dtype).reshape(rows, width)
    gate = vec("gate", dtype).reshape(rows, width)
    w = vec("w", torch.float32 if mode == 0 else dtype)
    expect = vec("expect", dtype).reshape(rows, width)
    # every literal must be exactly representable in its type
    for key, t in (("y", y), ("gate", gate), ("w", w), ("expect", expect)):
        exact = torch.tensor([float(v) for v in d[key]], dtype=torch.float64)
        assert torch.equal(t.double().reshape(-1), exact), f"{d['name']}: {key} not exact in type"
    return GoldenCase(d["name"], source, mode, dtype, rows, width, gs, float(d["eps"][0]), y, gate,
                      w, expect)


def load_all() -> list[GoldenCase]:
    out = []
    for fn in sorted(os.listdir(GOLDEN_DIR)):
        if fn.endswith(".txt"):
            out.extend(_parse_file(os.path.join(GOLDEN_DIR, fn)))
    return out
