"""Plausible mistakes planted in a copy of the oracle must fail at least one pin.

Each mutant is a textual edit of ``oracle/ggrn_oracle.cpp`` compiled into a
temporary library (CPU only).  This is how the pins are shown to pin
something: a dropped term, a wrong sign or index, or a missing rounding in the
oracle would not go unnoticed.
"""
import os

import pytest

import oracle
from tests import pins

MUTANTS = {
    # silu with the wrong sign in the exponent: x / (1 + exp(x))
    "silu_sign": ("return x / (1.0f + std::exp(-x));", "return x / (1.0f + std::exp(x));"),
    # eps dropped from the normaliser
    "drop_eps": ("v = v + eps;", "v = v + 0.0f;"),
    # sum of squares instead of the mean
    "sum_not_mean": ("float v = m2 / gs_f;", "float v = m2;"),
    # Mamba-2 weight indexed by j instead of col
    "weight_by_j": ("static_cast<const float*>(w)[col] * t;", "static_cast<const float*>(w)[j] * t;"),
    # no intermediate cast to T before the weight multiply
    "no_intermediate_cast": ("float t = round_to_t(pre, dtype);", "float t = pre;"),
    # ONNX gated before the norm (Mamba-2 ordering) -- the gate enters m2
    "onnx_gate_first": ("          x[j] = load_elem(y, n * y_row_stride + col0 + j, dtype);\n",
                        "          x[j] = load_elem(y, n * y_row_stride + col0 + j, dtype) *"
                        " silu_f32(load_elem(gate, n * gate_row_stride + col0 + j, dtype));\n"),
    # ONNX without the gate at all
    "onnx_no_gate": ("r = r * silu_f32(b);", "r = r * 1.0f; (void)b;"),
    # gate read with y's row stride
    "gate_stride": ("float b = load_elem(gate, n * gate_row_stride + col0 + j, dtype);\n          gated[j]",
                    "float b = load_elem(gate, n * y_row_stride + col0 + j, dtype);\n          gated[j]"),
    # bf16 cast truncates instead of rounding to nearest even
    "bf16_truncate": ("u += 0x7fffu + lsb;", "u += 0u * lsb;"),
    # fp16 cast rounds ties away from zero
    "f16_ties_away": ("if (rem > 0x1000u || (rem == 0x1000u && (m & 1u))) ++m;",
                      "if (rem >= 0x1000u) ++m;"),
    # rsqrt replaced by 1/x (square root forgotten)
    "no_sqrt": ("static_cast<float>(1.0 / std::sqrt(static_cast<double>(v)));",
                "static_cast<float>(1.0 / static_cast<double>(v));"),
    # squares not squared in the Mamba-2 reduction
    "abs_not_square": ("float sq = gated[j] * gated[j];", "float sq = std::fabs(gated[j]);"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC) as fh:
        return fh.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(name, source, tmp_path):
    before, after = MUTANTS[name]
    assert source.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / "mutant.cpp"
    src.write_text(source.replace(before, after))
    lib = oracle.compile_oracle(str(src), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, oracle.OracleError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
    os.remove(lib)
