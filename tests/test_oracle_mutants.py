"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a temporary copy of the oracle's C source
(on the CPU, never in the CUDA path), builds it, runs every pin against it and
requires at least one pin to fail.
"""
from __future__ import annotations

import os

import pytest

import oracle
from test_oracle_pins import ALL_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = {
    "gate_up_halves_swapped": [
        ("const uint16_t* wg = w_gu + (size_t)i * H;", "const uint16_t* wg = w_gu + (size_t)(I + i) * H;"),
        ("const uint16_t* wu = w_gu + (size_t)(I + i) * H;", "const uint16_t* wu = w_gu + (size_t)i * H;"),
    ],
    "ties_to_higher_index": [("return ia < ib;", "return ia > ib;")],
    "no_renormalisation": [("weights[j] = score[ids[j]] / sum;", "weights[j] = score[ids[j]];")],
    "shared_gate_sign": [("gate = 1.0 / (1.0 + exp(-s));", "gate = 1.0 / (1.0 + exp(s));")],
    "down_transposed": [("const uint16_t* wd = w_d + (size_t)h * I;", "const uint16_t* wd = w_d + (size_t)h;"),
                        ("acc += bf16_value(wd[i]) * a_scratch[i];", "acc += bf16_value(wd[(size_t)i * H]) * a_scratch[i];")],
    "silu_as_sigmoid": [("return g / (1.0 + exp(-g));", "return 1.0 / (1.0 + exp(-g));")],
    "score_fn_swapped": [("if (score_fn == ORACLE_SOFTMAX) {", "if (score_fn != ORACLE_SOFTMAX) {")],
    "shared_expert_dropped": [("for (int h = 0; h < H; ++h) o[h] += gate * y[h];", "")],
    "last_slot_dropped": [("for (int j = 0; j < k; ++j) {\n            int e = ids[j];",
                           "for (int j = 0; j < k - 1; ++j) {\n            int e = ids[j];")],
    "bf16_high_half_misread": [("uint32_t u = ((uint32_t)bits) << 16;", "uint32_t u = ((uint32_t)bits) << 15;")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
        src = src.replace(old, new)
    mut_src = tmp_path / "mutant.c"
    mut_src.write_text(src)
    lib = oracle.build(str(mut_src), str(tmp_path / "libmutant.so"), force=True)
    failed = []
    for check in ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
