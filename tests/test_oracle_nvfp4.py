"""Pins of the oracle's NVFP4 path (E2M1 values, E4M3 scale per 16 values, fp32
matrix scale), independent of its own decoder."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_03_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _vals(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def check_e2m1_table(lib=None):
    # the format's eight magnitudes, then the same with the sign bit set
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    tab = oracle.e2m1_table(lib)
    assert list(tab[:8]) == mags and list(-tab[8:]) == mags
    assert np.signbit(tab[8])


def check_hand_values(lib=None):
    # row 0: bytes 0x21 (values 0.5 then 1.0), 0xF7 (6.0 then -6.0); row 1: 0x3A (-1.0 then 1.5)
    codes = np.zeros((2, 8), dtype=np.uint8)
    codes[0, :2] = [0x21, 0xF7]
    codes[1, 0] = 0x3A
    scales = np.array([[0x38, 0x40]], dtype=np.uint8)   # E4M3 1.0 (row 0), 2.0 (row 1)
    v = _vals(oracle.nvfp4_to_bf16(codes, scales, lib))
    assert list(v[0, :4]) == [0.5, 1.0, 6.0, -6.0] and not v[0, 4:].any()
    assert list(v[1, :2]) == [-2.0, 3.0] and not v[1, 2:].any()


def check_roundtrip(lib=None):
    """quantise -> dequantise: every element within half an E2M1 step of the
    scaled value, or saturated at +-6 block steps."""
    g = torch.Generator().manual_seed(4)
    w = (torch.randn(48, 96, generator=g) * 0.02 * torch.exp2(
        torch.randint(-5, 6, (48, 1), generator=g).float())).to(torch.bfloat16)
    q, s, gs = wl.quantize_nvfp4(w)
    deq = _vals(oracle.nvfp4_to_bf16(q.numpy(), s.numpy(), lib)) * float(gs)
    x = w.double().numpy()
    step = s.view(torch.float8_e4m3fn).double().numpy().T.repeat(16, axis=1) * float(gs)
    v = np.abs(x) / step
    spacing = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0)) * step
    sat = v > 6
    # the quantiser divides in fp32, so a value at a midpoint may round either way
    assert np.all(np.abs(deq - x)[~sat] <= spacing[~sat] / 2 * (1 + 1e-6))
    assert np.allclose(np.abs(deq[sat]), 6 * step[sat])


def check_matrix_scales(lib=None):
    """Matrix scales 2^k equal the bf16 layer on weights multiplied by 2^k (exact
    in bf16): each scale multiplies its whole matrix (gate and up alike)."""
    cfg = wl.MoEConfig("nv", T=10, H=64, E=4, k=2, I=64, I_s=64, score_fn=wl.SIGMOID)
    inp = wl.make_inputs(cfg, seed=6)
    rng = np.random.default_rng(1)
    sc = {"w_gate_up_g": np.exp2(rng.integers(-3, 4, cfg.E)).astype(np.float64),
          "w_down_g": np.exp2(rng.integers(-3, 4, cfg.E)).astype(np.float64),
          "ws_gate_up_g": np.array([0.5]), "ws_down_g": np.array([4.0])}
    scaled = dict(inp)
    scaled["w_gate_up"] = (inp["w_gate_up"].double() * torch.from_numpy(sc["w_gate_up_g"])[:, None, None]).to(torch.bfloat16)
    scaled["w_down"] = (inp["w_down"].double() * torch.from_numpy(sc["w_down_g"])[:, None, None]).to(torch.bfloat16)
    scaled["ws_gate_up"] = (inp["ws_gate_up"].double() * 0.5).to(torch.bfloat16)
    scaled["ws_down"] = (inp["ws_down"].double() * 4.0).to(torch.bfloat16)
    want = oracle.moe_forward(scaled, cfg.k, cfg.score_fn, lib_path=lib)["out"]
    got = oracle.moe_forward({**inp, **sc}, cfg.k, cfg.score_fn, lib_path=lib)["out"]
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)


CHECKS = [check_e2m1_table, check_hand_values, check_roundtrip, check_matrix_scales]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_nvfp4_pin(check):
    check()


SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = {
    "e2m1_bias": [("const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);",
                   "const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 2);")],
    "nibble_order": [("const uint8_t nib = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);",
                      "const uint8_t nib = (c & 1) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4);")],
    "block_of_32": [("e4m3_value(scales[(size_t)(c / 16) * rows + r]);",
                     "e4m3_value(scales[(size_t)(c / 32) * rows + r]);")],
    "scale_on_gate_only": [("a_scratch[i] = silu(s_gu * g) * (s_gu * u);",
                            "a_scratch[i] = silu(s_gu * g) * u;")],
    "down_scale_dropped": [("        y[h] = s_d * acc;", "        y[h] = acc;")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_nvfp4_pins_catch_planted_mistake(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
        src = src.replace(old, new)
    mut = tmp_path / "mutant.c"
    mut.write_text(src)
    lib = oracle.build(str(mut), str(tmp_path / "libmutant.so"), force=True)
    failed = []
    for check in CHECKS:
        try:
            check(lib)
        except (AssertionError, ValueError):
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
