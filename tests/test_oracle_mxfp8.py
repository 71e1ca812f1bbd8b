"""Pins of the oracle's MXFP8 path (E4M3 codes, one power-of-two scale per 32
K elements), independent of its own decoder."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_03_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def check_e4m3_table(lib=None):
    tab = oracle.e4m3_table(lib)
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = lib.float().double().numpy()
    assert np.array_equal(np.isnan(tab), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(tab[ok], ref[ok])
    assert np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])


def check_hand_values(lib=None):
    # row 0: 1.0, smallest subnormal, -1.0, largest normal; scale 2^(s - 127)
    codes = np.zeros((2, 32), dtype=np.uint8)
    codes[0, :4] = [0x38, 0x01, 0xB8, 0x7E]
    codes[1, :2] = [0x40, 0x3C]          # 2.0, 1.5
    scales = np.array([[127, 130]], dtype=np.uint8)   # [K/32 = 1, rows = 2]
    bits = oracle.mxfp8_to_bf16(codes, scales, lib)
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert list(vals[0, :4]) == [1.0, 2.0 ** -9, -1.0, 448.0]
    assert list(vals[1, :2]) == [16.0, 12.0]       # x 2^3
    assert not vals[0, 4:].any() and not vals[1, 2:].any()


def check_roundtrip(lib=None):
    """quantize -> dequantize stays within half a E4M3 step of the scaled value."""
    g = torch.Generator().manual_seed(3)
    w = (torch.randn(8, 64, 96, generator=g) * 0.02 * torch.exp2(
        torch.randint(-6, 7, (8, 64, 1), generator=g).float())).to(torch.bfloat16)
    codes, scales = wl.quantize_mxfp8(w)
    deq = torch.from_numpy(oracle.mxfp8_to_bf16(codes.numpy(), scales.numpy(), lib).view(np.int16))
    deq = deq.view(torch.bfloat16).double().numpy()
    x = w.double().numpy().reshape(8, 64, 3, 32)
    d = deq.reshape(8, 64, 3, 32)
    X = np.floor(np.log2(np.abs(x).max(axis=-1, keepdims=True))) - 8   # block exponent
    v = x / np.exp2(X)                                                # element before rounding
    sat = np.abs(v) > 448
    # saturated elements become +-448 * 2^X
    assert np.array_equal(d[sat], np.sign(x[sat]) * 448 * np.exp2(np.broadcast_to(X, x.shape)[sat]))
    # the rest round to the nearest E4M3 value: spacing 2^(max(e, -6) - 3) at exponent e
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -30)))
    spacing = np.exp2(np.maximum(e, -6) - 3) * np.exp2(X)
    err = np.abs(d - x)
    assert np.all(err[~sat] <= spacing[~sat] / 2)


def check_exact_weights(lib=None):
    """Weights already of the form E4M3 value x 2^k per 32-block quantise to
    themselves, so the MXFP8 layer equals the bf16 layer on the same values."""
    cfg = wl.MoEConfig("mx", T=12, H=64, E=4, k=2, I=64, I_s=64, score_fn=wl.SOFTMAX)
    inp = wl.make_inputs(cfg, seed=5)
    g = torch.Generator().manual_seed(9)
    for name in ("w_gate_up", "w_down", "ws_gate_up", "ws_down"):
        shape = inp[name].shape
        codes = torch.randint(0, 256, shape, generator=g, dtype=torch.int32).to(torch.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x30                         # no NaN codes
        # the largest magnitude of every 32-block is 448 (E4M3 exponent 8), so the
        # MX block exponent floor(log2 amax) - 8 is exactly the chosen k
        blk = codes.reshape(*shape[:-1], shape[-1] // 32, 32)
        blk[..., 0] = torch.where(blk[..., 0] >= 0x80, 0xFE, 0x7E).to(torch.uint8)
        codes = blk.reshape(shape)
        vals = codes.view(torch.float8_e4m3fn).float()
        k = torch.randint(-12, -4, (*shape[:-1], shape[-1] // 32, 1), generator=g).float()
        w = (vals.reshape(*shape[:-1], shape[-1] // 32, 32) * torch.exp2(k)).reshape(shape)
        inp[name] = w.to(torch.bfloat16)
        assert torch.equal(inp[name].float(), w)                    # exact in bf16
    ref = oracle.moe_forward(inp, cfg.k, cfg.score_fn, lib_path=lib)["out"]
    mx = dict(inp)
    for name in ("w_gate_up", "w_down", "ws_gate_up", "ws_down"):
        q, s = wl.quantize_mxfp8(mx.pop(name))
        mx[name + "_q"], mx[name + "_s"] = q, s
    got = oracle.moe_forward_mxfp8(mx, cfg.k, cfg.score_fn, lib_path=lib)["out"]
    assert np.array_equal(got, ref)


CHECKS = [check_e4m3_table, check_hand_values, check_roundtrip, check_exact_weights]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_mxfp8_pin(check):
    check()


SRC = __import__("os").path.join(__import__("os").path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = {
    "e4m3_bias_8": [("else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 8.0, e - 8);")],
    "e4m3_subnormal_scale": [("if (e == 0) v = ldexp((double)m, -9);", "if (e == 0) v = ldexp((double)m, -10);")],
    "e4m3_mantissa_bits": [("else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 16.0, e - 7);")],
    "scale_bias": [("return s == 255 ? NAN : ldexp(1.0, (int)s - 127);", "return s == 255 ? NAN : ldexp(1.0, (int)s - 128);")],
    "scale_layout_transposed": [("ue8m0_value(scales[(size_t)(c / 32) * rows + r]);",
                                 "ue8m0_value(scales[(size_t)r * (cols / 32) + c / 32]);")],
    "sign_dropped": [("    else v = ldexp(1.0 + m / 8.0, e - 7);\n    return sign ? -v : v;",
                      "    else v = ldexp(1.0 + m / 8.0, e - 7);\n    return v;")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mxfp8_pins_catch_planted_mistake(name, tmp_path):
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
