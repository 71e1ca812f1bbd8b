"""The y16 format of the expert-output rows (include/moe.h, workspace layout):
per block of 32 consecutive values one exponent byte b = clamp(E_max - 13, 1,
240), E_max the biased fp32 exponent of the block's largest magnitude; per
value the sign and |v| + 2^(b-127) rounded to a 12-bit significand (nearest
even), kept as 4 exponent bits relative to b and 11 fraction bits; decoding
adds b back and subtracts 2^(b-127). NaN is kept as NaN.

`y16_reference` restates that definition in numpy (fp32 arithmetic, as the
device does it). The CPU tests pin the restatement to the format's stated
properties; the GPU test requires the device encoder and decoder
(moe_y16_roundtrip, the code the down GEMMs and the combine use) to match it
bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest

F32_MAX = np.float32(3.4028235e38)


def y16_reference(x: np.ndarray) -> np.ndarray:
    """x: float32, a multiple of 32 values; returns the decoded float32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, 32)
    bits = x.view(np.uint32)
    ax = bits & np.uint32(0x7FFFFFFF)
    e_max = (ax.max(axis=1, keepdims=True) >> np.uint32(23)).astype(np.int64)
    b = np.clip(e_max - 13, 1, 240).astype(np.uint32)
    d = (b << np.uint32(23)).view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        c = (ax.view(np.float32) + d).view(np.uint32).astype(np.uint64)
    em = ((c + 0x7FF + ((c >> np.uint64(12)) & np.uint64(1))) >> np.uint64(12)) \
        - (b.astype(np.uint64) << np.uint64(11))
    em = np.where(ax > np.uint32(0x7F800000), np.uint64(0x7C00), em).astype(np.uint32)
    code = em | ((bits >> np.uint32(16)) & np.uint32(0x8000))
    with np.errstate(over="ignore", invalid="ignore"):
        f = (((code & np.uint32(0x7FFF)) << np.uint32(12)) + (b << np.uint32(23))).view(np.float32) - d
    out = f.view(np.uint32) | ((code & np.uint32(0x8000)) << np.uint32(16))
    return out.view(np.float32).reshape(-1)


def block_step(x: np.ndarray) -> np.ndarray:
    """2^(b-127) of each value's block, broadcast per value."""
    ax = np.abs(x.reshape(-1, 32)).view(np.uint32)
    b = np.clip((ax.max(axis=1, keepdims=True) >> 23).astype(np.int64) - 13, 1, 240)
    return np.broadcast_to(np.exp2(b.astype(np.float64) - 127), (x.size // 32, 32)).reshape(-1)


def mixed_inputs(seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    normal = rng.standard_normal(32 * 2048).astype(np.float32)
    # log-uniform magnitudes over 2^-40 .. 2^40 within each block, random signs
    wide = (np.exp2(rng.uniform(-40, 40, 32 * 1024)) * rng.choice([-1.0, 1.0], 32 * 1024)).astype(np.float32)
    # one large outlier per block among small values
    outl = (rng.standard_normal((512, 32)) * 1e-3).astype(np.float32)
    outl[np.arange(512), rng.integers(0, 32, 512)] = 1e4
    # whole-tensor scales near both ends of the fp32 range
    huge = (rng.standard_normal(32 * 64) * 1e37).astype(np.float32)
    tiny = (rng.standard_normal(32 * 64) * 1e-38).astype(np.float32)
    return np.concatenate([normal, wide, outl.reshape(-1), huge, tiny])


def test_reference_zero_sign_and_small_values():
    x = np.zeros(64, np.float32)
    x[1] = -0.0
    x[2] = 1.0
    x[3] = -1.0
    x[32 + 5] = np.float32(1e-45)  # the smallest fp32 subnormal, alone in its block
    y = y16_reference(x)
    assert y.view(np.uint32)[0] == 0 and y.view(np.uint32)[1] == 0x80000000  # +0, -0 exact
    assert np.all(y[4:32] == 0)
    # 1 + D (D = 2^-13 here) rounds to 1 at 12 bits, so 1 decodes to 1 - 2^-13:
    # values are not kept exactly, but within 2^-12 (|v| + D)
    assert y[2] == np.float32(1 - 2.0 ** -13) and y[3] == -y[2]
    # below the block step the value is lost entirely (2^-149 against D = 2^-126)
    assert np.count_nonzero(y[32:]) == 0


def test_reference_error_bound_and_symmetry():
    x = mixed_inputs(1)
    y = y16_reference(x).astype(np.float64)
    xd = x.astype(np.float64)
    bound = 2.0 ** -12 * (np.abs(xd) + block_step(x)) * (1 + 2.0 ** -11)
    assert np.all(np.abs(y - xd) <= bound)
    # sign symmetric: negating the input negates the output
    assert np.array_equal(y16_reference(-x), -y16_reference(x))
    # values within 2^13 of their block's largest keep ~12 significant bits
    big = np.abs(xd) >= 2.0 ** 4 * block_step(x)
    rel = np.abs(y - xd)[big] / np.abs(xd)[big]
    assert rel.max() <= 2.0 ** -12 * (1 + 2.0 ** -4) * (1 + 2.0 ** -11)


def test_reference_nonfinite_values():
    x = np.ones(96, np.float32)
    x[3] = np.inf
    x[32 + 7] = -np.inf
    x[64 + 1] = np.nan
    y = y16_reference(x)
    assert y[3] == np.inf and y[32 + 7] == -np.inf and np.isnan(y[64 + 1])
    # a block holding an infinity or a NaN decodes its small finite values as zero
    assert np.all(y[[0, 1, 2, 32, 64]] == 0)
    # rounding past the largest finite value overflows to infinity, as fp32 rounding would
    x2 = np.full(32, F32_MAX, np.float32)
    assert np.all(np.isinf(y16_reference(x2)))


@pytest.mark.gpu
def test_device_encoder_decoder_match_the_definition():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_ffn_03_gb300 as moe
    moe.load_library()
    x = mixed_inputs(2)
    special = np.ones(32 * 4, np.float32)
    special[[0, 33, 66, 99]] = [np.inf, -np.inf, np.nan, -0.0]
    special[100] = np.float32(1e-45)
    x = np.concatenate([x, special, np.full(32, F32_MAX, np.float32), np.zeros(32, np.float32)])
    dev = moe.y16_roundtrip(torch.from_numpy(x).cuda()).cpu().numpy()
    ref = y16_reference(x)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(dev), nan)
    assert np.array_equal(dev.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])


def test_rejects_bad_lengths_on_host():
    import mixture_experts_ffn_03_gb300 as moe
    lib = moe.load_library()
    assert lib.moe_y16_roundtrip(None, None, 31, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_y16_roundtrip(None, None, -32, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_y16_roundtrip(None, None, 32, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_y16_roundtrip(None, None, 0, None) == moe.MOE_OK
