"""Parity of the NVFP4-weight path (moe_forward_nvfp4, moe_nvfp4_dequant) with
the fp64 CPU oracle, through the C ABI.

The dequantisation (E2M1 x E4M3, before the fp32 matrix scale) is bit-exact
against the oracle's decoder for every code and every finite scale code. The
layer's bar is the bf16 path's: routing bit-exact, outputs within
1e-2 |oracle| + 1e-3 RMS(oracle) of the oracle run on the same codes and scales.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_03_gb300 import workloads as wl
from test_gpu_parity import check_output, sample_tokens

pytestmark = pytest.mark.gpu

NAMES = ("w_gate_up", "w_down", "ws_gate_up", "ws_down")


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_ffn_03_gb300 as m
    m.load_library()
    return m


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_dequant_every_code_and_scale(moe):
    """All 16 codes in both nibbles against every finite E4M3 scale code."""
    e4 = oracle.e4m3_table()
    scale_codes = np.array([c for c in range(256) if not np.isnan(e4[c])], dtype=np.uint8)
    rows, cols = scale_codes.size, 64
    vals = np.array(list(range(16)) + list(range(15, -1, -1)) + list(range(16)) * 2, dtype=np.uint8)
    codes = np.tile((vals[0::2] | (vals[1::2] << 4)).astype(np.uint8), (rows, 1))  # [rows, 32]
    scales = np.tile(scale_codes[None, :], (cols // 16, 1))                          # [4, rows]
    dev = torch.device("cuda")
    got = _bits(moe.nvfp4_dequant(torch.from_numpy(codes).to(dev), torch.from_numpy(scales).to(dev)))
    want = oracle.nvfp4_to_bf16(codes, scales)
    assert np.array_equal(got, want), f"{int((got != want).sum())} mismatches"


def test_dequant_random_matrix(moe):
    g = torch.Generator().manual_seed(22)
    w = (torch.randn(96, 320, generator=g) * 0.02).to(torch.bfloat16)
    q, s, _ = wl.quantize_nvfp4(w)
    dev = torch.device("cuda")
    got = _bits(moe.nvfp4_dequant(q.to(dev), s.to(dev)))
    assert np.array_equal(got, oracle.nvfp4_to_bf16(q.numpy(), s.numpy()))


def run_nv(moe, cfg, inp):
    dev = torch.device("cuda")
    x = {n: t.to(dev) for n, t in inp.items()}
    tri = lambda n: (x[n + "_q"], x[n + "_s"], x[n + "_g"])  # noqa: E731
    layer = moe.MoELayerNVFP4(tri("w_gate_up"), tri("w_down"), tri("ws_gate_up"), tri("ws_down"),
                              x["w_g"], cfg.k, cfg.score_fn)
    T = cfg.T
    ids = torch.full((T, cfg.k), -1, dtype=torch.int32, device=dev)
    counts = torch.full((cfg.E,), -1, dtype=torch.int32, device=dev)
    out = layer.forward(x["hidden"], x["logits"], topk_ids=ids, counts=counts)
    st = moe.device_status(layer.workspace(T))
    assert st == moe.MOE_OK, moe.status_string(st)
    torch.cuda.synchronize()
    return layer, x, out, ids, counts


def run_nv_case(moe, cfg, inp, n_check=None):
    _, _, out, ids, counts = run_nv(moe, cfg, inp)
    o_ids, _ = oracle.route(inp["logits"], cfg.k, cfg.score_fn)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.array_equal(counts.cpu().numpy(), oracle.expert_counts(o_ids, cfg.E))
    toks = np.arange(cfg.T) if n_check is None else sample_tokens(cfg.T, n_check)
    ref = oracle.moe_forward_nvfp4(inp, cfg.k, cfg.score_fn, tokens=toks)["out"]
    return check_output(out[torch.as_tensor(toks, device=out.device)], ref, cfg.name)


SMALL = [
    wl.MoEConfig("nv_tiny", T=16, H=128, E=16, k=4, I=128, I_s=128, score_fn=wl.SOFTMAX),
    wl.MoEConfig("nv_single_token", T=1, H=128, E=8, k=2, I=128, I_s=128, score_fn=wl.SIGMOID),
    # I = 384: the down GEMM's last 256-value K stage is half past the end
    wl.MoEConfig("nv_ragged", T=37, H=256, E=24, k=5, I=384, I_s=128, score_fn=wl.SIGMOID),
    wl.MoEConfig("nv_bn32", T=256, H=256, E=64, k=4, I=128, I_s=128, score_fn=wl.SOFTMAX),
    wl.MoEConfig("nv_bn64", T=300, H=384, E=48, k=6, I=256, I_s=128, score_fn=wl.SIGMOID),
    wl.MoEConfig("nv_max_experts", T=40, H=128, E=1024, k=32, I=128, I_s=128,
                 score_fn=wl.SOFTMAX),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_nv_small_cases(moe, cfg):
    run_nv_case(moe, cfg, wl.make_inputs_nvfp4(cfg, seed=0))


@pytest.mark.parametrize("name,n_check", [("decode", None), ("prefill", None)])
def test_nv_full_size(moe, name, n_check):
    cfg = wl.CONFIGS[name]
    run_nv_case(moe, cfg, wl.make_inputs_nvfp4(cfg, seed=0, device="cuda"), n_check)


def test_nv_repeats_are_bitwise_identical(moe):
    cfg = wl.CONFIGS["prefill"]
    inp = wl.make_inputs_nvfp4(cfg, seed=2, device="cuda")
    layer, x, out0, _, _ = run_nv(moe, cfg, inp)
    out0 = out0.clone()
    out = torch.empty_like(out0)
    differ = torch.zeros((), dtype=torch.int64, device=out.device)
    for _ in range(300):
        layer.forward(x["hidden"], x["logits"], out=out)
        differ += (out != out0).any().to(torch.int64)
    assert int(differ) == 0
