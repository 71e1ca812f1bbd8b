"""Parity of the MXFP8-weight path (moe_forward_mxfp8, moe_mxfp8_dequant)
with the fp64 CPU oracle, through the C ABI.

The dequantisation is bit-exact against the oracle's decoder for every E4M3
code and every scale code whose products bf16 holds exactly. The layer's
bar is the bf16 path's: routing bit-exact, outputs within
1e-2 |oracle| + 1e-3 RMS(oracle) of the oracle run on the same codes.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_03_gb300 import workloads as wl
from test_gpu_parity import check_output, sample_tokens

pytestmark = pytest.mark.gpu

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
    """Every non-NaN E4M3 code against every scale code 0..254: bit-exact
    wherever the value is an exact bf16 number (all of them for scale codes
    3..246), the expected bits taken from the oracle's decoder."""
    vals = oracle.e4m3_table()
    codes_1 = np.array([c for c in range(256) if not np.isnan(vals[c])] + [0, 0x80],
                       dtype=np.uint8)                                  # 256 columns
    rows, cols = 255, codes_1.size
    codes = np.tile(codes_1, (rows, 1))
    scales = np.tile(np.arange(rows, dtype=np.uint8)[None, :], (cols // 32, 1))
    dev = torch.device("cuda")
    got = _bits(moe.mxfp8_dequant(torch.from_numpy(codes).to(dev),
                                  torch.from_numpy(scales).to(dev)))
    v = vals[codes] * np.exp2(np.arange(rows, dtype=np.float64) - 127)[:, None]
    f32 = v.astype(np.float32)
    exact = (f32.astype(np.float64) == v) & ((f32.view(np.uint32) & 0xFFFF) == 0)
    want = (f32.view(np.uint32) >> 16).astype(np.uint16)
    assert exact[3:247].all()
    # the oracle's own matrix routine agrees on the rows where every value is exact
    assert np.array_equal(oracle.mxfp8_to_bf16(codes[3:247], scales[:, 3:247]), want[3:247])
    bad = (got != want) & exact
    assert not bad.any(), f"{int(bad.sum())} mismatches, first at {np.argwhere(bad)[0]}"


def test_dequant_random_matrix(moe):
    g = torch.Generator().manual_seed(21)
    w = (torch.randn(96, 320, generator=g) * 0.02).to(torch.bfloat16)
    q, s = wl.quantize_mxfp8(w)
    dev = torch.device("cuda")
    got = _bits(moe.mxfp8_dequant(q.to(dev), s.to(dev)))
    assert np.array_equal(got, oracle.mxfp8_to_bf16(q.numpy(), s.numpy()))


def run_mx(moe, cfg, inp):
    dev = torch.device("cuda")
    x = {n: t.to(dev) for n, t in inp.items()}
    pair = lambda n: (x[n + "_q"], x[n + "_s"])  # noqa: E731
    layer = moe.MoELayerMXFP8(pair("w_gate_up"), pair("w_down"), pair("ws_gate_up"),
                              pair("ws_down"), x["w_g"], cfg.k, cfg.score_fn)
    T = cfg.T
    ids = torch.full((T, cfg.k), -1, dtype=torch.int32, device=dev)
    w = torch.zeros((T, cfg.k), dtype=torch.float32, device=dev)
    counts = torch.full((cfg.E,), -1, dtype=torch.int32, device=dev)
    out = layer.forward(x["hidden"], x["logits"], topk_ids=ids, topk_w=w, counts=counts)
    st = moe.device_status(layer.workspace(T))
    assert st == moe.MOE_OK, moe.status_string(st)
    torch.cuda.synchronize()
    return layer, out, ids, w, counts


def run_mx_case(moe, cfg, inp, n_check=None):
    layer, out, ids, w, counts = run_mx(moe, cfg, inp)
    o_ids, _ = oracle.route(inp["logits"], cfg.k, cfg.score_fn)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.array_equal(counts.cpu().numpy(), oracle.expert_counts(o_ids, cfg.E))
    toks = np.arange(cfg.T) if n_check is None else sample_tokens(cfg.T, n_check)
    ref = oracle.moe_forward_mxfp8(inp, cfg.k, cfg.score_fn, tokens=toks)["out"]
    return check_output(out[torch.as_tensor(toks, device=out.device)], ref, cfg.name)


SMALL = [
    wl.MoEConfig("mx_tiny", T=16, H=128, E=16, k=4, I=128, I_s=128, score_fn=wl.SOFTMAX),
    wl.MoEConfig("mx_single_token", T=1, H=128, E=8, k=2, I=128, I_s=128, score_fn=wl.SIGMOID),
    # I = 384: the down GEMM's last 256-value K stage is half past the end
    wl.MoEConfig("mx_ragged", T=37, H=256, E=24, k=5, I=384, I_s=128, score_fn=wl.SIGMOID),
    wl.MoEConfig("mx_k_equals_E", T=20, H=128, E=6, k=6, I=256, I_s=384, score_fn=wl.SOFTMAX),
    wl.MoEConfig("mx_bn32", T=256, H=256, E=64, k=4, I=128, I_s=128, score_fn=wl.SOFTMAX),
    wl.MoEConfig("mx_bn64", T=300, H=384, E=48, k=6, I=256, I_s=128, score_fn=wl.SIGMOID),
    # groups far above 64 tokens: many 64-token row tiles per expert
    wl.MoEConfig("mx_big_groups", T=1500, H=128, E=6, k=3, I=128, I_s=256, score_fn=wl.SOFTMAX),
    wl.MoEConfig("mx_max_experts", T=40, H=128, E=1024, k=32, I=128, I_s=128,
                 score_fn=wl.SOFTMAX),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_mx_small_cases(moe, cfg):
    run_mx_case(moe, cfg, wl.make_inputs_mxfp8(cfg, seed=0))


@pytest.mark.parametrize("name,n_check", [("decode", None), ("prefill", None)])
def test_mx_full_size(moe, name, n_check):
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs_mxfp8(cfg, seed=0, device="cuda")
    run_mx_case(moe, cfg, inp, n_check)


def test_mx_deterministic_repeat(moe):
    cfg = wl.MoEConfig("mx_repeat", T=200, H=256, E=16, k=4, I=128, I_s=128, score_fn=wl.SOFTMAX)
    inp = wl.make_inputs_mxfp8(cfg, seed=4)
    _, a, *_ = run_mx(moe, cfg, inp)
    _, b, *_ = run_mx(moe, cfg, inp)
    assert torch.equal(a, b)


def test_mx_unsupported_sizes(moe):
    cfg = wl.MoEConfig("mx_h64", T=4, H=64, E=4, k=2, I=128, I_s=128, score_fn=wl.SOFTMAX)
    d = moe.make_dims(**cfg.dims())
    st = moe.forward_mxfp8_raw(d, *([None] * 12), None)
    assert st == moe.MOE_ERR_UNSUPPORTED
