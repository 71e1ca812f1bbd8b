"""Parity of the FFN-side router path (moe_forward_router) with the fp64 oracle.

Logits: the GPU accumulates the exact bf16 products in fp32 (tensor-core
accumulators, split-K partial sums added in a fixed order), the oracle in
fp64; they must agree within LOGIT_TOL * sum_h |x_h w_eh| per logit.
Routing ranks fp32 logits on both sides, so it is unique except where two
logits lie within the accumulation error of each other: tokens whose
selection differs from the oracle's must be such near-ties (the GPU's
choice is then checked for validity instead of equality), and must be rare.
Outputs: the layer tolerance on every token routed as the oracle routes it.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_03_gb300 import workloads as wl
from test_gpu_parity import check_output, sample_tokens

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2.0 ** -14


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_ffn_03_gb300 as m
    m.load_library()
    return m


def run_router(moe, cfg, inp):
    dev = torch.device("cuda")
    x = {n: t.to(dev) for n, t in inp.items()}
    layer = moe.MoELayerRouter(x["w_router"], x["w_gate_up"], x["w_down"], x["ws_gate_up"],
                               x["ws_down"], x["w_g"], cfg.k, cfg.score_fn)
    T = cfg.T
    logits = torch.full((T, cfg.E), float("nan"), dtype=torch.float32, device=dev)
    ids = torch.full((T, cfg.k), -1, dtype=torch.int32, device=dev)
    w = torch.zeros((T, cfg.k), dtype=torch.float32, device=dev)
    out = layer.forward(x["hidden"], logits=logits, topk_ids=ids, topk_w=w)
    st = moe.device_status(layer.workspace(T))
    assert st == moe.MOE_OK, moe.status_string(st)
    torch.cuda.synchronize()
    return layer, x, out, logits, ids


def check_router_case(moe, cfg, inp, n_check=None):
    layer, x, out, logits, ids = run_router(moe, cfg, inp)
    lg64 = oracle.router_logits(inp["hidden"], inp["w_router"])
    mag = np.abs(x["hidden"].double().cpu().numpy()) @ np.abs(x["w_router"].double().cpu().numpy()).T
    band = LOGIT_TOL * mag + 1e-30
    g_lg = logits.double().cpu().numpy()
    assert np.all(np.abs(g_lg - lg64) <= band), \
        f"logits: worst err/band {np.max(np.abs(g_lg - lg64) / band):.3f}"

    o_ids, _ = oracle.route(lg64.astype(np.float32), cfg.k, cfg.score_fn)
    g_ids = ids.cpu().numpy()
    # the GPU's routing is exact on its own logits
    s_ids, _ = oracle.route(logits.cpu().numpy(), cfg.k, cfg.score_fn)
    assert np.array_equal(g_ids, s_ids)
    differ = np.nonzero((g_ids != o_ids).any(axis=1))[0]
    for t in differ:
        chosen = set(g_ids[t].tolist())
        rest = [e for e in range(cfg.E) if e not in chosen]
        worst_chosen = min(lg64[t, e] + 2 * band[t, e] for e in chosen)
        best_rest = max((lg64[t, e] - 2 * band[t, e] for e in rest), default=-np.inf)
        assert worst_chosen >= best_rest, f"token {t}: GPU selection is not a near-tie"
    assert len(differ) <= max(2, cfg.T // 20), f"{len(differ)} of {cfg.T} tokens differ"

    toks = np.arange(cfg.T) if n_check is None else sample_tokens(cfg.T, n_check)
    toks = np.array([t for t in toks if t not in set(differ.tolist())])
    ref = oracle.moe_forward_router(inp, cfg.k, cfg.score_fn, tokens=toks)["out"]
    return check_output(out[torch.as_tensor(toks, device=out.device)], ref, cfg.name), len(differ)


SMALL = [
    wl.MoEConfig("rt_tiny", T=16, H=128, E=16, k=4, I=64, I_s=64, score_fn=wl.SOFTMAX),
    # E not a multiple of 128 (a partial expert tile), H with an odd number of K steps
    wl.MoEConfig("rt_ragged", T=37, H=192, E=24, k=5, I=128, I_s=64, score_fn=wl.SIGMOID),
    wl.MoEConfig("rt_single_token", T=1, H=256, E=8, k=2, I=64, I_s=64, score_fn=wl.SOFTMAX),
    wl.MoEConfig("rt_many_splits", T=40, H=4096, E=64, k=4, I=64, I_s=64, score_fn=wl.SIGMOID),
    wl.MoEConfig("rt_max_experts", T=40, H=256, E=1024, k=32, I=64, I_s=64, score_fn=wl.SOFTMAX),
    wl.MoEConfig("rt_multiblock", T=700, H=512, E=96, k=3, I=64, I_s=128, score_fn=wl.SOFTMAX),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_router_small_cases(moe, cfg):
    check_router_case(moe, cfg, wl.make_inputs_router(cfg, seed=0))


@pytest.mark.parametrize("name,n_check", [("decode", None), ("prefill", None), ("wide", None)])
def test_router_full_size(moe, name, n_check):
    cfg = wl.CONFIGS[name]
    check_router_case(moe, cfg, wl.make_inputs_router(cfg, seed=0, device="cuda"), n_check)


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_router_repeats_are_bitwise_identical(moe, name):
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs_router(cfg, seed=1, device="cuda")
    layer, x, out0, logits0, _ = run_router(moe, cfg, inp)
    out0, logits0 = out0.clone(), logits0.clone()
    out = torch.empty_like(out0)
    logits = torch.empty_like(logits0)
    differ = torch.zeros((), dtype=torch.int64, device=out.device)
    for _ in range(200):
        layer.forward(x["hidden"], logits=logits, out=out)
        differ += ((out != out0).any() | (logits != logits0).any()).to(torch.int64)
    assert int(differ) == 0


def test_router_launch_count(moe):
    d = moe.make_dims(**wl.CONFIGS["decode"].dims())
    assert moe.launch_count_router(d) == moe.launch_count(d) + 1
