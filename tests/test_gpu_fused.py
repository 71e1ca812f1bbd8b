"""The fused expert launch (gate_up and down in one persistent kernel, down
tiles waiting on device counters for their row tile's gate_up tiles) against
the two separate launches and the fp64 oracle.

The fused kernel issues the same MMAs in the same order and applies the same
epilogue arithmetic as the separate kernels, so its output must be bitwise
theirs; that checks the readiness protocol (a down tile reading h before all
of it is written would change bits) on top of the oracle's tolerance.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from mixture_experts_ffn_03_gb300 import workloads as wl
from test_gpu_parity import check_output, run_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_ffn_03_gb300 as m
    m.load_library()
    return m


CASES = [
    wl.MoEConfig("f_tiny", T=16, H=128, E=16, k=4, I=64, I_s=64, score_fn=wl.SOFTMAX),
    # I = 192: the second gate_up feature block of a row tile is half full
    wl.MoEConfig("f_ragged", T=37, H=192, E=24, k=5, I=192, I_s=128, score_fn=wl.SIGMOID),
    wl.MoEConfig("f_bn32", T=256, H=256, E=64, k=4, I=128, I_s=128, score_fn=wl.SOFTMAX),
    wl.MoEConfig("f_bn64", T=300, H=320, E=48, k=6, I=256, I_s=64, score_fn=wl.SIGMOID),
    # 13 shared-expert row tiles of 3 feature blocks each
    wl.MoEConfig("f_shared_wide", T=200, H=128, E=64, k=2, I=64, I_s=384, score_fn=wl.SOFTMAX),
    wl.MoEConfig("f_max_experts", T=40, H=64, E=1024, k=32, I=64, I_s=64, score_fn=wl.SOFTMAX),
    wl.MoEConfig("f_single_token", T=1, H=64, E=8, k=2, I=64, I_s=64, score_fn=wl.SOFTMAX),
    # fewer gate_up tiles (68) than SMs: most CTAs start on a down tile and wait
    wl.MoEConfig("f_wait_heavy", T=64, H=2048, E=4, k=2, I=2048, I_s=512, score_fn=wl.SIGMOID),
]


def forward(moe, cfg, x, fused):
    layer = moe.MoELayer(x["w_gate_up"], x["w_down"], x["ws_gate_up"], x["ws_down"], x["w_g"],
                         cfg.k, cfg.score_fn)
    with moe.expert_fusion(fused):
        out = layer.forward(x["hidden"], x["logits"])
        st = moe.device_status(layer.workspace(cfg.T))
    assert st == moe.MOE_OK, moe.status_string(st)
    torch.cuda.synchronize()
    return layer, out


def fusion_applies(moe, cfg):
    d = moe.make_dims(**cfg.dims())
    with moe.expert_fusion(True):
        on = moe.launch_count(d)
    with moe.expert_fusion(False):
        off = moe.launch_count(d)
    return on == off - 1


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_fused_bitwise_equals_separate_and_matches_oracle(moe, cfg):
    assert fusion_applies(moe, cfg)
    inp = wl.make_inputs(cfg, seed=5)
    x = {n: t.cuda() for n, t in inp.items()}
    _, out_f = forward(moe, cfg, x, True)
    _, out_s = forward(moe, cfg, x, False)
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16)), \
        f"{(out_f != out_s).sum().item()} elements differ"
    ref = oracle.moe_forward(inp, cfg.k, cfg.score_fn)["out"]
    check_output(out_f, ref, cfg.name)


@pytest.mark.parametrize("name", ["decode", "wide"])
def test_fused_full_size_bitwise_equals_separate(moe, name):
    cfg = wl.CONFIGS[name]
    assert fusion_applies(moe, cfg)
    x = wl.make_inputs(cfg, seed=0, device="cuda")
    _, out_f = forward(moe, cfg, x, True)
    out_f = out_f.clone()
    _, out_s = forward(moe, cfg, x, False)
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16))


def test_separate_launches_still_match_oracle_at_decode(moe):
    cfg = wl.CONFIGS["decode"]
    with moe.expert_fusion(False):
        run_case(moe, cfg, wl.make_inputs(cfg, seed=0, device="cuda"), n_check=32)


@pytest.mark.parametrize("name", ["f_wait_heavy", "f_bn64"])
def test_fused_repeats_are_bitwise_identical(moe, name):
    cfg = next(c for c in CASES if c.name == name)
    x = {n: t.cuda() for n, t in wl.make_inputs(cfg, seed=6).items()}
    layer, out0 = forward(moe, cfg, x, True)
    out0 = out0.clone()
    out = torch.empty_like(out0)
    differ = torch.zeros((), dtype=torch.int64, device=out.device)
    with moe.expert_fusion(True):
        for _ in range(100):
            layer.forward(x["hidden"], x["logits"], out=out)
            differ += (out.view(torch.int16) != out0.view(torch.int16)).any().to(torch.int64)
        st = moe.device_status(layer.workspace(cfg.T))
    assert st == moe.MOE_OK, moe.status_string(st)
    assert int(differ) == 0


def test_fusion_launch_counts(moe):
    d = moe.make_dims(**wl.CONFIGS["decode"].dims())
    with moe.expert_fusion(True):
        assert moe.launch_count(d) == 3
        assert moe.launch_count_router(d) == 4
    with moe.expert_fusion(False):
        assert moe.launch_count(d) == 4
    assert moe.launch_count_quantized(d) == 4
    # prefill: gate_up and down tiles differ in width (160 / 128), never fused
    p = moe.make_dims(**wl.CONFIGS["prefill"].dims())
    with moe.expert_fusion(True):
        assert moe.launch_count(p) == 5


# ---------------------------------------------------------------- whole layer
# Level 2: routing, the permute, both expert GEMMs and the combine in one
# persistent launch (decode-sized batches, E <= 256). Same arithmetic as the
# separate launches, so the outputs, ids, weights and counts are bitwise
# theirs; the routing-to-experts and experts-to-combine hand-offs are the
# launch's bounded grid-wide waits.
LAYER_CASES = [c for c in CASES if c.E <= 256] + [
    # 256 tokens: more tokens than CTAs, so CTAs route and combine several each
    wl.MoEConfig("l_many_tokens", T=256, H=256, E=256, k=8, I=128, I_s=128, score_fn=wl.SOFTMAX),
    # fp32 y rows would take more than 64 MB: y16 rows and their combine
    wl.MoEConfig("l_y16_rows", T=256, H=7296, E=256, k=8, I=64, I_s=64, score_fn=wl.SIGMOID),
]


def layer_applies(moe, cfg):
    d = moe.make_dims(**cfg.dims())
    with moe.expert_fusion(2):
        return moe.launch_count(d) == 1


def run_layer(moe, cfg, x, level):
    layer = moe.MoELayer(x["w_gate_up"], x["w_down"], x["ws_gate_up"], x["ws_down"], x["w_g"],
                         cfg.k, cfg.score_fn)
    ids = torch.full((cfg.T, cfg.k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    counts = torch.full((cfg.E,), -1, dtype=torch.int32, device="cuda")
    with moe.expert_fusion(level):
        out = layer.forward(x["hidden"], x["logits"], topk_ids=ids, topk_w=w, counts=counts)
        st = moe.device_status(layer.workspace(cfg.T))
    assert st == moe.MOE_OK, moe.status_string(st)
    torch.cuda.synchronize()
    return layer, out, ids, w, counts


@pytest.mark.parametrize("cfg", LAYER_CASES, ids=lambda c: c.name)
def test_layer_launch_bitwise_equals_separate(moe, cfg):
    assert layer_applies(moe, cfg)
    inp = wl.make_inputs(cfg, seed=7)
    x = {n: t.cuda() for n, t in inp.items()}
    _, out_l, ids_l, w_l, c_l = run_layer(moe, cfg, x, 2)
    _, out_s, ids_s, w_s, c_s = run_layer(moe, cfg, x, 0)
    assert torch.equal(ids_l, ids_s) and torch.equal(c_l, c_s)
    assert torch.equal(w_l.view(torch.int32), w_s.view(torch.int32))
    assert torch.equal(out_l.view(torch.int16), out_s.view(torch.int16)), \
        f"{(out_l != out_s).sum().item()} elements differ"
    check_output(out_l, oracle.moe_forward(inp, cfg.k, cfg.score_fn)["out"], cfg.name)


def test_layer_launch_decode_full_size_and_repeats(moe):
    cfg = wl.CONFIGS["decode"]
    assert layer_applies(moe, cfg)
    x = wl.make_inputs(cfg, seed=0, device="cuda")
    layer, out0, *_ = run_layer(moe, cfg, x, 2)
    out0 = out0.clone()
    _, out_s, *_ = run_layer(moe, cfg, x, 0)
    assert torch.equal(out0.view(torch.int16), out_s.view(torch.int16))
    out = torch.empty_like(out0)
    differ = torch.zeros((), dtype=torch.int64, device=out.device)
    with moe.expert_fusion(2):
        for _ in range(100):
            layer.forward(x["hidden"], x["logits"], out=out)
            differ += (out.view(torch.int16) != out0.view(torch.int16)).any().to(torch.int64)
        st = moe.device_status(layer.workspace(cfg.T))
    assert st == moe.MOE_OK, moe.status_string(st)
    assert int(differ) == 0


def test_layer_launch_applies_only_to_decode_sized_batches(moe):
    with moe.expert_fusion(2):
        assert moe.launch_count(moe.make_dims(**wl.CONFIGS["decode"].dims())) == 1
        # more than 256 experts, or more than 2048 (token, slot) pairs: separate launches
        assert moe.launch_count(moe.make_dims(**wl.CONFIGS["wide"].dims())) == 4
        assert moe.launch_count(moe.make_dims(**wl.CONFIGS["prefill"].dims())) == 5
        # the router variant keeps its own launches
        assert moe.launch_count_router(moe.make_dims(**wl.CONFIGS["decode"].dims())) == 4
