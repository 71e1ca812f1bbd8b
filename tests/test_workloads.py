"""The seeded input generator: shapes, dtypes, determinism and the skew bias."""
import math

import torch

from mixture_experts_ffn_03_gb300 import workloads as wl


def test_shapes_dtypes_and_determinism():
    cfg = wl.CONFIGS["tiny"]
    a = wl.make_inputs(cfg, seed=0)
    b = wl.make_inputs(cfg, seed=0)
    c = wl.make_inputs(cfg, seed=1)
    T, H, E, I, I_s = cfg.T, cfg.H, cfg.E, cfg.I, cfg.I_s
    want = dict(hidden=(T, H), logits=(T, E), w_gate_up=(E, 2 * I, H), w_down=(E, H, I),
                ws_gate_up=(2 * I_s, H), ws_down=(H, I_s), w_g=(H,))
    for name, shape in want.items():
        assert tuple(a[name].shape) == shape, name
        assert a[name].is_contiguous()
        assert a[name].dtype == (torch.float32 if name == "logits" else torch.bfloat16)
        assert torch.equal(a[name], b[name])
    assert not torch.equal(a["hidden"], c["hidden"])


def test_distributions():
    cfg = wl.MoEConfig("probe", T=256, H=256, E=8, k=2, I=64, I_s=64, score_fn=wl.SOFTMAX)
    x = wl.make_inputs(cfg, seed=3)
    assert abs(x["hidden"].float().std().item() - 1.0) < 0.05
    assert abs(x["logits"].std().item() - 1.0) < 0.05
    assert abs(x["w_gate_up"].float().std().item() - 0.02) < 0.001
    assert abs(x["w_g"].float().std().item() - 0.02) < 0.005


def test_skew_bias():
    b = wl.skew_bias(5)
    for e in range(5):
        assert b[e].item() == torch.tensor(-2.0 * math.log(e + 1.0), dtype=torch.float32).item()
    cfg = wl.CONFIGS["skewed"].with_tokens(32)
    cfg = wl.MoEConfig("sk", T=32, H=64, E=16, k=2, I=64, I_s=64, score_fn=wl.SOFTMAX, skew=True)
    s = wl.make_inputs(cfg, seed=0)
    u = wl.make_inputs(wl.MoEConfig("u", T=32, H=64, E=16, k=2, I=64, I_s=64, score_fn=wl.SOFTMAX), seed=0)
    assert torch.equal(s["logits"], u["logits"] + wl.skew_bias(16))
