"""Failure detection on the GPU without a GPU fault: a bounded barrier wait on
a flag nothing sets runs out, the kernel reports it in the workspace status
word, and the context stays usable for the next layer call."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_03_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_ffn_03_gb300 as moe
    moe.load_library()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    assert moe.selftest_wait_limit(ws) == moe.MOE_OK
    st = moe.device_status(ws)          # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert st == moe.MOE_ERR_DEVICE_TIMEOUT, moe.status_string(st)
    word = int(ws[:4].view(torch.int32).item()) & 0xFFFFFFFF
    assert word != 0 and (word & 0x80000000) == 0   # timed out, never "completed"
    assert 1.5 < elapsed < 30.0                      # the 2 s limit, not a hang

    # The context is still usable: a normal layer call matches the oracle.
    cfg = wl.CONFIGS["tiny"]
    inp = wl.make_inputs(cfg, seed=0)
    x = {n: t.to("cuda") for n, t in inp.items()}
    layer = moe.MoELayer(x["w_gate_up"], x["w_down"], x["ws_gate_up"], x["ws_down"], x["w_g"],
                         cfg.k, cfg.score_fn)
    out = layer.forward(x["hidden"], x["logits"])
    assert moe.device_status(layer.workspace(cfg.T)) == moe.MOE_OK
    ref = oracle.moe_forward(inp, cfg.k, cfg.score_fn)["out"]
    g = out.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    assert np.all(np.abs(g - ref) <= 1e-2 * np.abs(ref) + 1e-3 * rms)
