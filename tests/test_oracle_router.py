"""Pins of the oracle's router (logits = hidden . W_router^T, fp32 router on
bf16 values), independent of the oracle's own loops."""
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


def check_hand_values(lib=None):
    # worked by hand: token 0 = (1, 2, -1, 1/2), token 1 = (0, 1, 0, 0)
    x = torch.tensor([[1, 2, -1, 0.5], [0, 1, 0, 0]], dtype=torch.bfloat16)
    w = torch.tensor([[1, 0, 0, 0], [0.5, 0.25, 2, -1], [1, 1, 1, 1]], dtype=torch.bfloat16)
    got = oracle.router_logits(x, w, lib)
    want = np.array([[1.0, 0.5 + 0.5 - 2.0 - 0.5, 1 + 2 - 1 + 0.5],
                     [0.0, 0.25, 1.0]])
    assert np.array_equal(got, want)


def check_one_hot_rows(lib=None):
    """A one-hot hidden row e_j picks column j of W_router exactly."""
    g = torch.Generator().manual_seed(1)
    E, H = 12, 40
    w = (torch.randn(E, H, generator=g) * 0.02).to(torch.bfloat16)
    cols = [0, 7, 39, 13]
    x = torch.zeros(len(cols), H, dtype=torch.bfloat16)
    for t, j in enumerate(cols):
        x[t, j] = 1.0
    got = oracle.router_logits(x, w, lib)
    assert np.array_equal(got, w.double().numpy()[:, cols].T)


def check_dense_matmul(lib=None):
    """Equals a float64 matrix product of the bf16 values (a library routine,
    not the oracle's loops), to the last bits of fp64 summation."""
    g = torch.Generator().manual_seed(2)
    T, E, H = 9, 33, 200
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, H, generator=g) * 0.02).to(torch.bfloat16)
    got = oracle.router_logits(x, w, lib)
    want = x.double().numpy() @ w.double().numpy().T
    assert np.max(np.abs(got - want)) <= 1e-12 * (np.abs(x.double().numpy()) @
                                                 np.abs(w.double().numpy()).T).max()


def check_routing_of_known_logits(lib=None):
    """W_router = 2^-3 times the first E unit vectors: the logits are the first
    E hidden values / 8, so the layer routes like a brute-force top-k on them."""
    cfg = wl.MoEConfig("r", T=10, H=64, E=16, k=3, I=64, I_s=64, score_fn=wl.SOFTMAX)
    inp = wl.make_inputs_router(cfg, seed=3)
    w = torch.zeros(cfg.E, cfg.H)
    w[torch.arange(cfg.E), torch.arange(cfg.E)] = 0.125
    inp["w_router"] = w.to(torch.bfloat16)
    res = oracle.moe_forward_router(inp, cfg.k, cfg.score_fn, lib_path=lib)
    lg = inp["hidden"].double().numpy()[:, :cfg.E] / 8
    for t in range(cfg.T):
        # descending value, ties to the lower index, by counting
        rank = [sum(1 for f in range(cfg.E) if lg[t, f] > lg[t, e] or (lg[t, f] == lg[t, e] and f < e))
                for e in range(cfg.E)]
        want = sorted(range(cfg.E), key=lambda e: rank[e])[:cfg.k]
        assert list(res["ids"][t]) == want


CHECKS = [check_hand_values, check_one_hot_rows, check_dense_matmul,
          check_routing_of_known_logits]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_router_pin(check):
    check()


SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

MUTANTS = {
    "w_router_transposed": [("bf16_value(w_router[(size_t)e * H + h]);",
                             "bf16_value(w_router[(size_t)h * E + e]);")],
    "last_term_dropped": [("            for (int h = 0; h < H; ++h)\n                acc += bf16_value(hidden",
                           "            for (int h = 0; h < H - 1; ++h)\n                acc += bf16_value(hidden")],
    "token_stride": [("acc += bf16_value(hidden[(size_t)t * H + h]) *",
                      "acc += bf16_value(hidden[(size_t)t * E + h]) *")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_router_pins_catch_planted_mistake(name, tmp_path):
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
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
