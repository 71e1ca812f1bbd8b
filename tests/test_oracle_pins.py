"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Every check is a function of a library path, so the same checks can be run
against deliberately broken builds of the oracle (test_oracle_mutants.py)
to show that a plausible mistake anywhere in it fails at least one of them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

import oracle
from brute_force import bf16_to_f64, dense_layer, f64_to_bf16_bits, rank_select, scores

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _expr(s):
    if isinstance(s, (int, float)):
        return float(s)
    env = {"e": math.e, "sig": lambda v: 1.0 / (1.0 + math.exp(-v)), "exp": math.exp,
           "log": math.log, "__builtins__": {}}
    return float(eval(s, env))  # expressions are fixed strings in tests/golden


def tiny_inputs(T, H, E, k, I, I_s, seed, ties=False, weight_scale=0.3):
    rng = np.random.default_rng(seed)
    if ties:
        logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    else:
        logits = rng.standard_normal((T, E)).astype(np.float32)
    return dict(
        hidden=f64_to_bf16_bits(rng.standard_normal((T, H))),
        logits=logits,
        w_gate_up=f64_to_bf16_bits(weight_scale * rng.standard_normal((E, 2 * I, H))),
        w_down=f64_to_bf16_bits(weight_scale * rng.standard_normal((E, H, I))),
        ws_gate_up=f64_to_bf16_bits(weight_scale * rng.standard_normal((2 * I_s, H))),
        ws_down=f64_to_bf16_bits(weight_scale * rng.standard_normal((H, I_s))),
        w_g=f64_to_bf16_bits(weight_scale * rng.standard_normal(H)),
    )


# ---------------------------------------------------------------- routing pins

def check_golden_routing(lib=None):
    cases = json.load(open(os.path.join(GOLDEN, "routing_cases.json")))
    for c in cases:
        lg = np.array(c["logits"], dtype=np.float32)
        ids, w = oracle.route(lg, c["k"], c["score_fn"], lib_path=lib)
        assert ids.tolist() == c["ids"], c["name"]
        want = np.array([[_expr(v) for v in row] for row in c["weights"]])
        assert np.max(np.abs(w - want)) <= c["tol"] * 4, c["name"]


def check_rank_bruteforce(lib=None):
    for seed, (E, k, ties) in enumerate([(16, 4, False), (16, 4, True), (8, 8, True),
                                          (33, 1, True), (64, 10, False), (7, 3, True)]):
        rng = np.random.default_rng(100 + seed)
        T = 40
        if ties:
            lg = rng.integers(-1, 2, size=(T, E)).astype(np.float32)
        else:
            lg = rng.standard_normal((T, E)).astype(np.float32)
        for score_fn in (oracle.SOFTMAX, oracle.SIGMOID):
            ids, _ = oracle.route(lg, k, score_fn, lib_path=lib)
            for t in range(T):
                assert ids[t].tolist() == rank_select(lg[t], k), (E, k, t)


def check_sum_to_one_and_closed_forms(lib=None):
    rng = np.random.default_rng(7)
    T, E, k = 64, 32, 6
    lg = (2.0 * rng.standard_normal((T, E))).astype(np.float32)
    for score_fn in (oracle.SOFTMAX, oracle.SIGMOID):
        ids, w = oracle.route(lg, k, score_fn, lib_path=lib)
        assert np.max(np.abs(w.sum(axis=1) - 1.0)) <= 1e-12
        assert np.all(np.diff(w, axis=1) <= 1e-15), "weights follow the descending-logit order"
        sel = np.take_along_axis(lg.astype(np.float64), ids.astype(np.int64), axis=1)
        if score_fn == oracle.SOFTMAX:
            # Closed form: renormalised softmax over E == softmax over the k selected logits.
            z = np.exp(sel - sel.max(axis=1, keepdims=True))
            want = z / z.sum(axis=1, keepdims=True)
        else:
            s = 1.0 / (1.0 + np.exp(-sel))
            want = s / s.sum(axis=1, keepdims=True)
        assert np.max(np.abs(w - want)) <= 1e-13


def check_k_equals_E(lib=None):
    rng = np.random.default_rng(8)
    T, E = 20, 12
    lg = rng.standard_normal((T, E)).astype(np.float32)
    for score_fn in (oracle.SOFTMAX, oracle.SIGMOID):
        ids, w = oracle.route(lg, E, score_fn, lib_path=lib)
        for t in range(T):
            full = np.zeros(E)
            full[ids[t]] = w[t]
            l = lg[t].astype(np.float64)
            if score_fn == oracle.SOFTMAX:
                want = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
            else:
                s = 1.0 / (1.0 + np.exp(-l))
                want = s / s.sum()
            assert np.max(np.abs(full - want)) <= 1e-13
            assert sorted(ids[t].tolist()) == list(range(E))


def check_counts(lib=None):
    rng = np.random.default_rng(9)
    T, E, k = 50, 20, 5
    lg = rng.integers(-1, 2, size=(T, E)).astype(np.float32)
    ids, _ = oracle.route(lg, k, oracle.SOFTMAX, lib_path=lib)
    counts = oracle.expert_counts(ids, E, lib_path=lib)
    want = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for e in rank_select(lg[t], k):
            want[e] += 1
    assert counts.tolist() == want.tolist()
    assert counts.sum() == T * k


# ------------------------------------------------------------------ layer pins

def check_golden_layer(lib=None):
    cases = json.load(open(os.path.join(GOLDEN, "layer_cases.json")))
    for c in cases:
        inp = dict(
            hidden=f64_to_bf16_bits(np.array(c["hidden"])),
            logits=np.array(c["logits"], dtype=np.float32),
            w_gate_up=f64_to_bf16_bits(np.array(c["w_gate_up"])),
            w_down=f64_to_bf16_bits(np.array(c["w_down"])),
            ws_gate_up=f64_to_bf16_bits(np.array(c["ws_gate_up"])),
            ws_down=f64_to_bf16_bits(np.array(c["ws_down"])),
            w_g=f64_to_bf16_bits(np.array(c["w_g"])),
        )
        r = oracle.moe_forward(inp, c["k"], c["score_fn"], lib_path=lib)
        want = np.array([[_expr(v) for v in row] for row in c["out"]])
        assert np.max(np.abs(r["out"] - want)) <= c["tol"], c["name"]
        assert np.max(np.abs(r["gate"] - np.array([_expr(v) for v in c["gate"]]))) <= c["tol"]


def check_dense_swiglu_e1_k1(lib=None):
    """E = 1, k = 1 with the shared down projection zeroed is a dense SwiGLU
    FFN; numpy float64 matmul gives it independently."""
    T, H, I = 6, 24, 10
    inp = tiny_inputs(T, H, 1, 1, I, 4, seed=11)
    inp["ws_down"] = np.zeros_like(inp["ws_down"])
    r = oracle.moe_forward(inp, 1, oracle.SOFTMAX, lib_path=lib)
    x = bf16_to_f64(inp["hidden"])
    w = bf16_to_f64(inp["w_gate_up"])[0]
    wd = bf16_to_f64(inp["w_down"])[0]
    g = x @ w[:I].T
    u = x @ w[I:].T
    want = ((g / (1.0 + np.exp(-g))) * u) @ wd.T
    assert np.all(r["ids"] == 0) and np.all(r["weights"] == 1.0)
    assert np.max(np.abs(r["out"] - want)) <= 1e-12 * max(1.0, np.abs(want).max())


def check_dense_masked(lib=None):
    for seed, (T, H, E, k, I, I_s, ties, sf) in enumerate([
            (5, 16, 8, 3, 8, 4, False, 0), (4, 12, 6, 2, 5, 7, True, 1),
            (3, 8, 4, 4, 4, 4, False, 1), (6, 10, 9, 1, 3, 2, True, 0)]):
        inp = tiny_inputs(T, H, E, k, I, I_s, seed=20 + seed, ties=ties)
        r = oracle.moe_forward(inp, k, sf, lib_path=lib)
        want = dense_layer(inp, k, sf)
        scale = max(1.0, np.abs(want).max())
        assert np.max(np.abs(r["out"] - want)) <= 1e-12 * scale, (T, H, E, k)


def check_gate_cases(lib=None):
    T, H, E, k, I, I_s = 4, 16, 6, 2, 8, 8
    inp = tiny_inputs(T, H, E, k, I, I_s, seed=31)
    # w_g = 0: the gate is sigmoid(0) = 1/2 exactly.
    z = dict(inp, w_g=np.zeros_like(inp["w_g"]))
    r = oracle.moe_forward(z, k, oracle.SOFTMAX, lib_path=lib)
    assert np.all(r["gate"] == 0.5)
    # gate forced to 0 removes the shared term: equals the dense routed-only sum.
    r0 = oracle.moe_forward(inp, k, oracle.SOFTMAX, gate_override=np.zeros(T), lib_path=lib)
    want = dense_layer(inp, k, oracle.SOFTMAX, gate_zero=True)
    assert np.max(np.abs(r0["out"] - want)) <= 1e-12 * max(1.0, np.abs(want).max())
    # zero shared down projection removes the term as well.
    zs = dict(inp, ws_down=np.zeros_like(inp["ws_down"]))
    r1 = oracle.moe_forward(zs, k, oracle.SOFTMAX, lib_path=lib)
    assert np.max(np.abs(r1["out"] - r0["out"])) <= 1e-12 * max(1.0, np.abs(want).max())
    # the gate value itself: sigmoid of x . w_g
    x = bf16_to_f64(inp["hidden"])
    want_gate = 1.0 / (1.0 + np.exp(-(x @ bf16_to_f64(inp["w_g"]))))
    r2 = oracle.moe_forward(inp, k, oracle.SOFTMAX, lib_path=lib)
    assert np.max(np.abs(r2["gate"] - want_gate)) <= 1e-14


def check_linearity_in_w_down(lib=None):
    """Doubling every W_down (exact in bf16) doubles the routed part."""
    T, H, E, k, I, I_s = 5, 16, 6, 3, 8, 8
    inp = tiny_inputs(T, H, E, k, I, I_s, seed=41)
    g0 = np.zeros(T)
    a = oracle.moe_forward(inp, k, oracle.SIGMOID, gate_override=g0, lib_path=lib)["out"]
    wd2 = f64_to_bf16_bits(2.0 * bf16_to_f64(inp["w_down"]))
    b = oracle.moe_forward(dict(inp, w_down=wd2), k, oracle.SIGMOID, gate_override=g0,
                           lib_path=lib)["out"]
    assert np.max(np.abs(b - 2.0 * a)) <= 1e-12 * max(1.0, np.abs(a).max())


def check_token_permutation(lib=None):
    T, H, E, k, I, I_s = 9, 16, 8, 3, 8, 8
    inp = tiny_inputs(T, H, E, k, I, I_s, seed=51)
    perm = np.random.default_rng(5).permutation(T)
    p = dict(inp, hidden=inp["hidden"][perm], logits=inp["logits"][perm])
    a = oracle.moe_forward(inp, k, oracle.SOFTMAX, lib_path=lib)["out"]
    b = oracle.moe_forward(p, k, oracle.SOFTMAX, lib_path=lib)["out"]
    assert np.array_equal(a[perm], b)
    # the token-subset mode evaluates the same rows
    sub = np.array([4, 0, 7])
    c = oracle.moe_forward(inp, k, oracle.SOFTMAX, tokens=sub, lib_path=lib)["out"]
    assert np.array_equal(c, a[sub])


def check_expert_relabel(lib=None):
    T, H, E, k, I, I_s = 6, 16, 8, 3, 8, 8
    inp = tiny_inputs(T, H, E, k, I, I_s, seed=61)
    q = np.random.default_rng(6).permutation(E)
    p = dict(inp, logits=inp["logits"][:, q], w_gate_up=inp["w_gate_up"][q],
             w_down=inp["w_down"][q])
    a = oracle.moe_forward(inp, k, oracle.SIGMOID, lib_path=lib)
    b = oracle.moe_forward(p, k, oracle.SIGMOID, lib_path=lib)
    assert np.array_equal(q[b["ids"]], a["ids"])  # no ties in continuous logits
    assert np.max(np.abs(a["out"] - b["out"])) <= 1e-12 * max(1.0, np.abs(a["out"]).max())


ALL_CHECKS = [check_golden_routing, check_rank_bruteforce, check_sum_to_one_and_closed_forms,
              check_k_equals_E, check_counts, check_golden_layer, check_dense_swiglu_e1_k1,
              check_dense_masked, check_gate_cases, check_linearity_in_w_down,
              check_token_permutation, check_expert_relabel]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()
