"""Independent brute-force evaluations used to pin the oracle on tiny inputs.

Nothing here is shared with the oracle: the selection is a rank count
(an O(E^2) formula with no sort and no repeated arg-max), and the layer is
evaluated densely over ALL experts with numpy float64 matmuls, then masked by
the renormalised routing weights.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact values of bf16 bit patterns."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even) via float32.

    Values used in the tests are exactly representable in float32, so the
    first rounding is exact."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def rank_select(row: np.ndarray, k: int) -> list[int]:
    """Experts with rank < k, in rank order. rank_e counts experts that rank
    before e: larger logit, or equal logit and lower index."""
    E = row.shape[0]
    rank = []
    for e in range(E):
        r = 0
        for j in range(E):
            if row[j] > row[e] or (row[j] == row[e] and j < e):
                r += 1
        rank.append(r)
    order = sorted(range(E), key=lambda e: rank[e])
    return [e for e in order if rank[e] < k]


def scores(row: np.ndarray, score_fn: int) -> np.ndarray:
    l = row.astype(np.float64)
    if score_fn == 0:
        z = np.exp(l - l.max())
        return z / z.sum()
    return 1.0 / (1.0 + np.exp(-l))


def dense_layer(inputs: dict, k: int, score_fn: int, gate_zero: bool = False) -> np.ndarray:
    """out[T,H] in float64: every expert evaluated for every token, then
    weighted by a mask that is zero off the selected set."""
    x_all = bf16_to_f64(inputs["hidden"])
    logits = np.asarray(inputs["logits"], dtype=np.float32)
    wgu = bf16_to_f64(inputs["w_gate_up"])
    wd = bf16_to_f64(inputs["w_down"])
    wsgu = bf16_to_f64(inputs["ws_gate_up"])
    wsd = bf16_to_f64(inputs["ws_down"])
    wg = bf16_to_f64(inputs["w_g"])
    T, H = x_all.shape
    E = logits.shape[1]
    I = wgu.shape[1] // 2
    I_s = wsgu.shape[0] // 2

    def silu(v):
        return v / (1.0 + np.exp(-v))

    out = np.zeros((T, H))
    for t in range(T):
        x = x_all[t]
        sel = rank_select(logits[t], k)
        s = scores(logits[t], score_fn)
        mask = np.zeros(E)
        mask[sel] = s[sel] / s[sel].sum()
        for e in range(E):
            h = silu(wgu[e, :I] @ x) * (wgu[e, I:] @ x)
            out[t] += mask[e] * (wd[e] @ h)
        hs = silu(wsgu[:I_s] @ x) * (wsgu[I_s:] @ x)
        gate = 0.0 if gate_zero else 1.0 / (1.0 + np.exp(-(wg @ x)))
        out[t] += gate * (wsd @ hs)
    return out
