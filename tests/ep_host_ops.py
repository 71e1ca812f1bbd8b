"""Host stand-in for the expert-parallel local steps (test infrastructure).

The same contracts as LibMoeEPOps (dispatch, experts, combine on one rank),
computed on the CPU in float64 from the oracle's routing and numpy matrix
products, so that the exchange logic of ExpertParallelMoE can run across
gloo ranks without a GPU. Expert rows travel as fp32, as on the GPU path."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def _f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def swiglu_ffn(x, w_gate_up, w_down):
    """Rows x [n, H] through one SwiGLU expert (float64): W_down (silu(G x) * U x)."""
    I = w_gate_up.shape[0] // 2
    g = x @ w_gate_up[:I].T
    u = x @ w_gate_up[I:].T
    h = g / (1.0 + np.exp(-g)) * u
    return h @ w_down.T


class HostEPOps:
    def workspace(self, d, device, old=None):
        return {} if old is None else old

    def dispatch(self, d, hidden, logits, w_g, ws, stream=None):
        T, k, E = d.T, d.k, d.E
        ids, w = oracle.route(logits.numpy(), k, d.score_fn) if T else (
            np.zeros((0, k), np.int32), np.zeros((0, k)))
        flat = ids.ravel()
        perm = np.argsort(flat, kind="stable")
        inv = np.empty_like(perm)
        inv[perm] = np.arange(perm.size)
        x = _f64(hidden)
        gate = 1.0 / (1.0 + np.exp(-(x @ _f64(w_g)))) if T else np.zeros(0)
        ws.update(perm=perm, inv=inv, w=w, gate=gate)
        x_send = hidden[torch.as_tensor(perm // k, dtype=torch.long)].contiguous()
        counts = torch.from_numpy(np.bincount(flat, minlength=E).astype(np.int32))
        return x_send, counts

    def experts(self, d, R, x_recv, recv_counts, hidden, w_gate_up, w_down, ws_gate_up, ws_down,
                ws, stream=None):
        cnt = recv_counts.cpu().numpy()
        assert int(cnt.sum()) == R
        x = _f64(x_recv)
        wgu, wd = _f64(w_gate_up), _f64(w_down)
        y = np.zeros((R, d.H))
        row = 0
        for s in range(cnt.shape[0]):          # source ranks in order,
            for e in range(cnt.shape[1]):      # each sorted by local expert
                n = int(cnt[s, e])
                y[row:row + n] = swiglu_ffn(x[row:row + n], wgu[e], wd[e])
                row += n
        shared = swiglu_ffn(_f64(hidden), _f64(ws_gate_up), _f64(ws_down)) if d.T else np.zeros(
            (0, d.H))
        ws["y_shared"] = shared * ws["gate"][:, None]
        return torch.from_numpy(y.astype(np.float32))

    def combine(self, d, R, y_back, ws, stream=None):
        T, k = d.T, d.k
        if T == 0:
            return torch.zeros(0, d.H, dtype=torch.float64)
        y = _f64(y_back)
        inv = ws["inv"].reshape(T, k)
        acc = np.zeros((T, d.H))
        for j in range(k):   # slot order, then the shared row
            acc += ws["w"][:, j:j + 1] * y[inv[:, j]]
        return torch.from_numpy(acc + ws["y_shared"])
