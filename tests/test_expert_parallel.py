"""Expert parallelism (mixture_experts_ffn_03_gb300.expert_parallel).

Host tests: the exchange logic of ExpertParallelMoE across world_size-2 gloo
ranks on the CPU, and the in-process exchange of G ranks, both with the local
steps computed on the host in float64 (tests/ep_host_ops.py), against the
single-GPU layer of the fp64 oracle on every rank's tokens. GPU tests: G
ranks emulated one after another on one GPU with the library's kernels
(moe_ep_dispatch, moe_ep_experts, moe_ep_combine) against the oracle, within
the parity tolerance, and the device-side check of inconsistent counts."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from ep_host_ops import HostEPOps
from mixture_experts_ffn_03_gb300 import expert_parallel as ep
from mixture_experts_ffn_03_gb300 import workloads as wl


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def make_case(T_ranks, E, k, score_fn, seed, H=64, I=64, I_s=128, bias=None):
    """One workload over all ranks' tokens (concatenated in rank order)."""
    cfg = wl.MoEConfig("ep", T=sum(T_ranks), H=H, E=E, k=k, I=I, I_s=I_s, score_fn=score_fn)
    inp = wl.make_inputs(cfg, seed=seed)
    if bias is not None:
        inp["logits"] = inp["logits"] + torch.as_tensor(bias, dtype=torch.float32)
    return cfg, inp


def rank_layer(inp, g, G, E, k, score_fn, max_tokens, ops):
    e_loc = E // G
    return ep.ExpertParallelMoE(g, G, inp["w_gate_up"][g * e_loc:(g + 1) * e_loc],
                                inp["w_down"][g * e_loc:(g + 1) * e_loc], inp["ws_gate_up"],
                                inp["ws_down"], inp["w_g"], E, k, score_fn, max_tokens, ops=ops)


def token_slices(T_ranks):
    starts = np.concatenate([[0], np.cumsum(T_ranks)])
    return [slice(int(starts[r]), int(starts[r + 1])) for r in range(len(T_ranks))]


def test_send_splits_by_hand():
    # E = 6 experts on G = 3 ranks: experts {0,1}, {2,3}, {4,5}
    assert ep.send_splits([1, 2, 0, 0, 5, 1], 3) == [3, 0, 6]
    assert ep.send_splits([4], 1) == [4]


# (T per rank, E, k, score, logit bias): plain; every token on rank 0's experts
# (rank 1 receives nothing); a rank without tokens.
SCENARIOS = [
    ([17, 9], 8, 3, wl.SOFTMAX, None),
    ([12, 7], 8, 2, wl.SIGMOID, [40.0] * 4 + [0.0] * 4),
    ([0, 11], 6, 2, wl.SOFTMAX, None),
]


@pytest.mark.parametrize("G", [1, 2, 4])
def test_local_exchange_matches_oracle(G):
    T_ranks = [5, 0, 9, 3][:G] if G > 1 else [14]
    E, k = 8, 3
    cfg, inp = make_case(T_ranks, E, k, wl.SOFTMAX, seed=31)
    layers = [rank_layer(inp, g, G, E, k, cfg.score_fn, max(T_ranks), HostEPOps())
              for g in range(G)]
    sl = token_slices(T_ranks)
    outs = ep.LocalExchange(layers).forward([inp["hidden"][s] for s in sl],
                                            [inp["logits"][s] for s in sl])
    ref = oracle.moe_forward(inp, k, cfg.score_fn)["out"]
    for r, s in enumerate(sl):
        got = outs[r].numpy()
        assert got.shape == (T_ranks[r], cfg.H)
        # expert rows travel as fp32: relative error ~1e-7
        np.testing.assert_allclose(got, ref[s], rtol=2e-6, atol=2e-6 * np.abs(ref).max())


def _gloo_rank(rank, world, port, scenario, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T_ranks, E, k, score_fn, bias = scenario
        cfg, inp = make_case(T_ranks, E, k, score_fn, seed=23, bias=bias)
        layer = rank_layer(inp, rank, world, E, k, score_fn, max(T_ranks), HostEPOps())
        s = token_slices(T_ranks)[rank]
        got = layer.forward(inp["hidden"][s], inp["logits"][s])
        out[rank] = got.numpy().tolist()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("scenario", SCENARIOS, ids=["plain", "one_rank_idle", "rank_no_tokens"])
def test_gloo_two_ranks_match_oracle(scenario):
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_gloo_rank, args=(world, _free_port(), scenario, out), nprocs=world,
                           join=True, start_method="spawn")
        got = dict(out)
    T_ranks, E, k, score_fn, bias = scenario
    cfg, inp = make_case(T_ranks, E, k, score_fn, seed=23, bias=bias)
    ref = oracle.moe_forward(inp, k, score_fn)["out"]
    for r, s in enumerate(token_slices(T_ranks)):
        g = np.asarray(got[r], dtype=np.float64).reshape(T_ranks[r], cfg.H)
        np.testing.assert_allclose(g, ref[s], rtol=2e-6, atol=2e-6 * np.abs(ref).max())


# ------------------------------------------------------------------ GPU
REL_TOL, RMS_TOL = 1e-2, 1e-3


def check_tol(got, ref, label):
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(got - ref)
    bad = err > REL_TOL * np.abs(ref) + RMS_TOL * rms
    assert not bad.any(), f"{label}: {int(bad.sum())} of {bad.size} elements outside tolerance"


@pytest.mark.gpu
@pytest.mark.parametrize("G,T_ranks,E,k,I", [
    (1, [64], 16, 4, 128),
    (2, [40, 25], 16, 4, 128),
    (4, [30, 0, 17, 50], 32, 6, 192),
    (4, [300, 280, 310, 260], 32, 8, 128),   # larger groups: wider tiles
])
def test_gpu_emulated_ranks_match_oracle(G, T_ranks, E, k, I):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    cfg, inp = make_case(T_ranks, E, k, wl.SIGMOID, seed=41, H=256, I=I, I_s=192)
    x = {n: t.to(dev) for n, t in inp.items()}
    layers = [rank_layer(x, g, G, E, k, cfg.score_fn, max(T_ranks), None) for g in range(G)]
    sl = token_slices(T_ranks)
    outs = ep.LocalExchange(layers).forward([x["hidden"][s] for s in sl],
                                            [x["logits"][s] for s in sl])
    torch.cuda.synchronize()
    import mixture_experts_ffn_03_gb300 as moe
    for layer in layers:
        assert moe.device_status(layer._ws) == moe.MOE_OK
    ref = oracle.moe_forward(inp, k, cfg.score_fn)["out"]
    for r, s in enumerate(sl):
        check_tol(outs[r].float().cpu().numpy().astype(np.float64), ref[s], f"rank {r}")


@pytest.mark.gpu
def test_gpu_inconsistent_counts_are_reported():
    """Counts that do not add up to the received rows: no received row is
    processed and the device status reports an invalid argument (no fault)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_ffn_03_gb300 as moe
    dev = torch.device("cuda")
    T_ranks, E, k = [20], 8, 2
    cfg, inp = make_case(T_ranks, E, k, wl.SOFTMAX, seed=5, H=128, I=64, I_s=64)
    x = {n: t.to(dev) for n, t in inp.items()}
    layer = rank_layer(x, 0, 1, E, k, cfg.score_fn, 20, None)
    disp = layer.step_dispatch(x["hidden"], x["logits"])
    bad = disp.counts.view(1, E).clone()
    bad[0, 0] += 1   # one row more than sent
    layer.step_experts(disp.T, disp.x_send, bad)
    assert moe.device_status(layer._ws) == moe.MOE_ERR_INVALID_ARG
    # the workspace is usable again on the next step
    out = ep.LocalExchange([layer]).forward([x["hidden"]], [x["logits"]])[0]
    assert moe.device_status(layer._ws) == moe.MOE_OK
    check_tol(out.float().cpu().numpy().astype(np.float64),
              oracle.moe_forward(inp, k, cfg.score_fn)["out"], "after the bad step")
