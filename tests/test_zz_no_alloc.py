"""moe_expert_counts_static: the allocation-free expert histogram.

It serves callers that cannot allocate device memory (no workspace can be
passed to them, or cudaMalloc is not allowed where they run); its scratch is
a fixed array inside the library. These tests call it through the C ABI on
consecutive calls that share the fixed scratch, and compare it with
moe_forward's own per-expert counts and offsets for the same routing and
with a numpy histogram of the ids (computed on the host, independent of
the GPU code).
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_ffn_03_gb300 import build as moe_build
from mixture_experts_ffn_03_gb300 import workloads as wl

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_CAPACITY = 0, 1, 6
STATIC_HIST_WORDS = 1 << 18


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    import mixture_experts_ffn_03_gb300 as moe
    lib = moe.load_library()
    f = lib.moe_expert_counts_static
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def call_static(lib, ids, T, k, E, counts, offsets, stream):
    return lib.moe_expert_counts_static(
        ctypes.c_void_p(ids.data_ptr()) if ids is not None else None, T, k, E,
        ctypes.c_void_p(counts.data_ptr()) if counts is not None else None,
        ctypes.c_void_p(offsets.data_ptr()) if offsets is not None else None,
        ctypes.c_void_p(stream.cuda_stream) if stream is not None else None)


def test_rejects_oversize_and_bad_args_on_host(lib):
    # Checked before any device work: no GPU needed.
    fake = ctypes.c_void_p(1 << 20)
    f = lib.moe_expert_counts_static
    too_many_tokens = (STATIC_HIST_WORDS // 256 + 1) * 256  # E = 256: one block too many
    assert f(fake, too_many_tokens, 8, 256, fake, None, None) == MOE_ERR_CAPACITY
    assert f(fake, 16, 0, 16, fake, None, None) == MOE_ERR_INVALID_ARG
    assert f(fake, 16, 4, 2048, fake, None, None) == MOE_ERR_INVALID_ARG
    assert f(fake, 16, 4, 16, None, None, None) == MOE_ERR_INVALID_ARG
    # more experts per token than experts, and E = 1 with k = 32 (which would
    # otherwise let T * k reach 2^31 within the scratch capacity)
    assert f(fake, 16, 5, 4, fake, None, None) == MOE_ERR_INVALID_ARG
    assert f(fake, 1 << 26, 32, 1, fake, None, None) == MOE_ERR_INVALID_ARG
    assert f(fake, 16, 33, 64, fake, None, None) == MOE_ERR_INVALID_ARG


def reference_routing(moe, cfg, seed):
    """Routing, counts and offsets computed by the existing moe_forward."""
    inp = wl.make_inputs(cfg, seed=seed, device="cuda")
    layer = moe.MoELayer(inp["w_gate_up"], inp["w_down"], inp["ws_gate_up"], inp["ws_down"],
                         inp["w_g"], cfg.k, cfg.score_fn)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    layer.forward(inp["hidden"], inp["logits"], topk_ids=ids, counts=counts)
    assert moe.device_status(layer.workspace(cfg.T)) == MOE_OK
    L = moe.workspace_layout(layer.dims(cfg.T))
    ws = layer.workspace(cfg.T)
    offsets = ws[L.offsets:L.offsets + 4 * (cfg.E + 1)].view(torch.int32).clone()
    return ids, counts, offsets


def host_counts(ids, E):
    """Counts and exclusive offsets of a [T, k] id table, by numpy on the host."""
    c = np.bincount(ids.cpu().numpy().ravel(), minlength=E).astype(np.int32)
    return c, np.concatenate([[0], np.cumsum(c)]).astype(np.int32)


@pytest.mark.gpu
def test_static_counts_match_moe_forward_on_consecutive_calls(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_ffn_03_gb300 as moe
    stream = torch.cuda.current_stream()
    cases = [
        wl.CONFIGS["tiny"],
        wl.CONFIGS["skewed"].with_tokens(2048),
        # four experts per thread in the last block's scan (E = 1024), k = 32
        wl.MoEConfig("e1024_k32", T=700, H=64, E=1024, k=32, I=64, I_s=64, score_fn=wl.SOFTMAX),
        # E not a multiple of 256: two experts per thread, the last thread partly idle
        wl.MoEConfig("e300", T=1000, H=64, E=300, k=6, I=64, I_s=64, score_fn=wl.SIGMOID),
    ]
    for cfg in cases:
        ids, counts_ref, offsets_ref = reference_routing(moe, cfg, seed=3)
        c_host, o_host = host_counts(ids, cfg.E)
        assert np.array_equal(counts_ref.cpu().numpy(), c_host)
        assert np.array_equal(offsets_ref.cpu().numpy(), o_host)
        for _ in range(2):  # two calls in a row share the fixed scratch
            counts = torch.full((cfg.E,), -7, dtype=torch.int32, device="cuda")
            offsets = torch.full((cfg.E + 1,), -7, dtype=torch.int32, device="cuda")
            st = call_static(lib, ids, cfg.T, cfg.k, cfg.E, counts, offsets, stream)
            assert st == MOE_OK, moe.status_string(st)
            torch.cuda.synchronize()
            assert np.array_equal(counts.cpu().numpy(), c_host), cfg.name
            assert np.array_equal(offsets.cpu().numpy(), o_host), cfg.name
            assert torch.equal(counts, counts_ref)
            assert torch.equal(offsets, offsets_ref)
    # Zero tokens: all counts and offsets are zero.
    counts = torch.full((16,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((17,), -7, dtype=torch.int32, device="cuda")
    empty = torch.empty(0, 4, dtype=torch.int32, device="cuda")
    assert call_static(lib, empty, 0, 4, 16, counts, offsets, stream) == MOE_OK
    torch.cuda.synchronize()
    assert int(counts.abs().sum()) == 0 and int(offsets.abs().sum()) == 0
    assert np.all(offsets.cpu().numpy() == 0)
