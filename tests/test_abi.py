"""The C-ABI library: it builds, loads without a GPU, exports every entry point
declared in include/moe.h, and rejects bad arguments on the host before any
CUDA call (none of these tests touches a GPU)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from mixture_experts_ffn_03_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    import mixture_experts_ffn_03_gb300 as moe
    return moe.load_library()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    import mixture_experts_ffn_03_gb300 as moe
    names = declared_functions()
    assert set(moe.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_size_and_layout():
    import mixture_experts_ffn_03_gb300 as moe
    from mixture_experts_ffn_03_gb300.workloads import CONFIGS
    for cfg in CONFIGS.values():
        d = moe.make_dims(**cfg.dims())
        n = moe.workspace_size(d)
        L = moe.workspace_layout(d)
        assert n == L.total > 0
        tk = cfg.T * cfg.k
        assert L.y + (tk + cfg.T) * cfg.H * 4 <= n
        offs = [L.topk_ids, L.topk_w, L.gate_logit, L.counts, L.offsets, L.perm, L.inv, L.h_hi,
                L.h_lo, L.hs_hi, L.hs_lo, L.y]
        assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert moe.workspace_size(moe.make_dims(16, 128, 16, 17, 64, 64, 0)) == 0  # k > E


def _call(lib, dims, **kw):
    import mixture_experts_ffn_03_gb300 as moe
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: the checks below fail first
    args = dict(hidden=fake, logits=fake, wgu=fake, wd=fake, wsgu=fake, wsd=fake, wg=fake,
                out=fake, ids=None, w=None, counts=None, ws=fake, ws_bytes=1 << 40, stream=None)
    args.update(kw)
    return lib.moe_forward(ctypes.byref(dims), args["hidden"], args["logits"], args["wgu"],
                           args["wd"], args["wsgu"], args["wsd"], args["wg"], args["out"],
                           args["ids"], args["w"], args["counts"], args["ws"],
                           ctypes.c_size_t(args["ws_bytes"]), args["stream"])


def test_host_validation(lib):
    import mixture_experts_ffn_03_gb300 as moe
    ok = moe.make_dims(16, 128, 16, 4, 64, 64, 0)
    assert _call(lib, moe.make_dims(16, 128, 16, 0, 64, 64, 0)) == 1      # k < 1
    assert _call(lib, moe.make_dims(16, 128, 16, 17, 64, 64, 0)) == 1     # k > E
    assert _call(lib, moe.make_dims(16, 128, 2048, 4, 64, 64, 0)) == 1    # E > 1024
    assert _call(lib, moe.make_dims(16, 128, 64, 33, 64, 64, 0)) == 1     # k > 32
    assert _call(lib, moe.make_dims(-1, 128, 16, 4, 64, 64, 0)) == 1      # T < 0
    assert _call(lib, moe.make_dims(16, 128, 16, 4, 64, 64, 2)) == 1      # score fn
    assert _call(lib, moe.make_dims(16, 96, 16, 4, 64, 64, 0)) == 2       # H % 64
    assert _call(lib, moe.make_dims(16, 128, 16, 4, 80, 64, 0)) == 2      # I % 64
    assert _call(lib, moe.make_dims(16, 128, 16, 4, 64, 32, 0)) == 2      # I_s % 64
    assert _call(lib, ok, hidden=None) == 1                                # null input
    assert _call(lib, ok, out=ctypes.c_void_p((1 << 20) + 8)) == 1         # misaligned
    assert _call(lib, ok, ws=None) == 3                                    # no workspace
    assert _call(lib, ok, ws_bytes=moe.workspace_size(ok) - 1) == 3        # too small
    assert _call(lib, ok, ws=ctypes.c_void_p((1 << 20) + 64)) == 3         # ws alignment
    assert _call(lib, moe.make_dims(0, 128, 16, 4, 64, 64, 0)) == 0        # T = 0: no work
    for s in range(7):
        assert moe.status_string(s)
    decode = moe.make_dims(64, 2048, 256, 8, 512, 512, 1)
    assert not moe.get_expert_fusion()                                      # off by default
    assert moe.launch_count(decode) == 4                                    # T*k <= 2048
    assert moe.launch_count_router(decode) == 5
    with moe.expert_fusion(True):
        assert moe.get_expert_fusion()
        assert moe.launch_count(decode) == 3  # one routing launch, fused experts, combine
        assert moe.launch_count_router(decode) == 4
        assert moe.launch_count_quantized(decode) == 4                      # never fused
        assert moe.launch_count(moe.make_dims(4096, 2048, 256, 8, 512, 512, 0)) == 5  # BN 160/128
        assert moe.launch_count(moe.make_dims(512, 2048, 256, 8, 512, 512, 0)) == 4   # BN 32/32
    with moe.expert_fusion(2):
        assert moe.get_expert_fusion() == 2
        assert moe.launch_count(decode) == 1               # the whole layer in one launch
        assert moe.launch_count_router(decode) == 4        # the router variant is not folded
        assert moe.launch_count(moe.make_dims(64, 2048, 512, 8, 512, 512, 1)) == 3  # E > 256
    assert not moe.get_expert_fusion()
    assert moe.launch_count(moe.make_dims(4096, 2048, 256, 8, 512, 512, 0)) == 5
    assert moe.launch_count(moe.make_dims(0, 2048, 256, 8, 512, 512, 0)) == 0
    assert moe.launch_count_quantized(moe.make_dims(64, 2048, 256, 8, 192, 512, 1)) == 0


def _call_mx(lib, dims, **kw):
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: the checks below fail first
    names = ["hidden", "logits", "gu_q", "gu_s", "d_q", "d_s", "sgu_q", "sgu_s", "sd_q", "sd_s",
             "wg", "out"]
    args = {n: fake for n in names}
    args.update(ids=None, w=None, counts=None, ws=fake, ws_bytes=1 << 40, stream=None)
    args.update(kw)
    return lib.moe_forward_mxfp8(ctypes.byref(dims), *[args[n] for n in names], args["ids"],
                                 args["w"], args["counts"], args["ws"],
                                 ctypes.c_size_t(args["ws_bytes"]), args["stream"])


def test_host_validation_mxfp8(lib):
    import mixture_experts_ffn_03_gb300 as moe
    ok = moe.make_dims(16, 128, 16, 4, 128, 128, 0)
    assert _call_mx(lib, moe.make_dims(16, 128, 16, 0, 128, 128, 0)) == 1    # k < 1
    assert _call_mx(lib, moe.make_dims(16, 64, 16, 4, 128, 128, 0)) == 2     # H % 128
    assert _call_mx(lib, moe.make_dims(16, 128, 16, 4, 192, 128, 0)) == 2    # I % 128
    assert _call_mx(lib, moe.make_dims(16, 128, 16, 4, 128, 64, 0)) == 2     # I_s % 128
    assert _call_mx(lib, ok, d_s=None) == 1                                   # null scales
    assert _call_mx(lib, ok, sgu_s=ctypes.c_void_p((1 << 20) + 4)) == 1      # misaligned scales
    assert _call_mx(lib, ok, ws=None) == 3                                    # no workspace
    assert _call_mx(lib, moe.make_dims(0, 128, 16, 4, 128, 128, 0)) == 0     # T = 0: no work
    fake = ctypes.c_void_p(1 << 20)
    assert lib.moe_mxfp8_dequant(fake, fake, 4, 48, fake, None) == 1         # cols % 32
    assert lib.moe_mxfp8_dequant(fake, fake, 0, 64, fake, None) == 0         # nothing to do
    assert lib.moe_mxfp8_dequant(None, fake, 4, 64, fake, None) == 1         # null codes


def test_host_validation_router(lib):
    import mixture_experts_ffn_03_gb300 as moe
    P = ctypes.c_void_p
    fake = P(1 << 20)
    ok = moe.make_dims(16, 128, 16, 4, 64, 64, 0)

    def call(dims, w_router=fake, ws_bytes=1 << 40, logits_out=None):
        return lib.moe_forward_router(ctypes.byref(dims), fake, w_router, fake, fake, fake, fake,
                                      fake, fake, logits_out, None, None, None, fake,
                                      ctypes.c_size_t(ws_bytes), None)
    assert call(ok, w_router=None) == 1                                       # no router weights
    assert call(ok, logits_out=P((1 << 20) + 4)) == 1                         # misaligned logits
    assert call(ok, ws_bytes=moe.workspace_size(ok)) == 3                     # plain size too small
    assert call(moe.make_dims(16, 96, 16, 4, 64, 64, 0)) == 2                 # H % 64
    assert call(moe.make_dims(0, 128, 16, 4, 64, 64, 0)) == 0                 # T = 0
    assert moe.workspace_size_router(ok) > moe.workspace_size(ok)


def test_host_validation_nvfp4(lib):
    import mixture_experts_ffn_03_gb300 as moe
    P = ctypes.c_void_p
    fake = P(1 << 20)
    ok = moe.make_dims(16, 128, 16, 4, 128, 128, 0)

    def call(dims, **kw):
        args = [fake] * 16
        for i, v in kw.items():
            args[int(i[1:])] = v
        return lib.moe_forward_nvfp4(ctypes.byref(dims), *args, None, None, None, fake,
                                     ctypes.c_size_t(1 << 40), None)
    assert call(moe.make_dims(16, 64, 16, 4, 128, 128, 0)) == 2              # H % 128
    assert call(ok, a4=None) == 1                                             # no gate/up matrix scales
    assert call(ok, a4=P((1 << 20) + 2)) == 1                                 # misaligned matrix scales
    assert call(ok, a3=P((1 << 20) + 8)) == 1                                 # misaligned block scales
    assert call(moe.make_dims(0, 128, 16, 4, 128, 128, 0)) == 0               # T = 0
    assert lib.moe_nvfp4_dequant(fake, fake, 4, 48, fake, None) == 1          # cols % 32


def _tile_width(tk, E, cap, gate_up):
    """Token-tile width rule as documented in moe_api.cu: the smallest
    supported width >= 1.25x the mean group size, capped; 160 for gate_up only."""
    mean = tk / E
    bn = 16
    for w in (16, 32, 64, 128, 160, 256):
        if w > cap or (w == 160 and not gate_up):
            continue
        bn = w
        if w >= 1.25 * mean:
            break
    return bn


def test_expert_fusion_applies_exactly_when_tile_widths_match(lib):
    import itertools
    import mixture_experts_ffn_03_gb300 as moe
    for T, E, k in itertools.product((1, 7, 64, 300, 512, 2048, 4096), (8, 64, 256, 512),
                                     (1, 2, 8)):
        if k > E:
            continue
        d = moe.make_dims(T, 256, E, k, 128, 128, 0)
        tk = T * k
        gu, dn = _tile_width(tk, E, 256, True), _tile_width(tk, E, 128, False)
        with moe.expert_fusion(True):
            on = moe.launch_count(d)
        off = moe.launch_count(d)
        assert on == off - (1 if gu == dn and gu <= 64 else 0), (T, E, k, gu, dn)


def test_expert_fusion_setting_is_per_host_thread(lib):
    import threading
    import mixture_experts_ffn_03_gb300 as moe
    seen = []
    with moe.expert_fusion(True):
        t = threading.Thread(target=lambda: seen.append(moe.get_expert_fusion()))
        t.start()
        t.join()
        assert moe.get_expert_fusion()
    assert seen == [False]


def test_pipeline_rejects_bad_arguments_on_host(lib):
    """The host-memory serving loop checks its arguments before allocating or
    enqueueing anything."""
    import mixture_experts_ffn_03_gb300 as moe
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced
    h = P()
    d = moe.make_dims(16, 128, 16, 4, 64, 64, 0)
    create = lib.moe_pipeline_create
    assert create(ctypes.byref(d), fake, fake, fake, fake, fake, None, None) == moe.MOE_ERR_INVALID_ARG
    for i in range(5):
        w = [fake] * 5
        w[i] = None
        assert create(ctypes.byref(d), *w, None, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
        assert h.value is None
    for bad in (moe.make_dims(0, 128, 16, 4, 64, 64, 0), moe.make_dims(16, 128, 16, 17, 64, 64, 0)):
        assert create(ctypes.byref(bad), *([fake] * 5), None, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
        assert h.value is None
    assert create(None, *([fake] * 5), None, ctypes.byref(h)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_pipeline_submit(None, fake, fake, fake) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_pipeline_drain(None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_pipeline_streams(None, None, None) == moe.MOE_ERR_INVALID_ARG
    lib.moe_pipeline_destroy(None)  # a no-op

