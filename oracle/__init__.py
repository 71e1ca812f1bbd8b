"""CPU fp64 oracle of the MoE FFN layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. The library it wraps (``moe_oracle.c``) is plain C,
compiled with gcc; it shares no code with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None

SOFTMAX = 0
SIGMOID = 1


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", src, "-o", out + ".tmp",
               "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(out + ".tmp", out)
    return out


def _load(path: str | None = None):
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_route.argtypes = [i, i, i, i, P, P, P]
    lib.oracle_route.restype = i
    lib.oracle_expert_counts.argtypes = [i, i, i, P, P]
    lib.oracle_expert_counts.restype = None
    d = ctypes.c_double
    lib.oracle_moe_forward.argtypes = ([i, i, i, i, i, i, i] + [P] * 8 + [i] + [P] * 3 + [d, d] +
                                       [P] * 4 + [i])
    lib.oracle_mxfp8_to_bf16.argtypes = [i, i, P, P, P]
    lib.oracle_mxfp8_to_bf16.restype = i
    lib.oracle_e4m3_table.argtypes = [P]
    lib.oracle_router_logits.argtypes = [i, i, i, P, P, P]
    lib.oracle_nvfp4_to_bf16.argtypes = [i, i, P, P, P]
    lib.oracle_nvfp4_to_bf16.restype = i
    lib.oracle_e2m1_table.argtypes = [P]
    lib.oracle_router_logits.restype = None
    lib.oracle_moe_forward.restype = i
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """Accept a torch bf16 tensor or a numpy uint16 array of bf16 bits."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return a.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _f32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().contiguous().cpu().numpy()
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def route(logits, k: int, score_fn: int, lib_path: str | None = None):
    """Routing of every token: (ids [T,k] int32, weights [T,k] fp64)."""
    lib = _load(lib_path)
    lg = _f32(logits)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    bad = lib.oracle_route(T, E, k, score_fn, _ptr(lg), _ptr(ids), _ptr(w))
    assert bad == 0, f"{bad} tokens: fp64 score order contradicts the logit order"
    return ids, w


def expert_counts(ids, E: int, lib_path: str | None = None) -> np.ndarray:
    lib = _load(lib_path)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.empty(E, dtype=np.int32)
    lib.oracle_expert_counts(T, E, k, _ptr(ids), _ptr(counts))
    return counts


def moe_forward(inputs: dict, k: int, score_fn: int, tokens=None, gate_override=None,
                n_threads: int | None = None, lib_path: str | None = None):
    """Evaluate the layer in fp64 for ``tokens`` (default: all tokens).

    ``inputs`` holds hidden, logits, w_gate_up, w_down, ws_gate_up, ws_down,
    w_g (torch tensors or numpy bf16-bit arrays), and optionally the matrix
    scales w_gate_up_g / w_down_g [E] and ws_gate_up_g / ws_down_g (scalars)
    that multiply each matrix's dot products (NVFP4 weights; 1 if absent).
    Returns a dict with out [n,H] fp64, ids [n,k], weights [n,k] fp64 and
    gate [n] fp64.
    """
    lib = _load(lib_path)
    hidden = _u16(inputs["hidden"])
    logits = _f32(inputs["logits"])
    wgu = _u16(inputs["w_gate_up"])
    wd = _u16(inputs["w_down"])
    wsgu = _u16(inputs["ws_gate_up"])
    wsd = _u16(inputs["ws_down"])
    wg = _u16(inputs["w_g"])
    T, H = hidden.shape
    E = logits.shape[1]
    I = wgu.shape[1] // 2
    I_s = wsgu.shape[0] // 2
    assert wgu.shape == (E, 2 * I, H) and wd.shape == (E, H, I)
    assert wsgu.shape == (2 * I_s, H) and wsd.shape == (H, I_s) and wg.shape == (H,)
    if tokens is None:
        tok = None
        n = T
    else:
        tok = np.ascontiguousarray(tokens, dtype=np.int64)
        n = tok.shape[0]
        assert n == 0 or (tok.min() >= 0 and tok.max() < T)
    go = None if gate_override is None else np.ascontiguousarray(gate_override, dtype=np.float64)
    if go is not None:
        assert go.shape == (n,)
    def scales(name, shape):
        if name not in inputs:
            return None
        v = np.ascontiguousarray(np.asarray(_np(inputs[name]), dtype=np.float64).reshape(shape))
        return v
    s_gu, s_d = scales("w_gate_up_g", (E,)), scales("w_down_g", (E,))
    ss_gu, ss_d = scales("ws_gate_up_g", (1,)), scales("ws_down_g", (1,))
    out = np.empty((n, H), dtype=np.float64)
    ids = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k), dtype=np.float64)
    gate = np.empty((n,), dtype=np.float64)
    if n == 0:
        return dict(out=out, ids=ids, weights=w, gate=gate)
    bad = lib.oracle_moe_forward(T, H, E, k, I, I_s, score_fn, _ptr(hidden), _ptr(logits),
                                 _ptr(wgu), _ptr(wd), _ptr(wsgu), _ptr(wsd), _ptr(wg), _ptr(tok),
                                 n, _ptr(go), _ptr(s_gu), _ptr(s_d),
                                 1.0 if ss_gu is None else float(ss_gu[0]),
                                 1.0 if ss_d is None else float(ss_d[0]),
                                 _ptr(out), _ptr(ids), _ptr(w), _ptr(gate),
                                 n_threads or default_threads())
    assert bad == 0, f"{bad} tokens: fp64 score order contradicts the logit order"
    return dict(out=out, ids=ids, weights=w, gate=gate)


def e4m3_table(lib_path: str | None = None) -> np.ndarray:
    """Values of the 256 FP8 E4M3 codes (NaN for the two NaN codes)."""
    lib = _load(lib_path)
    out = np.empty(256, dtype=np.float64)
    lib.oracle_e4m3_table(_ptr(out))
    return out


def mxfp8_to_bf16(codes, scales, lib_path: str | None = None):
    """Exact dequantisation of MXFP8 weights to bf16 bit patterns.

    codes: uint8 [..., rows, cols] E4M3 codes; scales: uint8 [..., cols/32, rows]
    UE8M0 codes (leading dimensions: experts). Returns uint16 bf16 bits of the
    same shape as codes; raises if any value is not exactly a bf16 value."""
    lib = _load(lib_path)
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    sc = np.ascontiguousarray(np.asarray(scales, dtype=np.uint8))
    rows, cols = c.shape[-2], c.shape[-1]
    lead = int(np.prod(c.shape[:-2])) if c.ndim > 2 else 1
    c2 = c.reshape(lead, rows, cols)
    s2 = sc.reshape(lead, cols // 32, rows)
    out = np.empty((lead, rows, cols), dtype=np.uint16)
    for e in range(lead):
        ce, se, oe = np.ascontiguousarray(c2[e]), np.ascontiguousarray(s2[e]), out[e]
        bad = lib.oracle_mxfp8_to_bf16(rows, cols, _ptr(ce), _ptr(se), _ptr(oe))
        if bad:
            raise ValueError(f"{bad} MXFP8 values are not exact bf16 values")
    return out.reshape(c.shape)


def moe_forward_mxfp8(inputs: dict, k: int, score_fn: int, tokens=None, gate_override=None,
                      lib_path: str | None = None):
    """The layer with MXFP8 expert weights: every quantised matrix is
    dequantised exactly (every MXFP8 value is a bf16 value) and the fp64
    layer runs on the result. inputs holds <name>_q / <name>_s (codes and
    scales) instead of <name> for w_gate_up and w_down, and for the shared
    expert's ws_gate_up and ws_down where those are quantised too."""
    import torch
    plain = dict(inputs)
    for name in ("w_gate_up", "w_down", "ws_gate_up", "ws_down"):
        if name + "_q" not in inputs:
            continue
        bits = mxfp8_to_bf16(_np(plain.pop(name + "_q")), _np(plain.pop(name + "_s")), lib_path)
        plain[name] = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    return moe_forward(plain, k, score_fn, tokens=tokens, gate_override=gate_override,
                       lib_path=lib_path)


def e2m1_table(lib_path: str | None = None) -> np.ndarray:
    """Values of the 16 FP4 E2M1 codes."""
    lib = _load(lib_path)
    out = np.empty(16, dtype=np.float64)
    lib.oracle_e2m1_table(_ptr(out))
    return out


def nvfp4_to_bf16(codes, scales, lib_path: str | None = None):
    """Exact dequantisation of NVFP4 weights (without the fp32 matrix scale)
    to bf16 bit patterns. codes: uint8 [..., rows, cols/2] (two E2M1 values
    per byte, low nibble first); scales: uint8 [..., cols/16, rows] E4M3.
    Returns uint16 [..., rows, cols]; raises on non-finite scales."""
    lib = _load(lib_path)
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    sc = np.ascontiguousarray(np.asarray(scales, dtype=np.uint8))
    rows, cols = c.shape[-2], 2 * c.shape[-1]
    lead = int(np.prod(c.shape[:-2])) if c.ndim > 2 else 1
    c2 = c.reshape(lead, rows, cols // 2)
    s2 = sc.reshape(lead, cols // 16, rows)
    out = np.empty((lead, rows, cols), dtype=np.uint16)
    for e in range(lead):
        bad = lib.oracle_nvfp4_to_bf16(rows, cols, _ptr(np.ascontiguousarray(c2[e])),
                                       _ptr(np.ascontiguousarray(s2[e])), _ptr(out[e]))
        if bad:
            raise ValueError(f"{bad} NVFP4 values are not exact bf16 values")
    return out.reshape(*c.shape[:-1], cols)


def moe_forward_nvfp4(inputs: dict, k: int, score_fn: int, tokens=None, gate_override=None,
                      lib_path: str | None = None):
    """The layer with NVFP4 expert weights: each matrix's E2M1 x E4M3 values
    are dequantised exactly to bf16 and its fp32 matrix scale <name>_g
    multiplies the matrix's dot products. inputs holds <name>_q / <name>_s /
    <name>_g for w_gate_up, w_down, ws_gate_up and ws_down."""
    import torch
    plain = dict(inputs)
    for name in ("w_gate_up", "w_down", "ws_gate_up", "ws_down"):
        bits = nvfp4_to_bf16(_np(plain.pop(name + "_q")), _np(plain.pop(name + "_s")), lib_path)
        plain[name] = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    return moe_forward(plain, k, score_fn, tokens=tokens, gate_override=gate_override,
                       lib_path=lib_path)


def router_logits(hidden, w_router, lib_path: str | None = None) -> np.ndarray:
    """fp64 router logits [T, E] = hidden [T, H] (bf16) . w_router [E, H] (bf16)^T."""
    lib = _load(lib_path)
    x = _u16(hidden)
    w = _u16(w_router)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape[1] == H
    out = np.empty((T, E), dtype=np.float64)
    lib.oracle_router_logits(T, H, E, _ptr(x), _ptr(w), _ptr(out))
    return out


def moe_forward_router(inputs: dict, k: int, score_fn: int, tokens=None,
                       lib_path: str | None = None):
    """The layer with the router computed on the FFN side: inputs holds
    w_router [E, H] bf16 instead of logits. The fp32 router's logits are the
    fp64 sums rounded once to fp32 (round to nearest even), and the layer
    routes on them; returns moe_forward's dict plus logits64 (the fp64 sums)."""
    import torch
    lg64 = router_logits(inputs["hidden"], inputs["w_router"], lib_path)
    plain = {n: v for n, v in inputs.items() if n != "w_router"}
    plain["logits"] = torch.from_numpy(lg64.astype(np.float32))
    res = moe_forward(plain, k, score_fn, tokens=tokens, lib_path=lib_path)
    res["logits64"] = lg64
    return res


def _np(t):
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu()
            if t.dtype == torch.float8_e4m3fn:
                t = t.view(torch.uint8)
            return t.numpy()
    except ImportError:
        pass
    return np.asarray(t)

