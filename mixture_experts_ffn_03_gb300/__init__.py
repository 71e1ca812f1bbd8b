"""Python binding of libmoe, the sm_103a MoE FFN layer (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. PyTorch supplies device memory and the current stream. Importing
this package loads ``libmoe.so`` from this directory and fails loudly if it
has not been built (``python -m mixture_experts_ffn_03_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

SOFTMAX = 0
SIGMOID = 1

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_CAPACITY = 6
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT",
                6: "MOE_ERR_CAPACITY"}

EXPORTED = ["moe_workspace_size", "moe_forward", "moe_device_status", "moe_status_string",
            "moe_workspace_layout", "moe_set_stage_events", "moe_launch_count",
            "moe_selftest_wait_limit", "moe_forward_mxfp8", "moe_mxfp8_dequant",
            "moe_forward_router", "moe_workspace_size_router", "moe_launch_count_router",
            "moe_forward_nvfp4", "moe_nvfp4_dequant", "moe_launch_count_quantized",
            "moe_set_expert_fusion", "moe_get_expert_fusion", "moe_pipeline_create",
            "moe_pipeline_submit", "moe_pipeline_drain", "moe_pipeline_streams",
            "moe_pipeline_destroy", "moe_y16_roundtrip"]
NUM_STAGES = 5
STAGE_NAMES = ["route", "scatter", "gate_up", "down", "combine"]


class MoEDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32), ("I_s", ctypes.c_int32),
                ("score_fn", ctypes.c_int32)]


class MoEWorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("topk_ids", "topk_w", "gate_logit", "counts", "offsets", "perm", "inv", "h_hi",
                 "h_lo", "hs_hi", "hs_lo", "y", "total")]


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmoe.so (once). Raises if the CUDA library has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe.so not found at {path}; build it first "
                           "(python -m mixture_experts_ffn_03_gb300.build)")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.moe_workspace_size.argtypes = [ctypes.POINTER(MoEDims)]
    lib.moe_workspace_size.restype = ctypes.c_size_t
    lib.moe_forward.argtypes = [ctypes.POINTER(MoEDims)] + [P] * 11 + [P, ctypes.c_size_t, P]
    lib.moe_forward.restype = ctypes.c_int
    lib.moe_device_status.argtypes = [P, P]
    lib.moe_device_status.restype = ctypes.c_int
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_workspace_layout.argtypes = [ctypes.POINTER(MoEDims), ctypes.POINTER(MoEWorkspaceLayout)]
    lib.moe_workspace_layout.restype = ctypes.c_int
    lib.moe_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
    lib.moe_set_stage_events.restype = ctypes.c_int
    lib.moe_launch_count.argtypes = [ctypes.POINTER(MoEDims)]
    lib.moe_launch_count.restype = ctypes.c_int
    lib.moe_selftest_wait_limit.argtypes = [P, P]
    lib.moe_selftest_wait_limit.restype = ctypes.c_int
    lib.moe_forward_mxfp8.argtypes = [ctypes.POINTER(MoEDims)] + [P] * 15 + [P, ctypes.c_size_t, P]
    lib.moe_forward_mxfp8.restype = ctypes.c_int
    lib.moe_y16_roundtrip.argtypes = [P, P, ctypes.c_int64, P]
    lib.moe_y16_roundtrip.restype = ctypes.c_int
    lib.moe_mxfp8_dequant.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P, P]
    lib.moe_mxfp8_dequant.restype = ctypes.c_int
    lib.moe_forward_router.argtypes = [ctypes.POINTER(MoEDims)] + [P] * 12 + [P, ctypes.c_size_t, P]
    lib.moe_forward_nvfp4.argtypes = [ctypes.POINTER(MoEDims)] + [P] * 19 + [P, ctypes.c_size_t, P]
    lib.moe_forward_nvfp4.restype = ctypes.c_int
    lib.moe_nvfp4_dequant.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P, P]
    lib.moe_nvfp4_dequant.restype = ctypes.c_int
    lib.moe_forward_router.restype = ctypes.c_int
    lib.moe_workspace_size_router.argtypes = [ctypes.POINTER(MoEDims)]
    lib.moe_workspace_size_router.restype = ctypes.c_size_t
    lib.moe_launch_count_router.argtypes = [ctypes.POINTER(MoEDims)]
    lib.moe_launch_count_router.restype = ctypes.c_int
    lib.moe_launch_count_quantized.argtypes = [ctypes.POINTER(MoEDims)]
    lib.moe_launch_count_quantized.restype = ctypes.c_int
    lib.moe_set_expert_fusion.argtypes = [ctypes.c_int]
    lib.moe_set_expert_fusion.restype = None
    lib.moe_get_expert_fusion.argtypes = []
    lib.moe_get_expert_fusion.restype = ctypes.c_int
    lib.moe_pipeline_create.argtypes = [ctypes.POINTER(MoEDims)] + [P] * 6 + [
        ctypes.POINTER(ctypes.c_void_p)]
    lib.moe_pipeline_create.restype = ctypes.c_int
    lib.moe_pipeline_submit.argtypes = [P, P, P, P]
    lib.moe_pipeline_submit.restype = ctypes.c_int
    lib.moe_pipeline_drain.argtypes = [P]
    lib.moe_pipeline_drain.restype = ctypes.c_int
    lib.moe_pipeline_streams.argtypes = [P, ctypes.POINTER(ctypes.c_void_p),
                                         ctypes.POINTER(ctypes.c_void_p)]
    lib.moe_pipeline_streams.restype = ctypes.c_int
    lib.moe_pipeline_destroy.argtypes = [P]
    lib.moe_pipeline_destroy.restype = None
    _lib = lib
    return lib


def make_dims(T, H, E, k, I, I_s, score_fn) -> MoEDims:
    return MoEDims(int(T), int(H), int(E), int(k), int(I), int(I_s), int(score_fn))


def workspace_size(dims: MoEDims) -> int:
    return int(load_library().moe_workspace_size(ctypes.byref(dims)))


def workspace_layout(dims: MoEDims) -> MoEWorkspaceLayout:
    out = MoEWorkspaceLayout()
    st = load_library().moe_workspace_layout(ctypes.byref(dims), ctypes.byref(out))
    if st != MOE_OK:
        raise MoEError(st, "moe_workspace_layout")
    return out


def launch_count(dims: MoEDims) -> int:
    """Kernels one moe_forward launches for these sizes (from this thread)."""
    return int(load_library().moe_launch_count(ctypes.byref(dims)))


def launch_count_quantized(dims: MoEDims) -> int:
    """Kernels one moe_forward_mxfp8 / moe_forward_nvfp4 launches for these sizes."""
    return int(load_library().moe_launch_count_quantized(ctypes.byref(dims)))


def set_expert_fusion(level) -> None:
    """Launch fusion for bf16 weights, for calls from this host thread: 0 or
    False (the default) none; 1 or True the fused gate_up + down launch on
    decode-sized batches; 2 also the whole layer in one launch where it
    applies (T*k <= 2048, E <= 256, logits given)."""
    load_library().moe_set_expert_fusion(int(level))


def get_expert_fusion() -> int:
    return int(load_library().moe_get_expert_fusion())


class expert_fusion:  # noqa: N801 (used like a function: `with expert_fusion(True):`)
    """Context manager: `with expert_fusion(level): ...` runs the block with
    that fusion level (set_expert_fusion), then restores the setting."""

    def __init__(self, enable):
        self.enable = int(enable)

    def __enter__(self):
        self.prev = get_expert_fusion()
        set_expert_fusion(self.enable)
        return self

    def __exit__(self, *exc):
        set_expert_fusion(self.prev)
        return False


def status_string(status: int) -> str:
    return load_library().moe_status_string(int(status)).decode()


def set_stage_events(events) -> None:
    """Record torch.cuda.Event objects around each kernel of subsequent
    moe_forward calls from this thread (NUM_STAGES + 1 events), or stop (None)."""
    lib = load_library()
    if events is None:
        st = lib.moe_set_stage_events(None, 0)
    else:
        arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        st = lib.moe_set_stage_events(arr, len(events))
    if st != MOE_OK:
        raise MoEError(st, "moe_set_stage_events")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def forward_raw(dims: MoEDims, hidden, logits, w_gate_up, w_down, ws_gate_up, ws_down, w_g, out,
                workspace, topk_ids_out=None, topk_w_out=None, counts_out=None,
                stream=None) -> int:
    """Direct call of moe_forward on tensors (or None); returns the status code."""
    lib = load_library()
    return int(lib.moe_forward(ctypes.byref(dims), _ptr(hidden), _ptr(logits), _ptr(w_gate_up),
                               _ptr(w_down), _ptr(ws_gate_up), _ptr(ws_down), _ptr(w_g),
                               _ptr(out), _ptr(topk_ids_out), _ptr(topk_w_out), _ptr(counts_out),
                               _ptr(workspace),
                               ctypes.c_size_t(0 if workspace is None else workspace.numel()),
                               _stream_handle(stream)))


def forward_mxfp8_raw(dims: MoEDims, hidden, logits, w_gate_up_q, w_gate_up_s, w_down_q, w_down_s,
                      ws_gate_up_q, ws_gate_up_s, ws_down_q, ws_down_s, w_g, out, workspace,
                      topk_ids_out=None, topk_w_out=None, counts_out=None, stream=None) -> int:
    """Direct call of moe_forward_mxfp8 on tensors (or None); returns the status code."""
    lib = load_library()
    return int(lib.moe_forward_mxfp8(
        ctypes.byref(dims), _ptr(hidden), _ptr(logits), _ptr(w_gate_up_q), _ptr(w_gate_up_s),
        _ptr(w_down_q), _ptr(w_down_s), _ptr(ws_gate_up_q), _ptr(ws_gate_up_s), _ptr(ws_down_q),
        _ptr(ws_down_s), _ptr(w_g), _ptr(out), _ptr(topk_ids_out), _ptr(topk_w_out),
        _ptr(counts_out), _ptr(workspace),
        ctypes.c_size_t(0 if workspace is None else workspace.numel()), _stream_handle(stream)))


def forward_nvfp4_raw(dims: MoEDims, hidden, logits, w_gate_up, w_down, ws_gate_up, ws_down, w_g,
                      out, workspace, topk_ids_out=None, topk_w_out=None, counts_out=None,
                      stream=None) -> int:
    """Direct call of moe_forward_nvfp4; each weight is a (codes, scales, g) triple."""
    lib = load_library()
    return int(lib.moe_forward_nvfp4(
        ctypes.byref(dims), _ptr(hidden), _ptr(logits), *[_ptr(t) for t in w_gate_up],
        *[_ptr(t) for t in w_down], *[_ptr(t) for t in ws_gate_up], *[_ptr(t) for t in ws_down],
        _ptr(w_g), _ptr(out), _ptr(topk_ids_out), _ptr(topk_w_out), _ptr(counts_out),
        _ptr(workspace), ctypes.c_size_t(0 if workspace is None else workspace.numel()),
        _stream_handle(stream)))


def nvfp4_dequant(codes, scales, out=None, stream=None):
    """bf16 values E2M1 x E4M3 of an NVFP4 matrix (moe_nvfp4_dequant): codes uint8
    [rows, cols/2], scales uint8 [cols/16, rows] on the GPU; returns out [rows, cols]."""
    import torch
    rows, half = codes.shape
    cols = 2 * half
    if out is None:
        out = torch.empty(rows, cols, dtype=torch.bfloat16, device=codes.device)
    st = load_library().moe_nvfp4_dequant(_ptr(codes), _ptr(scales), int(rows), int(cols),
                                          _ptr(out), _stream_handle(stream))
    if st != MOE_OK:
        raise MoEError(st, "moe_nvfp4_dequant")
    return out


def mxfp8_dequant(codes, scales, out=None, stream=None):
    """bf16 values of an MXFP8 matrix (moe_mxfp8_dequant): codes uint8 [rows,
    cols], scales uint8 [cols/32, rows] on the GPU; returns out [rows, cols]."""
    import torch
    rows, cols = codes.shape
    if out is None:
        out = torch.empty(rows, cols, dtype=torch.bfloat16, device=codes.device)
    st = load_library().moe_mxfp8_dequant(_ptr(codes), _ptr(scales), int(rows), int(cols),
                                          _ptr(out), _stream_handle(stream))
    if st != MOE_OK:
        raise MoEError(st, "moe_mxfp8_dequant")
    return out


def y16_roundtrip(x, out=None, stream=None):
    """fp32 values through the y16 format (moe_y16_roundtrip): x float32 on the
    GPU with a multiple of 32 elements, each block of 32 consecutive values
    sharing one exponent byte; returns the decoded values."""
    import torch
    if out is None:
        out = torch.empty_like(x)
    st = load_library().moe_y16_roundtrip(_ptr(x), _ptr(out), int(x.numel()), _stream_handle(stream))
    if st != MOE_OK:
        raise MoEError(st, "moe_y16_roundtrip")
    return out


def forward_router_raw(dims: MoEDims, hidden, w_router, w_gate_up, w_down, ws_gate_up, ws_down,
                       w_g, out, workspace, logits_out=None, topk_ids_out=None, topk_w_out=None,
                       counts_out=None, stream=None) -> int:
    """Direct call of moe_forward_router on tensors (or None); returns the status code."""
    lib = load_library()
    return int(lib.moe_forward_router(
        ctypes.byref(dims), _ptr(hidden), _ptr(w_router), _ptr(w_gate_up), _ptr(w_down),
        _ptr(ws_gate_up), _ptr(ws_down), _ptr(w_g), _ptr(out), _ptr(logits_out),
        _ptr(topk_ids_out), _ptr(topk_w_out), _ptr(counts_out), _ptr(workspace),
        ctypes.c_size_t(0 if workspace is None else workspace.numel()), _stream_handle(stream)))


def workspace_size_router(dims: MoEDims) -> int:
    return int(load_library().moe_workspace_size_router(ctypes.byref(dims)))


def launch_count_router(dims: MoEDims) -> int:
    """Kernels one moe_forward_router launches for these sizes on the current device."""
    return int(load_library().moe_launch_count_router(ctypes.byref(dims)))


def device_status(workspace, stream=None) -> int:
    return int(load_library().moe_device_status(_ptr(workspace), _stream_handle(stream)))


def selftest_wait_limit(workspace, stream=None) -> int:
    """Enqueue the bounded-wait self-test on `workspace`'s status word (see
    moe_selftest_wait_limit in include/moe.h); returns the call's status."""
    return int(load_library().moe_selftest_wait_limit(_ptr(workspace), _stream_handle(stream)))


class MoELayer:
    """The layer's weights plus a reusable workspace on one CUDA device.

    ``forward(hidden, logits)`` enqueues one moe_forward on the current
    stream; outputs are allocated by PyTorch unless ``out`` is given. The
    subclasses differ only in how the expert weights are held and which
    entry point ``_enqueue`` calls."""

    entry = "moe_forward"

    def __init__(self, w_gate_up, w_down, ws_gate_up, ws_down, w_g, k: int, score_fn: int):
        import torch
        self.w_gate_up, self.w_down = w_gate_up, w_down
        self.ws_gate_up, self.ws_down, self.w_g = ws_gate_up, ws_down, w_g
        self.E, two_i, self.H = self._shape(w_gate_up)
        self.I = two_i // 2
        self.I_s = self._shape(ws_gate_up)[0] // 2
        self.k, self.score_fn = int(k), int(score_fn)
        self.device = self._first(w_gate_up).device
        self._ws = torch.empty(0, dtype=torch.uint8, device=self.device)

    @staticmethod
    def _first(w):
        return w

    def _shape(self, w):
        """Logical shape of a weight: (E, 2I, H) for the routed gate/up
        weights, (2I_s, H) for the shared ones."""
        return tuple(self._first(w).shape)

    def _workspace_size(self, dims: MoEDims) -> int:
        return workspace_size(dims)

    def _enqueue(self, dims, hidden, logits, out, ws, topk_ids, topk_w, counts, stream):
        return forward_raw(dims, hidden, logits, self.w_gate_up, self.w_down, self.ws_gate_up,
                           self.ws_down, self.w_g, out, ws, topk_ids, topk_w, counts, stream)

    def dims(self, T: int) -> MoEDims:
        return make_dims(T, self.H, self.E, self.k, self.I, self.I_s, self.score_fn)

    def workspace(self, T: int):
        import torch
        need = self._workspace_size(self.dims(T))
        if self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, hidden, logits, out=None, topk_ids=None, topk_w=None, counts=None,
                stream=None):
        import torch
        T = hidden.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device)
        ws = self.workspace(T)
        st = self._enqueue(self.dims(T), hidden, logits, out, ws, topk_ids, topk_w, counts,
                           stream)
        if st != MOE_OK:
            raise MoEError(st, self.entry)
        return out

    def forward_from_host(self, hidden_host, logits_host, out_host, stream=None):
        """End-to-end call from pinned host buffers: copy hidden and logits in
        (no logits for a layer that computes them itself: pass None), run the
        layer, copy the output back (all on one stream)."""
        import torch
        T = hidden_host.shape[0]
        if not hasattr(self, "_io") or self._io[0].shape[0] != T:
            self._io = (torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device),
                        torch.empty(T, self.E, dtype=torch.float32, device=self.device),
                        torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device))
        h, l, o = self._io
        s = stream or torch.cuda.current_stream()
        with torch.cuda.stream(s):
            h.copy_(hidden_host, non_blocking=True)
            if logits_host is not None:
                l.copy_(logits_host, non_blocking=True)
                self.forward(h, l, out=o, stream=s)
            else:
                self.forward(h, out=o, stream=s)
            out_host.copy_(o, non_blocking=True)
        return out_host


class MoELayerMXFP8(MoELayer):
    """MoELayer with MXFP8 expert weights (moe_forward_mxfp8): each of
    w_gate_up, w_down, ws_gate_up, ws_down is a pair (codes uint8 [..., rows,
    K], scales uint8 [..., K/32, rows]); w_g stays bf16."""

    entry = "moe_forward_mxfp8"

    @staticmethod
    def _first(w):
        return w[0]

    def _enqueue(self, dims, hidden, logits, out, ws, topk_ids, topk_w, counts, stream):
        return forward_mxfp8_raw(dims, hidden, logits, *self.w_gate_up, *self.w_down,
                                 *self.ws_gate_up, *self.ws_down, self.w_g, out, ws, topk_ids,
                                 topk_w, counts, stream)


class MoELayerNVFP4(MoELayer):
    """MoELayer with NVFP4 expert weights (moe_forward_nvfp4): each of w_gate_up,
    w_down, ws_gate_up, ws_down is a triple (codes uint8 [..., rows, K/2],
    scales uint8 [..., K/16, rows], g fp32 [E] or [1]); w_g stays bf16."""

    entry = "moe_forward_nvfp4"

    @staticmethod
    def _first(w):
        return w[0]

    def _shape(self, w):
        *lead, half_k = self._first(w).shape  # two E2M1 codes per byte along K
        return (*lead, 2 * half_k)

    def _enqueue(self, dims, hidden, logits, out, ws, topk_ids, topk_w, counts, stream):
        return forward_nvfp4_raw(dims, hidden, logits, self.w_gate_up, self.w_down,
                                 self.ws_gate_up, self.ws_down, self.w_g, out, ws, topk_ids,
                                 topk_w, counts, stream)


class MoELayerRouter(MoELayer):
    """MoELayer that computes the router logits itself (moe_forward_router):
    forward(hidden) with w_router [E, H] bf16 held by the layer; the logits
    [T, E] fp32 are returned through `logits` when given."""

    entry = "moe_forward_router"

    def __init__(self, w_router, w_gate_up, w_down, ws_gate_up, ws_down, w_g, k: int,
                 score_fn: int):
        super().__init__(w_gate_up, w_down, ws_gate_up, ws_down, w_g, k, score_fn)
        self.w_router = w_router

    def _workspace_size(self, dims: MoEDims) -> int:
        return workspace_size_router(dims)

    def _enqueue(self, dims, hidden, logits, out, ws, topk_ids, topk_w, counts, stream):
        return forward_router_raw(dims, hidden, self.w_router, self.w_gate_up, self.w_down,
                                  self.ws_gate_up, self.ws_down, self.w_g, out, ws, logits,
                                  topk_ids, topk_w, counts, stream)

    def forward(self, hidden, logits=None, out=None, topk_ids=None, topk_w=None, counts=None,
                stream=None):
        return super().forward(hidden, logits, out, topk_ids, topk_w, counts, stream)


class NativePipeline:
    """The library's serving loop from host memory (moe_pipeline_*) for a bf16
    MoELayer with router logits as input: two device staging sets, an input
    and an output copy stream owned by the library, compute on
    ``compute_stream``. ``submit`` passes pinned host tensors (hidden [T, H]
    bf16, logits [T, E] fp32, out [T, H] bf16) to the C call; a step's host
    tensors must stay untouched until ``drain()`` or two further submits.
    ``xs`` / ``ys`` are the library's input / output copy streams."""

    def __init__(self, layer, T, compute_stream=None):
        import torch
        if type(layer) is not MoELayer:
            raise TypeError("NativePipeline runs the bf16 moe_forward layer (MoELayer)")
        self.layer, self.T = layer, int(T)
        self._lib = load_library()
        dev = layer.device
        cs = compute_stream or torch.cuda.current_stream(dev)
        self._dims = layer.dims(self.T)
        h = ctypes.c_void_p()
        with torch.cuda.device(dev):
            st = self._lib.moe_pipeline_create(
                ctypes.byref(self._dims), _ptr(layer.w_gate_up), _ptr(layer.w_down),
                _ptr(layer.ws_gate_up), _ptr(layer.ws_down), _ptr(layer.w_g),
                _stream_handle(cs), ctypes.byref(h))
        if st != MOE_OK:
            raise MoEError(st, "moe_pipeline_create")
        self._h = h
        ins, outs = ctypes.c_void_p(), ctypes.c_void_p()
        self._lib.moe_pipeline_streams(self._h, ctypes.byref(ins), ctypes.byref(outs))
        self.xs = torch.cuda.ExternalStream(ins.value, device=dev)
        self.ys = torch.cuda.ExternalStream(outs.value, device=dev)

    def _check(self, t, dtype, cols):
        if t.device.type != "cpu" or t.dtype != dtype or not t.is_contiguous() or \
                tuple(t.shape) != (self.T, cols):
            raise ValueError(f"expected a contiguous host tensor [{self.T}, {cols}] of {dtype}")

    def submit(self, hidden_host, logits_host, out_host):
        import torch
        self._check(hidden_host, torch.bfloat16, self.layer.H)
        self._check(logits_host, torch.float32, self.layer.E)
        self._check(out_host, torch.bfloat16, self.layer.H)
        st = self._lib.moe_pipeline_submit(self._h, _ptr(hidden_host), _ptr(logits_host),
                                           _ptr(out_host))
        if st != MOE_OK:
            raise MoEError(st, "moe_pipeline_submit")
        return out_host

    def drain(self):
        st = self._lib.moe_pipeline_drain(self._h)
        if st != MOE_OK:
            raise MoEError(st, "moe_pipeline_drain")

    def close(self):
        if getattr(self, "_h", None):
            self._lib.moe_pipeline_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()


class HostPipeline:
    """Serving loop from pinned host buffers that overlaps host transfers with
    compute. Each submit() copies one step's hidden rows and router logits on an
    input copy stream into one of two device staging sets, runs the layer on
    the compute stream once they have landed, and copies the output back on an
    output copy stream once the layer is done. The two directions use separate
    streams, so the next step's input copy overlaps this step's compute (it
    does not queue behind this step's output copy, which waits for the
    compute). Every byte still crosses between host and device on every step.
    A caller reuses an out_host buffer only after drain() (or after two
    further submits). For a layer that computes its own router logits
    (MoELayerRouter) pass logits_host=None: only the hidden rows go in."""

    def __init__(self, layer, T, compute_stream=None, copy_stream=None, out_stream=None):
        import torch
        self.layer = layer
        dev = layer.device
        self.cs = compute_stream or torch.cuda.current_stream(dev)
        self.xs = copy_stream or torch.cuda.Stream(dev)      # host -> device
        self.ys = out_stream or torch.cuda.Stream(dev)       # device -> host
        self.h = [torch.empty(T, layer.H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.l = [torch.empty(T, layer.E, dtype=torch.float32, device=dev) for _ in range(2)]
        self.o = [torch.empty(T, layer.H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.done = [torch.cuda.Event() for _ in range(2)]
        self.out_read = [torch.cuda.Event() for _ in range(2)]
        self.i = 0

    def submit(self, hidden_host, logits_host, out_host):
        import torch
        b = self.i % 2
        if self.i >= 2:
            self.xs.wait_event(self.done[b])      # step i-2 no longer reads set b
        with torch.cuda.stream(self.xs):
            self.h[b].copy_(hidden_host, non_blocking=True)
            if logits_host is not None:
                self.l[b].copy_(logits_host, non_blocking=True)
            self.in_ready[b].record(self.xs)
        self.cs.wait_event(self.in_ready[b])
        if self.i >= 2:
            self.cs.wait_event(self.out_read[b])  # step i-2's output has been copied out
        if logits_host is not None:
            self.layer.forward(self.h[b], self.l[b], out=self.o[b], stream=self.cs)
        else:
            self.layer.forward(self.h[b], out=self.o[b], stream=self.cs)
        self.done[b].record(self.cs)
        self.ys.wait_event(self.done[b])
        with torch.cuda.stream(self.ys):
            out_host.copy_(self.o[b], non_blocking=True)
            self.out_read[b].record(self.ys)
        self.i += 1
        return out_host

    def drain(self):
        self.xs.synchronize()
        self.cs.synchronize()
        self.ys.synchronize()

