"""Expert parallelism: the layer spread over G ranks, one GPU each.

Rank g owns the routed experts [g E/G, (g+1) E/G) and a copy of the shared
expert; every rank brings its own tokens. The pages run the experts this way
("FastAFD" pull request, What the model needed: expert workers at EP 4;
"qwen3_5_moe is TP=1-only ...", first comment: routed experts sharded across
ranks). One step on a rank (include/moe.h, moe_ep_*):

1. dispatch  routing and permute of the rank's tokens over all E experts, the
             (token, slot) rows in expert-sorted order (x_send) and the rows
             per expert (counts): the rows for rank g are one contiguous range;
2. exchange  an all-to-all of the per-expert counts, then of the rows;
3. experts   the rank's experts on the received rows, in source-rank order
             with each source's rows sorted by local expert, plus the shared
             expert on the rank's own tokens;
4. exchange  the expert rows travel back to their source ranks (the reverse
             all-to-all), landing in the rank's own sorted order;
5. combine   the same fixed-order gather combine as the single-GPU layer.

The local steps run in libmoe's kernels (LibMoeEPOps); this module only moves
buffers between the steps. ExpertParallelMoE.forward does the exchanges with
torch.distributed (NCCL between GPUs); LocalExchange runs G ranks one after
another in one process, for a single GPU (no collective and no kernel that
waits on another rank).
"""
from __future__ import annotations

import ctypes
import dataclasses

from . import MOE_OK, MoEError, _ptr, _stream_handle, load_library


class EPDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "H", "E", "k", "I", "I_s", "score_fn", "G", "R_max")]


class EPLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("topk_ids", "topk_w", "gate_logit", "counts", "offsets", "perm", "inv", "y",
                 "total")]


def _lib():
    lib = load_library()
    if getattr(lib, "_ep_bound", False):
        return lib
    P, S, I32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    D = ctypes.POINTER(EPDims)
    lib.moe_ep_workspace_size.argtypes = [D]
    lib.moe_ep_workspace_size.restype = S
    lib.moe_ep_workspace_layout.argtypes = [D, ctypes.POINTER(EPLayout)]
    lib.moe_ep_workspace_layout.restype = ctypes.c_int
    lib.moe_ep_dispatch.argtypes = [D, P, P, P, P, P, P, P, P, S, P]
    lib.moe_ep_dispatch.restype = ctypes.c_int
    lib.moe_ep_experts.argtypes = [D, I32, P, P, P, P, P, P, P, P, S, P]
    lib.moe_ep_experts.restype = ctypes.c_int
    lib.moe_ep_combine.argtypes = [D, I32, P, P, P, S, P]
    lib.moe_ep_combine.restype = ctypes.c_int
    lib._ep_bound = True
    return lib


def ep_dims(T, H, E, k, I, I_s, score_fn, G, R_max) -> EPDims:
    return EPDims(*(int(v) for v in (T, H, E, k, I, I_s, score_fn, G, R_max)))


def ep_workspace_size(d: EPDims) -> int:
    return int(_lib().moe_ep_workspace_size(ctypes.byref(d)))


def ep_workspace_layout(d: EPDims) -> EPLayout:
    out = EPLayout()
    st = _lib().moe_ep_workspace_layout(ctypes.byref(d), ctypes.byref(out))
    if st != MOE_OK:
        raise MoEError(st, "moe_ep_workspace_layout")
    return out


def send_splits(counts, G: int):
    """Rows for each destination rank: the per-expert counts [E] summed over
    each rank's block of E/G experts (host ints)."""
    E = len(counts)
    e_loc = E // G
    return [int(sum(counts[g * e_loc:(g + 1) * e_loc])) for g in range(G)]


class LibMoeEPOps:
    """The local steps on the GPU, through libmoe (moe_ep_dispatch, moe_ep_experts,
    moe_ep_combine). Tensors are CUDA tensors; `ws` is the rank's workspace."""

    def workspace(self, d: EPDims, device, old=None):
        import torch
        need = ep_workspace_size(d)
        if need == 0:
            raise MoEError(1, "moe_ep_workspace_size")
        if old is not None and old.numel() >= need:
            return old
        return torch.empty(need, dtype=torch.uint8, device=device)

    def dispatch(self, d: EPDims, hidden, logits, w_g, ws, stream=None):
        import torch
        x_send = torch.empty(d.T * d.k, d.H, dtype=torch.bfloat16, device=hidden.device)
        counts = torch.empty(d.E, dtype=torch.int32, device=hidden.device)
        st = _lib().moe_ep_dispatch(ctypes.byref(d), _ptr(hidden), _ptr(logits), _ptr(w_g),
                                    _ptr(x_send), _ptr(counts), None, None, _ptr(ws),
                                    ctypes.c_size_t(ws.numel()), _stream_handle(stream))
        if st != MOE_OK:
            raise MoEError(st, "moe_ep_dispatch")
        return x_send, counts

    def experts(self, d: EPDims, R: int, x_recv, recv_counts, hidden, w_gate_up, w_down,
                ws_gate_up, ws_down, ws, stream=None):
        """Returns the expert rows of the received rows, [R, H] fp32 (a view of
        the workspace, valid until the rank's next experts call)."""
        st = _lib().moe_ep_experts(ctypes.byref(d), int(R), _ptr(x_recv) if R else None,
                                   _ptr(recv_counts), _ptr(hidden), _ptr(w_gate_up),
                                   _ptr(w_down), _ptr(ws_gate_up), _ptr(ws_down), _ptr(ws),
                                   ctypes.c_size_t(ws.numel()), _stream_handle(stream))
        if st != MOE_OK:
            raise MoEError(st, "moe_ep_experts")
        import torch
        L = ep_workspace_layout(d)
        return ws[L.y:L.y + R * d.H * 4].view(torch.float32).view(R, d.H)

    def combine(self, d: EPDims, R: int, y_back, ws, stream=None):
        import torch
        out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device=ws.device)
        st = _lib().moe_ep_combine(ctypes.byref(d), int(R), _ptr(y_back), _ptr(out), _ptr(ws),
                                   ctypes.c_size_t(ws.numel()), _stream_handle(stream))
        if st != MOE_OK:
            raise MoEError(st, "moe_ep_combine")
        return out


@dataclasses.dataclass
class Dispatched:
    """What a rank's dispatch step leaves for the exchange: its rows in
    expert-sorted order, the rows per expert and per destination rank."""
    T: int
    x_send: object
    counts: object          # [E] int32, on the rank's device
    splits: list            # rows for each destination rank (host ints)


class ExpertParallelMoE:
    """One rank's share of the layer: routed experts [rank E/G, (rank+1) E/G)
    (w_gate_up_local [E/G, 2I, H], w_down_local [E/G, H, I]) and the shared
    expert. max_tokens_per_rank bounds every rank's T; it sizes the received
    rows (at most G * max_tokens_per_rank * min(k, E/G))."""

    def __init__(self, rank, G, w_gate_up_local, w_down_local, ws_gate_up, ws_down, w_g, E,
                 k, score_fn, max_tokens_per_rank, ops=None, group=None):
        self.rank, self.G, self.E, self.k, self.score_fn = int(rank), int(G), int(E), int(k), int(score_fn)
        if self.E % self.G:
            raise ValueError("E must be a multiple of the number of ranks")
        self.e_loc = self.E // self.G
        self.w_gate_up, self.w_down = w_gate_up_local, w_down_local
        self.ws_gate_up, self.ws_down, self.w_g = ws_gate_up, ws_down, w_g
        e_loc, two_i, self.H = tuple(w_gate_up_local.shape)
        if e_loc != self.e_loc:
            raise ValueError("w_gate_up_local must hold E/G experts")
        self.I = two_i // 2
        self.I_s = ws_gate_up.shape[0] // 2
        self.max_tokens = int(max_tokens_per_rank)
        self.R_max = self.G * self.max_tokens * min(self.k, self.e_loc)
        self.ops = ops if ops is not None else LibMoeEPOps()
        self.group = group
        self._ws = None
        self._hidden = None

    def dims(self, T: int) -> EPDims:
        if T > self.max_tokens:
            raise ValueError(f"{T} tokens exceed max_tokens_per_rank={self.max_tokens}")
        return ep_dims(T, self.H, self.E, self.k, self.I, self.I_s, self.score_fn, self.G,
                       self.R_max)

    # ------------------------------------------------------------- local steps
    def step_dispatch(self, hidden, logits) -> Dispatched:
        T = hidden.shape[0]
        d = self.dims(T)
        self._ws = self.ops.workspace(d, hidden.device, self._ws)
        self._hidden = hidden
        x_send, counts = self.ops.dispatch(d, hidden, logits, self.w_g, self._ws)
        splits = send_splits(counts.cpu().tolist(), self.G)
        return Dispatched(T=T, x_send=x_send, counts=counts, splits=splits)

    def step_experts(self, T: int, x_recv, recv_counts):
        """x_recv [R, H]: the received rows; recv_counts [G, E/G] int32 on the
        rank's device. Returns the expert rows [R, H] fp32."""
        R = x_recv.shape[0]
        if R > self.R_max:
            raise ValueError(f"{R} received rows exceed the bound {self.R_max}")
        return self.ops.experts(self.dims(T), R, x_recv, recv_counts, self._hidden,
                                self.w_gate_up, self.w_down, self.ws_gate_up, self.ws_down,
                                self._ws)

    def step_combine(self, T: int, R: int, y_back):
        return self.ops.combine(self.dims(T), R, y_back, self._ws)

    # ------------------------------------------------------- one step, G ranks
    def forward(self, hidden, logits):
        """The layer for this rank's tokens, with the two exchanges done by
        all-to-alls on the process group (every rank calls forward together)."""
        import torch
        import torch.distributed as dist
        dev = hidden.device
        disp = self.step_dispatch(hidden, logits)
        # counts of this rank's experts from every source (equal splits of E/G)
        recv_counts = torch.empty_like(disp.counts)
        dist.all_to_all_single(recv_counts, disp.counts, group=self.group)
        recv_counts = recv_counts.view(self.G, self.e_loc)
        recv_splits = [int(v) for v in recv_counts.sum(dim=1).cpu().tolist()]
        R = sum(recv_splits)
        # rows travel as bytes (2 H per row): every backend moves uint8
        x_recv = torch.empty(R, self.H, dtype=torch.bfloat16, device=dev)
        dist.all_to_all_single(x_recv.view(torch.uint8), disp.x_send.view(torch.uint8),
                               recv_splits, disp.splits, group=self.group)
        y = self.step_experts(disp.T, x_recv, recv_counts)
        y_back = torch.empty(disp.T * self.k, self.H, dtype=torch.float32, device=dev)
        dist.all_to_all_single(y_back, y, disp.splits, recv_splits, group=self.group)
        return self.step_combine(disp.T, R, y_back)


class LocalExchange:
    """Runs one step of G ranks in one process (one GPU or the host): every
    rank's dispatch, then the exchange by slicing, every rank's experts, the
    exchange back, every rank's combine. The ranks' kernels run one after
    another; none waits on another rank."""

    def __init__(self, layers):
        self.layers = list(layers)
        self.G = len(self.layers)

    def forward(self, hiddens, logits):
        import torch
        G = self.G
        e_loc = self.layers[0].e_loc
        disp = [self.layers[s].step_dispatch(hiddens[s], logits[s]) for s in range(G)]
        starts = [[0] * (G + 1) for _ in range(G)]   # starts[s][g]: first row of s's rows for g
        for s in range(G):
            for g in range(G):
                starts[s][g + 1] = starts[s][g] + disp[s].splits[g]
        ys, Rs = [], []
        for g in range(G):
            x_recv = torch.cat([disp[s].x_send[starts[s][g]:starts[s][g + 1]] for s in range(G)])
            recv_counts = torch.stack([disp[s].counts[g * e_loc:(g + 1) * e_loc]
                                       for s in range(G)])
            Rs.append(x_recv.shape[0])
            # a view of rank g's workspace, valid until rank g's next step
            ys.append(self.layers[g].step_experts(disp[g].T, x_recv, recv_counts))
        outs = []
        for s in range(G):
            parts, row = [], [0] * G
            for g in range(G):   # rank g's rows from source s follow sources 0..s-1
                row[g] = sum(disp[q].splits[g] for q in range(s))
                parts.append(ys[g][row[g]:row[g] + disp[s].splits[g]])
            y_back = torch.cat(parts) if parts else None
            outs.append(self.layers[s].step_combine(disp[s].T, Rs[s], y_back))
        return outs
