"""Seeded synthetic workloads for the MoE FFN layer.

This module only draws random inputs; it holds none of the layer's arithmetic.
Both the CUDA path (through the tests and the benchmark) and the CPU oracle read
the tensors it returns, byte for byte.

Shapes follow the Qwen3.5-style MoE block described in
"Add Qwen3.5-35B-A3B (support vision and text input)" (Description: 256 routed
experts, top-8, one sigmoid-gated shared expert) and the wider 512-expert /
top-10 family member named in the FastAFD pull request ("What the model needed").

Recipe (fixed draw order, one ``torch.randn`` call per tensor or per expert):

1. hidden      [T, H]      N(0, 1)     -> bf16 (round to nearest even)
2. logits      [T, E]      N(0, 1)     fp32; the skewed workload adds
                                       b_e = fp32(-2 ln(e + 1)) to column e
3. W_gate_up   E x [2I, H] N(0, 0.02)  -> bf16, rows [0, I) gate, [I, 2I) up
4. W_down      E x [H, I]  N(0, 0.02)  -> bf16
5. Ws_gate_up  [2I_s, H]   N(0, 0.02)  -> bf16
6. Ws_down     [H, I_s]    N(0, 0.02)  -> bf16
7. w_g         [H]         N(0, 0.02)  -> bf16

The generator runs on ``device`` ("cpu" or "cuda"); the two devices give
different streams for the same seed, so a workload is named by
(config, seed, generator device).
"""
from __future__ import annotations

import dataclasses
import math

import torch

SOFTMAX = 0
SIGMOID = 1


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    I_s: int
    score_fn: int
    skew: bool = False

    def dims(self):
        return dict(T=self.T, H=self.H, E=self.E, k=self.k, I=self.I, I_s=self.I_s,
                    score_fn=self.score_fn)

    def with_tokens(self, T: int) -> "MoEConfig":
        return dataclasses.replace(self, T=T)


# The five workloads: tiny correctness case, decode-shaped, prefill-shaped,
# wide-expert (512 experts, top-10) and Zipf-skewed routing.
CONFIGS = {
    "tiny": MoEConfig("tiny", T=16, H=128, E=16, k=4, I=64, I_s=64, score_fn=SOFTMAX),
    "decode": MoEConfig("decode", T=64, H=2048, E=256, k=8, I=512, I_s=512, score_fn=SIGMOID),
    "prefill": MoEConfig("prefill", T=4096, H=2048, E=256, k=8, I=512, I_s=512, score_fn=SOFTMAX),
    "wide": MoEConfig("wide", T=2048, H=4096, E=512, k=10, I=1024, I_s=1024, score_fn=SIGMOID),
    "skewed": MoEConfig("skewed", T=8192, H=2048, E=256, k=8, I=512, I_s=512, score_fn=SOFTMAX,
                        skew=True),
}
CONFIG_ORDER = ["tiny", "decode", "prefill", "wide", "skewed"]


def skew_bias(E: int) -> torch.Tensor:
    """Per-expert logit bias of the skewed workload: fp32(-2 ln(rank)), rank = e + 1."""
    return torch.tensor([-2.0 * math.log(e + 1.0) for e in range(E)], dtype=torch.float64).to(
        torch.float32)


def _bf16(x: torch.Tensor, scale: float) -> torch.Tensor:
    if scale != 1.0:
        x = x * scale
    return x.to(torch.bfloat16)


def make_inputs(cfg: MoEConfig, seed: int = 0, device: str = "cpu",
                weights_device: str | None = None) -> dict:
    """Draw one workload. Returns a dict of tensors on ``weights_device``
    (default: ``device``). All tensors are contiguous row-major."""
    dev = torch.device(device)
    out_dev = torch.device(weights_device) if weights_device is not None else dev
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    T, H, E, I, I_s = cfg.T, cfg.H, cfg.E, cfg.I, cfg.I_s

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)

    hidden = _bf16(randn(T, H), 1.0).to(out_dev)
    logits = randn(T, E)
    if cfg.skew:
        logits = logits + skew_bias(E).to(dev)
    logits = logits.to(out_dev)
    w_gate_up = torch.empty(E, 2 * I, H, dtype=torch.bfloat16, device=out_dev)
    for e in range(E):
        w_gate_up[e].copy_(_bf16(randn(2 * I, H), 0.02))
    w_down = torch.empty(E, H, I, dtype=torch.bfloat16, device=out_dev)
    for e in range(E):
        w_down[e].copy_(_bf16(randn(H, I), 0.02))
    ws_gate_up = _bf16(randn(2 * I_s, H), 0.02).to(out_dev)
    ws_down = _bf16(randn(H, I_s), 0.02).to(out_dev)
    w_g = _bf16(randn(H), 0.02).to(out_dev)
    return dict(hidden=hidden, logits=logits.contiguous(), w_gate_up=w_gate_up, w_down=w_down,
                ws_gate_up=ws_gate_up, ws_down=ws_down, w_g=w_g)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def quantize_mxfp8(w: torch.Tensor):
    """MXFP8 encoding of bf16 weights [..., rows, K] (K a multiple of 32), the
    input format of the quantised-expert entry point: per row, each run of 32
    consecutive K elements shares the power-of-two scale 2^X with
    X = floor(log2(max |w|)) - 8 (8 = the largest E4M3 exponent), clamped to
    [-127, 127]; the elements are w / 2^X saturated to +-448 and rounded to
    the nearest E4M3 value (ties to even). Returns (codes uint8 [..., rows, K],
    scales uint8 [..., K / 32, rows] holding X + 127). Every step is exact
    (frexp, division by a power of two) up to the final rounding, so the codes
    are the same on every device. Input preparation only: the layer consumes
    the codes and scales as given."""
    *lead, rows, K = w.shape
    assert K % 32 == 0
    f = w.float().reshape(*lead, rows, K // 32, 32)
    amax = f.abs().amax(dim=-1)
    _, e = torch.frexp(amax)                      # amax = m 2^e, m in [0.5, 1)
    X = torch.where(amax > 0, e.float() - 1 - 8, torch.full_like(amax, -127.0)).clamp(-127, 127)
    q = (f / torch.exp2(X).unsqueeze(-1)).clamp(-448.0, 448.0)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(*lead, rows, K)
    scales = (X + 127).to(torch.uint8).transpose(-1, -2).contiguous()  # [..., K/32, rows]
    return codes.contiguous(), scales


def make_inputs_mxfp8(cfg: MoEConfig, seed: int = 0, device: str = "cpu") -> dict:
    """The bf16 inputs of make_inputs (drawn on ``device``) with every expert
    weight matrix (routed and shared) replaced by its MXFP8 encoding: <name>_q
    codes and <name>_s scales for w_gate_up, w_down, ws_gate_up and ws_down;
    hidden, logits and w_g unchanged."""
    inp = make_inputs(cfg, seed=seed, device=device)
    for name in ("w_gate_up", "w_down", "ws_gate_up", "ws_down"):
        w = inp.pop(name)
        if w.dim() == 3:   # expert by expert: bounded temporary memory
            pairs = [quantize_mxfp8(w[e]) for e in range(w.shape[0])]
            q, s = torch.stack([p[0] for p in pairs]), torch.stack([p[1] for p in pairs])
        else:
            q, s = quantize_mxfp8(w)
        inp[name + "_q"], inp[name + "_s"] = q, s
    return inp


def make_inputs_router(cfg: MoEConfig, seed: int = 0, device: str = "cpu") -> dict:
    """The inputs of make_inputs with the router logits replaced by router
    weights: w_router [E, H] ~ N(0, 0.02) -> bf16, drawn after w_g from the
    same generator (so the logits x . w_router^T have a spread close to the
    N(0, 1) logits of make_inputs). No logits entry."""
    dev = torch.device(device)
    inp = make_inputs(cfg, seed=seed, device=device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 7919)
    inp.pop("logits")
    inp["w_router"] = _bf16(torch.randn(cfg.E, cfg.H, generator=g, device=dev,
                                        dtype=torch.float32), 0.02)
    return inp


_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _round_e2m1(v: torch.Tensor) -> torch.Tensor:
    """E2M1 code (0..15) of the value nearest to v, ties to the even mantissa,
    saturating at +-6."""
    a = v.abs()
    # midpoints with the tie going to the even code: 0.25->0, 0.75->1.0, 1.25->1.0,
    # 1.75->2.0, 2.5->2.0, 3.5->4.0, 5->4.0
    mag = torch.zeros_like(a, dtype=torch.uint8)
    mag = torch.where(a > 0.25, 1, mag)
    mag = torch.where(a >= 0.75, 2, mag)
    mag = torch.where(a > 1.25, 3, mag)
    mag = torch.where(a >= 1.75, 4, mag)
    mag = torch.where(a > 2.5, 5, mag)
    mag = torch.where(a >= 3.5, 6, mag)
    mag = torch.where(a > 5.0, 7, mag)
    return (mag | torch.where(v < 0, 8, 0)).to(torch.uint8)


def quantize_nvfp4(w: torch.Tensor):
    """NVFP4 encoding of one bf16 weight matrix [rows, K] (K a multiple of 16),
    the input format of the NVFP4 entry point: a matrix scale
    g = max|w| / (6 * 448) (fp32), per row and 16 consecutive K values a block
    scale b = E4M3(max|w_block| / (6 g)) (round to nearest), and codes
    E2M1(w / (b g)) (nearest, ties to even, saturating at +-6), two per byte
    with the lower K index in the low nibble. Returns (codes uint8 [rows, K/2],
    scales uint8 [K/16, rows], g fp32 scalar tensor). Input preparation only."""
    rows, K = w.shape
    assert K % 16 == 0
    f = w.float()
    amax = f.abs().max()
    g = (amax / (6.0 * 448.0)).clamp_min(2.0 ** -126)
    blk = f.reshape(rows, K // 16, 16)
    bmax = blk.abs().amax(dim=-1)
    b = (bmax / (6.0 * g)).clamp(max=448.0).to(torch.float8_e4m3fn)
    bv = b.float()
    q = blk / (bv * g).clamp_min(2.0 ** -126).unsqueeze(-1)
    codes = _round_e2m1(q).reshape(rows, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8).contiguous()
    scales = b.view(torch.uint8).transpose(0, 1).contiguous()
    return packed, scales, g.to(torch.float32)


def make_inputs_nvfp4(cfg: MoEConfig, seed: int = 0, device: str = "cpu") -> dict:
    """The bf16 inputs of make_inputs (drawn on ``device``) with every expert
    weight matrix encoded by quantize_nvfp4: <name>_q codes, <name>_s block
    scales and <name>_g matrix scales (fp32, [E] for the expert stacks, [1]
    for the shared expert) for w_gate_up, w_down, ws_gate_up and ws_down."""
    inp = make_inputs(cfg, seed=seed, device=device)
    for name in ("w_gate_up", "w_down", "ws_gate_up", "ws_down"):
        w = inp.pop(name)
        mats = [w[e] for e in range(w.shape[0])] if w.dim() == 3 else [w]
        enc = [quantize_nvfp4(m) for m in mats]
        q = torch.stack([x[0] for x in enc])
        s = torch.stack([x[1] for x in enc])
        g = torch.stack([x[2] for x in enc]).reshape(-1)
        if w.dim() == 2:
            q, s = q[0], s[0]
        inp[name + "_q"], inp[name + "_s"], inp[name + "_g"] = q, s, g
    return inp
