"""Host-side accounting of bench.py (no GPU): the algorithmic bytes and FLOPs
the roofline divides by, and the rule that a committed ncu summary's DRAM
traffic counts only while its recorded source hash matches the kernel
sources."""
from __future__ import annotations

import hashlib
import os

import pytest

import bench
from mixture_experts_ffn_03_gb300 import workloads as wl


def test_algorithmic_work_by_hand():
    # T=2, H=64, E=4, k=2, I=64, I_s=128; experts 0 and 2 receive tokens
    cfg = wl.MoEConfig("w", T=2, H=64, E=4, k=2, I=64, I_s=128, score_fn=wl.SOFTMAX)
    w = bench.algorithmic_work(cfg, [3, 0, 1, 0])
    T, H, E, k, I, Is = 2, 64, 4, 2, 64, 128
    assert w["touched"] == 2
    # routed: 2 T k H I (gate) + 2 T k H I (up) + 2 T k I H (down); shared likewise; gate x.w_g
    assert w["flops"] == 6 * H * I * T * k + 6 * H * Is * T + 2 * H * T
    weights = 2 * (3 * I * H) * 2 + 3 * Is * H * 2  # two touched experts + shared, bf16
    act = 2 * T * H + 4 * T * E + 2 * T * H          # hidden in, logits in, out
    assert w["bytes"] == weights + 2 * H + act
    assert w["gate_up_bytes"] == 2 * (2 * I * H) * 2 + 2 * Is * H * 2 + 2 * T * H
    assert w["down_bytes"] == 2 * (I * H) * 2 + Is * H * 2
    assert w["gate_up_flops"] + w["down_flops"] == w["flops"] - 2 * H * T


def test_algorithmic_work_quantised_weight_bytes():
    cfg = wl.CONFIGS["decode"]
    counts = [1] * cfg.E
    bf = bench.algorithmic_work(cfg, counts)
    mx = bench.algorithmic_work(cfg, counts, wbytes=1.0 + 1.0 / 32)
    w_bf = 3.0 * cfg.H * (cfg.E * cfg.I + cfg.I_s) * 2.0
    assert bf["bytes"] - mx["bytes"] == pytest.approx(w_bf / 2.0 * (1.0 - 1.0 / 32))
    assert mx["flops"] == bf["flops"]


def _write_profile(path, sha, nbytes):
    path.write_text("# summary\n\n- kernel: k\n- workload: decode\n"
                    f"- dram_bytes_per_launch_full: {nbytes}\n- source_sha256: {sha}\n")


def test_read_traffic_requires_matching_source_hash(tmp_path, monkeypatch):
    csrc = os.path.join(bench.ROOT, "mixture_experts_ffn_03_gb300", "csrc")
    h = hashlib.sha256()
    for f in bench.KERNEL_SOURCES["moe_gate_up"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    root = tmp_path
    (root / "profiles").mkdir()
    os.symlink(os.path.join(bench.ROOT, "mixture_experts_ffn_03_gb300"),
               root / "mixture_experts_ffn_03_gb300")
    monkeypatch.setattr(bench, "ROOT", str(root))
    prof = root / "profiles" / "moe_gate_up_decode.md"
    _write_profile(prof, h.hexdigest(), 123456)
    assert bench.read_traffic("moe_gate_up", "decode") == 123456.0
    _write_profile(prof, "0" * 64, 123456)                 # taken on other sources
    assert bench.read_traffic("moe_gate_up", "decode") is None
    assert bench.read_traffic("moe_gate_up", "prefill") is None  # no summary

