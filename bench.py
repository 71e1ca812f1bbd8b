"""Benchmark of the MoE FFN layer on GB300: tokens/s and roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One step = one moe_forward (route, permute, gate_up GEMM, down GEMM, shared
expert, combine) over the workload's T tokens, inputs resident in HBM. The
headline workload is the largest one that fits one GPU (wide: T=2048,
H=4096, 512 experts, top-10, I=1024, ~13 GB of expert weights). Each timed
step is bracketed by CUDA events on the launching stream; between steps L2 is
flushed by a 256 MB write followed by a 256 MB read of a second buffer, so
each step starts with no layer data in L2 and no dirty lines whose
write-back would fall inside the step. Per-kernel times come from events the
library records around each of its kernels on the same stream. At one GPU the
decode, prefill and skewed workloads are then timed the same way and
reported under per_config. Prints one JSON line (rank 0).

--impl reference times the fp64 CPU oracle on the host cores instead (a
bounded token sample per step), with the same metric and workload.
Multi-GPU runs (torchrun) are independent replicas by default; --ep spreads
the experts over the ranks instead (expert parallelism, two all-to-alls per
step), and --ep --ep-ranks G runs G such ranks one after another on one GPU.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
DEFAULT_CONFIG = "wide"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        hbm = float(p.get("hbm_gbs"))
        tf = float(p.get("bf16_tflops"))
        tfs = float(p.get("bf16_tflops_sustained", tf))
        return dict(hbm_gbs=hbm, bf16_tflops=tf, bf16_tflops_sustained=tfs, source="measured")
    except Exception:
        return dict(hbm_gbs=FALLBACK_HBM_GBS, bf16_tflops=FALLBACK_BF16_TFLOPS,
                    bf16_tflops_sustained=1700.0, source="fallback")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(local_ms: float, dist, device) -> float:
    """The slowest rank's timed total: every rank's time is all-reduced with MAX."""
    import torch
    t = torch.tensor([local_ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_step: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: the tokens every replica processed over the slowest rank's time."""
    return world * tokens_per_step * steps / (total_ms / 1e3)


def workload_name(cfg):
    sf = "softmax" if cfg.score_fn == 0 else "sigmoid"
    from mixture_experts_ffn_03_gb300 import workloads as wl
    full = wl.CONFIGS.get(cfg.name)
    reduced = full is not None and (full.T, full.E) != (cfg.T, cfg.E)
    return (f"{cfg.name}{' (reduced)' if reduced else ''}: T={cfg.T} H={cfg.H} E={cfg.E} "
            f"k={cfg.k} I={cfg.I} I_s={cfg.I_s} "
            f"{sf}+renorm{', zipf-skewed logits' if cfg.skew else ''}")


def algorithmic_work(cfg, counts, wbytes=2.0):
    """Layer FLOPs and touched bytes from the actual routing (counts per expert);
    wbytes = bytes per expert weight (2 for bf16, 1 + 1/32 for MXFP8 codes and
    scales)."""
    T, H, E, k, I, I_s = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.I_s
    touched = int(sum(1 for c in counts if c > 0))
    flops = 6.0 * H * I * T * k + 6.0 * H * I_s * T + 2.0 * H * T
    w_routed = touched * 3.0 * wbytes * I * H
    w_shared = 3.0 * wbytes * I_s * H
    act = 2.0 * T * H + 4.0 * T * E + 2.0 * T * H
    bytes_total = w_routed + w_shared + 2.0 * H + act
    gate_up_bytes = touched * 2.0 * wbytes * I * H + 2.0 * wbytes * I_s * H + 2.0 * T * H
    gate_up_flops = 4.0 * H * I * T * k + 4.0 * H * I_s * T
    down_bytes = touched * wbytes * I * H + wbytes * I_s * H
    down_flops = 2.0 * H * I * T * k + 2.0 * H * I_s * T
    return dict(touched=touched, flops=flops, bytes=bytes_total, gate_up_bytes=gate_up_bytes,
                gate_up_flops=gate_up_flops, down_bytes=down_bytes, down_flops=down_flops)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        time.sleep(0.06)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(smax) if smax else None, reasons=sorted(reasons),
                    samples=len(sm))


# Sources of each profiled kernel: a summary's traffic counts only while
# their hash matches the one recorded with it.
KERNEL_SOURCES = {
    "moe_gate_up": ("moe_gemm.cu", "gemm_common.cuh", "ptx.cuh", "moe_internal.cuh"),
    "moe_gate_up_mxfp8": ("moe_gemm_mx.cu", "mxfp8.cuh", "gemm_common.cuh", "ptx.cuh",
                          "moe_internal.cuh"),
    "moe_gate_up_nvfp4": ("moe_gemm_mx.cu", "mxfp8.cuh", "gemm_common.cuh", "ptx.cuh",
                          "moe_internal.cuh"),
    "moe_expert_fused": ("moe_fused.cu", "moe_fused.cuh", "routing.cuh", "gemm_common.cuh",
                         "ptx.cuh", "moe_internal.cuh"),
    "moe_layer_fused": ("moe_fused.cu", "moe_fused.cuh", "routing.cuh", "gemm_common.cuh",
                        "ptx.cuh", "moe_internal.cuh"),
}


def read_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if the
    summary was taken on the current kernel source."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "mixture_experts_ffn_03_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            key, _, v = line.strip()[2:].partition(":")
            vals[key.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != h.hexdigest():
        return None
    try:
        return float(vals["dram_bytes_per_launch_full"])
    except (KeyError, ValueError):
        return None


def torch_index(toks):
    import torch
    return torch.as_tensor(toks, dtype=torch.long)


def run_reference(args, cfg):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from mixture_experts_ffn_03_gb300 import workloads as wl
    inp = wl.make_inputs(cfg, seed=0)
    threads = oracle.default_threads()
    # Size the per-step token sample so that the whole timed run takes about
    # a minute (at most ~2 s per step), at least one token per thread.
    batch = np.arange(min(cfg.T, threads))
    for _ in range(args.warmup):
        oracle.moe_forward(inp, cfg.k, cfg.score_fn, tokens=batch, n_threads=threads)
    t0 = time.perf_counter()
    oracle.moe_forward(inp, cfg.k, cfg.score_fn, tokens=batch, n_threads=threads)
    per_batch = time.perf_counter() - t0
    budget = min(2.0, 60.0 / max(args.steps, 1))
    n_tok = int(max(len(batch), len(batch) * int(budget / max(per_batch, 1e-3))))
    toks = np.arange(n_tok) % cfg.T
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.moe_forward(inp, cfg.k, cfg.score_fn, tokens=toks, n_threads=threads)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = n_tok * len(times) / total
    sample = (f"{n_tok} token evaluations per step (token index mod {cfg.T}), fp64, all routed "
              f"+ shared experts, {threads} OpenMP threads")
    line = dict(impl="reference", metric="MoE-layer tokens/s", value=value, unit="tokens/s",
                n_gpus=world, steps=args.steps, warmup=args.warmup,
                ms_per_step=1e3 * total / len(times), higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic",
                config=dict(workload=workload_name(cfg), seed=0),
                cpu_baseline=dict(value=value, unit="tokens/s", cores=threads, kind="oracle",
                                  sample=sample),
                e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


def time_cpu_baseline(cfg, inp_cpu, budget_s=12.0, router=False, threads=None):
    """The oracle on the host cores over a bounded token sample (about budget_s
    of CPU work): tokens/s and the threads it used."""
    import numpy as np
    import oracle
    threads = threads or oracle.default_threads()
    n = min(cfg.T, threads)
    if router:  # the router's logits for the sampled tokens, then the layer
        def run(toks):
            x = inp_cpu["hidden"][torch_index(toks)]
            lg = oracle.router_logits(x, inp_cpu["w_router"]).astype(np.float32)
            plain = {k: v for k, v in inp_cpu.items() if k != "w_router"}
            plain["hidden"] = x
            plain["logits"] = lg
            oracle.moe_forward(plain, cfg.k, cfg.score_fn, n_threads=threads)
    else:
        def run(toks):
            oracle.moe_forward(inp_cpu, cfg.k, cfg.score_fn, tokens=toks, n_threads=threads)
    t0 = time.perf_counter()
    run(np.arange(n))
    dt = time.perf_counter() - t0
    reps = max(1, int(budget_s / max(dt, 1e-3)))
    n_tok = n * reps  # about budget_s of CPU work
    toks = np.arange(n_tok) % cfg.T
    t0 = time.perf_counter()
    run(toks)
    dt = time.perf_counter() - t0
    return dict(value=n_tok / dt, unit="tokens/s", cores=threads, kind="oracle",
                sample=f"{n_tok} tokens of the {cfg.name} workload (token t mod {cfg.T}), fp64, "
                       f"{dt:.1f} s")


# Workloads timed after the headline one, each with the same step timing and
# L2 flush, and reported under per_config (one GPU, bf16 weights only).
PER_CONFIG = ("decode", "prefill", "skewed")


def make_layer(args, cfg, dev):
    """Seeded inputs on the device and the layer object for the chosen weights."""
    from mixture_experts_ffn_03_gb300 import workloads as wl
    import mixture_experts_ffn_03_gb300 as moe
    if args.router:
        inp = wl.make_inputs_router(cfg, seed=0, device=str(dev))
        layer = moe.MoELayerRouter(inp["w_router"], inp["w_gate_up"], inp["w_down"],
                                   inp["ws_gate_up"], inp["ws_down"], inp["w_g"], cfg.k,
                                   cfg.score_fn)
        inp["logits"] = None
    elif args.weights == "nvfp4":
        inp = wl.make_inputs_nvfp4(cfg, seed=0, device=str(dev))
        tri = lambda n: (inp[n + "_q"], inp[n + "_s"], inp[n + "_g"])  # noqa: E731
        layer = moe.MoELayerNVFP4(tri("w_gate_up"), tri("w_down"), tri("ws_gate_up"),
                                  tri("ws_down"), inp["w_g"], cfg.k, cfg.score_fn)
    elif args.weights == "mxfp8":
        inp = wl.make_inputs_mxfp8(cfg, seed=0, device=str(dev))
        pair = lambda n: (inp[n + "_q"], inp[n + "_s"])  # noqa: E731
        layer = moe.MoELayerMXFP8(pair("w_gate_up"), pair("w_down"), pair("ws_gate_up"),
                                  pair("ws_down"), inp["w_g"], cfg.k, cfg.score_fn)
    else:
        inp = wl.make_inputs(cfg, seed=0, device=str(dev))
        layer = moe.MoELayer(inp["w_gate_up"], inp["w_down"], inp["ws_gate_up"], inp["ws_down"],
                             inp["w_g"], cfg.k, cfg.score_fn)
    return inp, layer


class L2Flush:
    """Between timed steps: write 256 MB (evicts the layer's data), then read
    another 256 MB so the written lines leave L2 before the step; their
    write-back would otherwise take DRAM bandwidth inside the next step."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self, i):
        import torch
        self.w.fill_(i & 0xFF)
        torch.sum(self.r, dim=(0,), out=self.sink)


def measure(args, cfg, dev, layer, inp, stream, flush, K, sampler=None, dist=None):
    """Warm-up, then K timed steps (CUDA events on the launching stream around
    each step), then a separate pass of K steps with the library's per-kernel
    events. Returns the step times, per-stage times, routing counts and the
    launch accounting."""
    import torch
    import mixture_experts_ffn_03_gb300 as moe
    mx, nv = args.weights == "mxfp8", args.weights == "nvfp4"
    T = cfg.T
    out = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=dev)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            layer.forward(inp["hidden"], inp["logits"], out=out, counts=counts, stream=stream)
    st = moe.device_status(layer.workspace(T), stream)
    if st != moe.MOE_OK:
        raise RuntimeError(moe.status_string(st))
    if mx or nv:
        n_launch = n_separate = moe.launch_count_quantized(layer.dims(T))
    else:
        count = moe.launch_count_router if args.router else moe.launch_count
        n_launch = count(layer.dims(T))
        with moe.expert_fusion(False):
            n_separate = count(layer.dims(T))
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.NUM_STAGES + 1)]
                for _ in range(K)]
    # torch creates CUDA events lazily; record each once so the handles exist.
    with torch.cuda.stream(stream):
        for evs in stage_ev:
            for e in evs:
                e.record(stream)
    torch.cuda.synchronize(dev)

    # Timed region: K steps, each bracketed by events on the launching stream.
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if sampler is not None:
        sampler.start()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush(i)
            step_ev[i][0].record(stream)
            layer.forward(inp["hidden"], inp["logits"], out=out, stream=stream)
            step_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler is not None else None
    if dist is not None:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]

    # Per-kernel pass: the library records events around each of its kernels
    # on the same stream (this serialises the kernels, so it is a separate
    # pass of K steps and not part of the step timing above).
    with torch.cuda.stream(stream):
        for i in range(K):
            flush(i)
            moe.set_stage_events(stage_ev[i])
            layer.forward(inp["hidden"], inp["logits"], out=out, stream=stream)
    moe.set_stage_events(None)
    torch.cuda.synchronize(dev)
    st = moe.device_status(layer.workspace(T), stream)
    if st != moe.MOE_OK:
        raise RuntimeError(moe.status_string(st))
    stage_ms = [[evs[j].elapsed_time(evs[j + 1]) for evs in stage_ev]
                for j in range(moe.NUM_STAGES)]
    return dict(step_ms=step_ms, stage_ms=stage_ms, counts=counts.cpu().tolist(), out=out,
                n_launch=n_launch, fused=n_launch < n_separate, layer=n_launch == 1, wall=wall,
                clocks=clocks)


def work_of(args, cfg, m):
    """Algorithmic work of one step and the name of the dominant kernel."""
    mx, nv = args.weights == "mxfp8", args.weights == "nvfp4"
    work = algorithmic_work(cfg, m["counts"],
                            wbytes=1.0 + 1.0 / 32 if mx else (0.5 + 1.0 / 16 if nv else 2.0))
    if args.router:  # W_router read and x . W_router^T computed instead of logits read
        work["flops"] += 2.0 * cfg.T * cfg.E * cfg.H
        work["bytes"] += 2.0 * cfg.E * cfg.H - 4.0 * cfg.T * cfg.E
    gu_kernel = "moe_gate_up_mxfp8" if mx else ("moe_gate_up_nvfp4" if nv else "moe_gate_up")
    if m["layer"]:
        # the whole layer is one launch (the routing stage of the per-kernel events)
        gu_kernel = "moe_layer_fused"
        work["gate_up_bytes"] = work["bytes"]
        work["gate_up_flops"] = work["flops"]
    elif m["fused"]:
        # gate_up and down run as one launch (the gate_up stage of the per-kernel events)
        gu_kernel = "moe_expert_fused"
        work["gate_up_bytes"] += work["down_bytes"]
        work["gate_up_flops"] += work["down_flops"]
    return work, gu_kernel


def rooflines(cfg, work, m, peaks, gu_kernel):
    """`roofline` of the dominant kernel (gate_up, or the fused expert launch)
    and `layer_roofline` of the whole step."""
    ms_step = sum(m["step_ms"]) / len(m["step_ms"])
    gu_ms = statistics.mean(m["stage_ms"][0 if m["layer"] else 2])
    hbm_bound = work["bytes"] / (peaks["hbm_gbs"] * 1e9) >= work["flops"] / (
        peaks["bf16_tflops_sustained"] * 1e12)
    kname = ("moe_layer_fused (routing, gate_up, down and combine in one launch)" if m["layer"]
             else f"{gu_kernel} grouped GEMM" + (" (gate_up + down)" if m["fused"] else ""))
    if hbm_bound:
        achieved = work["gate_up_bytes"] / (gu_ms / 1e3) / 1e9
        roof = dict(bound="hbm", achieved=achieved, peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=achieved / peaks["hbm_gbs"], traffic=read_traffic(gu_kernel, cfg.name),
                    kernel=kname, peak_source=peaks["source"])
    else:
        achieved = work["gate_up_flops"] / (gu_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = dict(bound="tensor", achieved=achieved, peak=peak, unit="TFLOP/s",
                    frac=achieved / peak, traffic=read_traffic(gu_kernel, cfg.name),
                    kernel=kname, peak_source=peaks["source"])
    t_roof = max(work["bytes"] / (peaks["hbm_gbs"] * 1e9),
                 work["flops"] / (peaks["bf16_tflops_sustained"] * 1e12))
    layer_roof = dict(bound="hbm" if hbm_bound else "tensor", roofline_ms=t_roof * 1e3,
                      frac=t_roof * 1e3 / ms_step, bytes=work["bytes"], flops=work["flops"],
                      experts_touched=work["touched"],
                      frac_vs_nominal_8tbs=(work["bytes"] / 8e12 * 1e3) / ms_step)
    return roof, layer_roof


def kernel_us(m):
    import mixture_experts_ffn_03_gb300 as moe
    return {n: round(statistics.mean(v) * 1e3, 2) for n, v in zip(moe.STAGE_NAMES, m["stage_ms"])}


def measure_per_config(args, dev, stream, flush, peaks, names):
    """The other workloads at one GPU: ms/step, tokens/s, the layer and
    dominant-kernel roofline fractions and the per-kernel times."""
    import torch
    from mixture_experts_ffn_03_gb300 import workloads as wl
    res = {}
    for name in names:
        cfg = wl.CONFIGS[name]
        inp, layer = make_layer(args, cfg, dev)
        m = measure(args, cfg, dev, layer, inp, stream, flush, args.steps)
        work, gu_kernel = work_of(args, cfg, m)
        roof, layer_roof = rooflines(cfg, work, m, peaks, gu_kernel)
        ms = sum(m["step_ms"]) / len(m["step_ms"])
        res[name] = dict(workload=workload_name(cfg), ms_per_step=ms, value=cfg.T / (ms / 1e3),
                         unit="tokens/s",
                         layer_roofline=dict(bound=layer_roof["bound"],
                                             roofline_ms=layer_roof["roofline_ms"],
                                             frac=layer_roof["frac"]),
                         roofline=dict(bound=roof["bound"], kernel=roof["kernel"],
                                       achieved=roof["achieved"], unit=roof["unit"],
                                       frac=roof["frac"]),
                         kernel_us=kernel_us(m), gpu_launches=m["n_launch"] * args.steps)
        del inp, layer, m
        torch.cuda.empty_cache()
    return res


def run_expert_parallel(args, cfg):
    """--ep: the layer spread over the ranks by expert parallelism (rank g holds
    experts [g E/N, (g+1) E/N) and the shared expert; every rank routes the
    workload's T tokens; two all-to-all exchanges per step over NCCL). At one
    GPU, --ep-ranks G runs G ranks one after another on that GPU (in-process
    exchange). Whole-job tokens/s over the slowest rank's time."""
    import torch
    import mixture_experts_ffn_03_gb300 as moe
    from mixture_experts_ffn_03_gb300 import expert_parallel as ep
    from mixture_experts_ffn_03_gb300 import workloads as wl
    rank, world, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    moe.load_library()
    G = world if world > 1 else max(1, args.ep_ranks)
    if cfg.E % G:
        raise SystemExit(f"E={cfg.E} is not a multiple of {G} ranks")
    e_loc = cfg.E // G
    full = wl.make_inputs(cfg, seed=0, device=str(dev))
    mine = [rank] if world > 1 else list(range(G))
    layers = []
    for g in mine:
        layers.append(ep.ExpertParallelMoE(
            g, G, full["w_gate_up"][g * e_loc:(g + 1) * e_loc].clone(),
            full["w_down"][g * e_loc:(g + 1) * e_loc].clone(), full["ws_gate_up"],
            full["ws_down"], full["w_g"], cfg.E, cfg.k, cfg.score_fn, cfg.T))
    hidden, logits = full["hidden"], full["logits"]
    del full["w_gate_up"], full["w_down"]
    torch.cuda.empty_cache()
    flush = L2Flush(dev)

    def step():
        if world > 1:
            return [layers[0].forward(hidden, logits)]
        return ep.LocalExchange(layers).forward([hidden] * G, [logits] * G)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index)
    sampler.start()
    for i in range(K):
        flush(i)
        evs[i][0].record()
        step()
        evs[i][1].record()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    total_ms = sum(a.elapsed_time(b) for a, b in evs)
    if dist is not None:
        total_ms = max_over_ranks(total_ms, dist, dev)
    for layer in layers:
        st = moe.device_status(layer._ws)
        if st != moe.MOE_OK:
            raise RuntimeError(moe.status_string(st))
    if rank == 0:
        tokens = G * cfg.T   # every rank routes T tokens per step
        line = dict(
            metric="MoE-layer tokens/s", value=tokens * K / (total_ms / 1e3), unit="tokens/s",
            n_gpus=world, steps=K, warmup=args.warmup, ms_per_step=total_ms / K,
            higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16",
            data="synthetic",
            config=dict(workload=workload_name(cfg), seed=0, weights="bf16",
                        parallelism=f"ep{G}" + (" (ranks emulated on one GPU)" if world == 1 else ""),
                        experts_per_rank=e_loc, tokens_per_rank=cfg.T,
                        l2="flushed between timed steps: 256 MB write, then 256 MB read",
                        launch="stream; host synchronises once per exchange for the row counts"),
            gpu_launches=None, clocks=clocks)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the --config workload (skip per_config)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "mxfp8", "nvfp4"],
                    help="expert weight format: bf16, MXFP8 (moe_forward_mxfp8) or NVFP4 "
                         "(moe_forward_nvfp4)")
    ap.add_argument("--router", action="store_true",
                    help="compute the router logits in the layer from W_router (moe_forward_router)")
    ap.add_argument("--ep", action="store_true",
                    help="expert parallelism over the ranks (NCCL all-to-all exchanges)")
    ap.add_argument("--ep-ranks", type=int, default=1,
                    help="with --ep on one GPU: ranks to run one after another on it")
    ap.add_argument("--tokens", type=int, default=None,
                    help="reduced workload for profiling captures: this many tokens")
    ap.add_argument("--experts", type=int, default=None,
                    help="reduced workload for profiling captures: this many experts")
    ap.add_argument("--fusion", type=int, nargs="?", const=1, default=0,
                    help="launch fusion (bf16 weights, decode-sized batches; off by default): "
                         "1 gate_up + down in one launch, 2 the whole layer in one launch")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from mixture_experts_ffn_03_gb300 import workloads as wl
    cfg = wl.CONFIGS[args.config]
    if args.tokens is not None or args.experts is not None:
        # same shapes per expert, fewer tokens or experts (a capture that fits the
        # profiler's memory budget); never the headline line's workload
        import dataclasses
        cfg = dataclasses.replace(cfg, T=args.tokens if args.tokens is not None else cfg.T,
                                  E=args.experts if args.experts is not None else cfg.E)
        args.no_per_config = True
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.ep:
        return run_expert_parallel(args, cfg)

    import numpy as np
    import torch
    import mixture_experts_ffn_03_gb300 as moe

    rank, world, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    moe.load_library()
    moe.set_expert_fusion(args.fusion)

    mx = args.weights == "mxfp8"
    nv = args.weights == "nvfp4"
    if (mx or nv) and args.router:
        raise SystemExit("--router runs with bf16 expert weights")
    inp, layer = make_layer(args, cfg, dev)
    T = cfg.T
    K = args.steps
    stream = torch.cuda.Stream(dev)
    flush = L2Flush(dev)
    m = measure(args, cfg, dev, layer, inp, stream, flush, K, sampler=ClockSampler(dev.index),
                dist=dist)
    out = m["out"]
    total_ms = sum(m["step_ms"])
    if dist is not None:
        total_ms = max_over_ranks(total_ms, dist, dev)
    work, gu_kernel = work_of(args, cfg, m)

    # The same step replayed as a CUDA graph (launch overhead removed).
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            layer.forward(inp["hidden"], inp["logits"], out=out)
        cap.synchronize()
        with torch.cuda.graph(g, stream=cap):
            layer.forward(inp["hidden"], inp["logits"], out=out)
        torch.cuda.synchronize(dev)
        g_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(K)]
        with torch.cuda.stream(stream):
            for i in range(K):
                flush(i)
                g_ev[i][0].record(stream)
                g.replay()
                g_ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        g_ms = sum(a.elapsed_time(b) for a, b in g_ev) / K
        graph = dict(ms_per_step=g_ms, value=T / (g_ms / 1e3), unit="tokens/s")
        del g
    except Exception as exc:  # capture unsupported here: report, do not fail the bench
        graph = dict(error=str(exc)[:200])

    # End to end through the public API: pinned host inputs in, output back,
    # every step's transfers inside the timed region. Serial: one step at a time
    # on one stream (L2 flushed between steps, outside the step events).
    h_host = inp["hidden"].cpu().pin_memory()
    l_host = None if args.router else inp["logits"].cpu().pin_memory()
    o_hosts = [torch.empty(T, cfg.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    o_host = o_hosts[0]
    with torch.cuda.stream(stream):
        for _ in range(3):
            layer.forward_from_host(h_host, l_host, o_host, stream=stream)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(K):
            flush(i)
            e2e_ev[i][0].record(stream)
            layer.forward_from_host(h_host, l_host, o_host, stream=stream)
            e2e_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_serial_ms = sum(a.elapsed_time(b) for a, b in e2e_ev)
    # Serving loop (moe.HostPipeline): each step's input copy overlaps the previous
    # step's compute and its output copy the next step's (input and output copies on
    # streams of their own). The weights streamed every step are far larger than L2,
    # so no flush is interleaved; the timed span runs from before the first input
    # copy to after the last output copy.
    # The plain bf16 layer runs the library's own serving loop (moe_pipeline_submit:
    # host buffers through the C ABI); the other entry points the binding's loop.
    native = type(layer) is moe.MoELayer
    pipe = (moe.NativePipeline if native else moe.HostPipeline)(layer, T, compute_stream=stream)
    for i in range(3):
        pipe.submit(h_host, l_host, o_hosts[i % 2])
    pipe.drain()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    pipe.xs.wait_event(p0)
    for i in range(K):
        pipe.submit(h_host, l_host, o_hosts[i % 2])
    p1.record(pipe.ys)  # after the last output copy
    pipe.drain()
    e2e_ms = p0.elapsed_time(p1)
    if native:
        pipe.close()
    del pipe

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks = load_peaks()
    value = job_tokens_per_s(world, T, K, total_ms)
    ms_step = total_ms / K
    roof, layer_roof = rooflines(cfg, work, m, peaks, gu_kernel)
    layer_roof["frac"] = layer_roof["roofline_ms"] / ms_step  # the slowest rank's time
    dn_ms = statistics.mean(m["stage_ms"][3])
    h2d = T * cfg.H * 2 + (0 if args.router else T * cfg.E * 4)
    d2h = T * cfg.H * 2
    line = dict(
        metric="MoE-layer tokens/s", value=value, unit="tokens/s", n_gpus=world, steps=K,
        warmup=args.warmup, ms_per_step=ms_step, higher_is_better=True, scaling="weak",
        vs_baseline=None,
        dtype=("bf16 (MXFP8 E4M3 weights, exact to bf16)" if mx else
               "bf16 (NVFP4 E2M1 weights with E4M3 block scales, exact to bf16; fp32 matrix scales)"
               if nv else "bf16"),
        data="synthetic",
        config=dict(workload=workload_name(cfg), seed=0, weights=args.weights,
                    router="in the layer (moe_forward_router)" if args.router else "logits input",
                    parallelism="replicas" if world > 1 else "1gpu",
                    l2="flushed between timed steps: 256 MB write, then 256 MB read of a "
                       "second buffer (no dirty lines left)", launch="stream",
                    experts=("the whole layer in one launch" if m["layer"] else
                             "one fused gate_up + down launch" if m["fused"]
                             else "gate_up and down launches"),
                    wall_s=round(m["wall"], 3)),
        roofline=roof, layer_roofline=layer_roof, kernel_us=kernel_us(m),
        kernel_timing="separate pass of K steps with library-recorded events around each kernel",
        down_gbs=None if (m["fused"] or m["layer"]) else work["down_bytes"] / (dn_ms / 1e3) / 1e9,
        e2e=dict(value=world * T * K / (e2e_ms / 1e3), unit="tokens/s", h2d_bytes_per_step=h2d,
                 d2h_bytes_per_step=d2h,
                 mode=("serving loop through the C ABI (moe_pipeline_submit, host buffers)"
                       if native else "serving loop (moe.HostPipeline)") +
                      ": transfers overlap neighbouring steps' compute",
                 serial_value=world * T * K / (e2e_serial_ms / 1e3)),
        gpu_launches=m["n_launch"] * K,
        clocks=m["clocks"], cuda_graph=graph)
    if world == 1 and not args.no_cpu_baseline:
        inp_cpu = {n: t.cpu() for n, t in inp.items() if t is not None}
        if mx or nv:
            # the oracle's quantised layer is its bf16 layer on the exactly dequantised
            # weights (NVFP4: plus the matrix scales): dequantise once, then time that layer
            import oracle
            deq = oracle.nvfp4_to_bf16 if nv else oracle.mxfp8_to_bf16
            for n in ("w_gate_up", "w_down", "ws_gate_up", "ws_down"):
                bits = deq(oracle._np(inp_cpu.pop(n + "_q")), oracle._np(inp_cpu.pop(n + "_s")))
                inp_cpu[n] = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        line["cpu_baseline"] = time_cpu_baseline(cfg, inp_cpu, router=args.router)
        del inp_cpu
    del inp, layer, m, out
    torch.cuda.empty_cache()
    others = [n for n in PER_CONFIG if n != cfg.name]
    if world == 1 and not args.no_per_config and others:
        line["per_config"] = measure_per_config(args, dev, stream, flush, peaks, others)
        line["per_config_timing"] = ("same step timing, L2 flush and per-kernel pass as the "
                                     "headline, K steps each, after the headline's timed region")
    if world == 1 and not args.no_cpu_baseline and not (mx or nv or args.router):
        # the oracle on one host core, on the decode workload
        dcfg = wl.CONFIGS["decode"]
        d_cpu = wl.make_inputs(dcfg, seed=0, device=str(dev))
        d_cpu = {n: t.cpu() for n, t in d_cpu.items()}
        line["cpu_baseline"]["single_core"] = dict(
            workload=workload_name(dcfg),
            **time_cpu_baseline(dcfg, d_cpu, budget_s=8.0, threads=1))
        del d_cpu
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
