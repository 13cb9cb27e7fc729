#!/usr/bin/env python
"""Throughput of the DeepSeekMoE layer forward with auxiliary-loss-free routing.

Workload (default): the DeepSeek-V3-shaped bf16 layer — T=8192 tokens (2 sequences of
4096), d=7168, 256 routed experts with top-8 routing limited to 4 of 8 expert groups,
1 shared expert, SwiGLU width 2048.  One step = route (affinity GEMM, sigmoid, biased
group-limited top-8, gates, per-sequence P sums) -> dispatch (counts, permutation,
row gather) -> gate/up GEMM with SwiGLU -> down GEMM -> combine with residual -> bias
update -> sequence-wise balance statistic, all through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The timed region replays a CUDA graph of exactly K captured steps (kernel launches
through the C ABI, recorded once), so the host adds no per-kernel overhead.

Prints one JSON line.  Under torchrun each rank runs an independent replica of the
layer on its own batch (weak scaling); rank 0 prints the line with the whole-job
throughput computed from the slowest rank's time.  ``--impl reference`` times the
CPU oracle on bounded samples of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer fwd tokens/s at d=7168, 256e top-8; tensor-pipe & HBM % of peak"

# DRAM traffic of the gate/up GEMM, from one ncu capture (not measured in the bench
# run): dram__bytes_read.sum + dram__bytes_write.sum = 2.2442 GB + 0.0354 GB on the
# V3-shaped slice (32 experts, 1024 tokens, d=7168, I=2048, ~3 GB on the device), whose
# algorithmic bytes are 2.108 GB: 1.081 bytes moved per algorithmic byte.  A full V3
# launch holds eight times the slice's segments with the same mean load (256 tokens), so
# its traffic is taken as that ratio times its own algorithmic bytes.  Valid only for
# the kernel source with this hash.
NCU_TRAFFIC = {"kernel_src_sha": "92b1cd4f04c98f6f", "ratio": 2.2796e9 / 2.108e9,
               "capture": "ncu --set full --clock-control none -k regex:tc_gate_up -s 3 -c 1 "
                          "python bench.py --config v3slice --steps 2 --warmup 3 --no-cpu-baseline"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ environment ---

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, v: float) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.index = vis.split(",")[local_rank] if vis else str(local_rank)
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.index, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.out.flush()
        self.out.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.out.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------ algorithmic counts ---

def work(cfg):
    T, d, N_r, K_r, N_s, I = cfg.T, cfg.d, cfg.N_r, cfg.K_r, cfg.N_s, cfg.I
    rows = T * K_r + N_s * T
    q = 1 if cfg.fp8 else 2        # bytes per FFN operand element (E4M3 or bf16)
    return {
        "router_flop": 2.0 * T * d * N_r,
        "router_bytes": T * d * 2 + N_r * d * 2 + T * K_r * 8,
        "gather_bytes": T * d * q + T * K_r * d * q,
        "gate_up_flop": 2.0 * rows * d * 2 * I,
        "gate_up_bytes": (N_r + N_s) * 2 * I * d * q + rows * d * q + rows * I * q,
        "down_flop": 2.0 * rows * I * d,
        "down_bytes": (N_r + N_s) * d * I * q + rows * I * q + rows * d * 2,
        "combine_bytes": T * d * 2 + rows * d * 2 + T * d * 4 + T * K_r * 8,
        "layer_flop": 2.0 * T * d * N_r + 2.0 * rows * d * 3 * I,
    }


def kernel_src_sha() -> str:
    with open(os.path.join(ROOT, "aux_loss_free_router_b300", "csrc", "tc_gate_up.cu"), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# ------------------------------------------------------------------ oracle timing ---

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


class OracleSample:
    """The CPU oracle on single tokens of the workload (inputs drawn on the host)."""

    def __init__(self, cfg):
        import oracle
        self.oracle = oracle
        self.cfg = cfg
        x = synth.make_inputs(cfg, device="cpu", with_weights=False)
        self.u = x["u"].float().numpy()
        self.e = x["e"].float().numpy()
        self.b = x["b"].numpy()
        self.cache = {}
        self.shared = [tuple(w.float().numpy() for w in synth.expert_weights(cfg, "shared", j))
                       for j in range(cfg.N_s)]

    def expert(self, i):
        if i not in self.cache:
            self.cache[i] = tuple(w.float().numpy() for w in synth.expert_weights(self.cfg, "routed", i))
        return self.cache[i]

    def prepare(self, tokens):
        """Draw (untimed) the weights of every expert these tokens select."""
        r = self.oracle.route(self.u[tokens], self.e, self.b, self.cfg.K_r, self.cfg.G, self.cfg.M)
        for i in np.unique(r["idx"]):
            self.expert(int(i))

    def run(self, tokens) -> float:
        o, c = self.oracle, self.cfg
        t0 = time.perf_counter()
        u = self.u[tokens]
        r = o.route(u, self.e, self.b, c.K_r, c.G, c.M)
        o.layer_output(u, r["idx"], r["gate"], self.expert, self.shared)
        return time.perf_counter() - t0


def cpu_baseline(cfg, n_tokens: int, group: int = 4) -> dict:
    """Oracle time for n_tokens tokens, taken `group` tokens at a time; each group's
    expert weights are drawn (untimed) before it runs and dropped after, which bounds
    host memory."""
    s = OracleSample(cfg)
    dt = 0.0
    for g0 in range(0, n_tokens, group):
        tokens = list(range(g0, min(n_tokens, g0 + group)))
        s.cache.clear()
        s.prepare(tokens)
        dt += s.run(tokens)
    s.cache.clear()
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"{n_tokens} tokens of the {cfg.name} workload (route + all "
                      f"{cfg.K_r} routed and {cfg.N_s} shared expert FFNs + combine), "
                      f"float64 NumPy, {dt:.2f} s"}


def run_reference(args, cfg, ws, rank):
    if rank != 0:
        return
    s = OracleSample(cfg)
    tok = lambda k: [k % cfg.T]
    total = 0.0
    for k in range(args.warmup + args.steps):
        s.cache.clear()
        s.prepare(tok(k))            # untimed: draws the weights this token needs
        dt = s.run(tok(k))
        if k >= args.warmup:
            total += dt
    value = args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": "one token of the workload per step (route + expert FFNs "
                                   "+ combine), float64 NumPy on the host cores"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(cfg):
    return {"workload": f"{cfg.name}: DeepSeek-V3-shaped MoE layer forward" if cfg.name == "v3"
            else f"{cfg.name} MoE layer forward",
            "T": cfg.T, "d": cfg.d, "N_r": cfg.N_r, "K_r": cfg.K_r, "N_s": cfg.N_s, "I": cfg.I,
            "G": cfg.G, "M": cfg.M, "n_seq": cfg.n_seq, "parallelism": "replicas",
            "l2": "inputs larger than L2: every step reads all expert weights "
                  f"({(cfg.N_r + cfg.N_s) * 3 * cfg.I * cfg.d * (1 if cfg.fp8 else 2) / 1e9:.2f} GB)"}


# --------------------------------------------------------------------- our arm ---

def run_ours(args, cfg, ws, rank, local):
    import aux_loss_free_router_b300 as moe
    moe.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = synth.make_inputs(cfg, device=dev, u_seed=cfg.seed + rank)
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    layer = moe.MoELayer(T=cfg.T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I,
                         G=cfg.G, M=cfg.M, e=x["e"], b=x["b"].clone(), weights=w,
                         n_seq=cfg.n_seq, gamma=cfg.gamma, alpha=cfg.alpha, fp8=cfg.fp8)
    u, off = x["u"], x["seq_offsets"]
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        layer.step(u, off)
    torch.cuda.synchronize()
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # The timed region replays one CUDA graph holding exactly K steps (one untimed
    # replay first).  The per-stage times come from a second graph of the same K steps
    # with events recorded between the stages, replayed after the timed region: its
    # event nodes break the programmatic-launch overlap between kernels, so they stay
    # out of the timed graph.
    K = args.steps
    moe.launch_counter_reset()
    graph = layer.capture(u, off, steps=K)
    launches = moe.launch_counter()
    graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    ms = max_over_ranks(ws, t0.elapsed_time(t1) / K)
    del graph
    evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(6)]
           for _ in range(K)]
    sgraph = layer.capture(u, off, steps=K, events=evs)
    sgraph.replay()
    torch.cuda.synchronize()
    del sgraph
    stage_names = ["route", "dispatch", "gate_up", "down", "combine_bias_stat"]
    stage_ms = {n: [evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K)]
                for i, n in enumerate(stage_names)}
    stages = {n: statistics.mean(v) for n, v in stage_ms.items()}
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during the timed steps")

    # end to end through MoELayer.pipeline: every step copies its batch of tokens in
    # from pinned host memory and its layer output, loads and statistic out to pinned
    # host memory; the copies of neighbouring steps overlap the compute (three streams)
    u_host = [u.cpu().pin_memory() for _ in range(2)]
    h_host = [torch.empty(layer.out.shape, dtype=layer.out.dtype).pin_memory() for _ in range(2)]
    load_host = [torch.empty(cfg.N_r, dtype=torch.int32).pin_memory() for _ in range(2)]
    stat_host = [torch.empty(cfg.n_seq, dtype=torch.float32).pin_memory() for _ in range(2)]
    pick = lambda xs, n: [xs[k % 2] for k in range(n)]
    layer.pipeline(pick(u_host, args.warmup), pick(h_host, args.warmup), off,
                   pick(load_host, args.warmup), pick(stat_host, args.warmup))
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    layer.pipeline(pick(u_host, K), pick(h_host, K), off, pick(load_host, K), pick(stat_host, K))
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(ws, e0.elapsed_time(e1) / K)
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during the end-to-end steps")

    balance = decode = None
    if cfg.skew:
        balance = balance_run(moe, cfg, layer, off, dev, stream)
        decode = decode_pass(moe, cfg, x, dev, stream)

    bwd = None
    # the backward kernels take N_r a multiple of 64 (the v3slice workload has 32 experts)
    if cfg.dtype == "bf16" and cfg.N_r % 64 == 0 and not args.no_backward:
        del layer                      # the backward gets its own layer (it keeps s)
        torch.cuda.empty_cache()
        bwd = backward_pass(moe, cfg, x, dev, stream, steps=max(3, min(K, 10)))

    if rank != 0:
        return
    wk = work(cfg)
    pk = peaks()
    t_gu = stages["gate_up"] / 1e3
    achieved = wk["gate_up_flop"] / t_gu / 1e12
    # the timed region is K steps of a few ms (well under a second), so each GEMM
    # launch is measured against the burst rate of a dense bf16 GEMM, not the rate it
    # settles at after seconds under the power cap
    peak = pk["bf16_tflops"]
    peak_source = f"{pk['source']} bf16 burst"
    if cfg.fp8:   # E4M3 dense rate = 2x bf16 (nominal 4.5 vs 2.25 PFLOP/s)
        peak *= 2.0
        peak_source += " x 2 (nominal E4M3/bf16 ratio)"
    sha = kernel_src_sha()
    traffic = (NCU_TRAFFIC["ratio"] * wk["gate_up_bytes"]
               if NCU_TRAFFIC["kernel_src_sha"] == sha and cfg.name in ("v3", "v3slice") else None)
    tok_s = cfg.T * ws / (ms / 1e3)
    kernels = {
        "route": {"ms": stages["route"], "GB/s": wk["router_bytes"] / (stages["route"] / 1e3) / 1e9,
                  "TFLOP/s": wk["router_flop"] / (stages["route"] / 1e3) / 1e12},
        "dispatch": {"ms": stages["dispatch"],
                     "GB/s": wk["gather_bytes"] / (stages["dispatch"] / 1e3) / 1e9},
        "gate_up": {"ms": stages["gate_up"], "TFLOP/s": achieved},
        "down": {"ms": stages["down"],
                 "TFLOP/s": wk["down_flop"] / (stages["down"] / 1e3) / 1e12},
        "combine_bias_stat": {"ms": stages["combine_bias_stat"],
                              "GB/s": wk["combine_bytes"] / (stages["combine_bias_stat"] / 1e3) / 1e9},
    }
    for n, v in stage_ms.items():      # the per-stage median over the K timed steps
        kernels[n]["ms_median"] = statistics.median(v)
    wq = 1 if cfg.fp8 else 2
    layer_roof_ms = 1e3 * max(wk["layer_flop"] / (peak * 1e12),
                              ((cfg.N_r + cfg.N_s) * 3 * cfg.I * cfg.d * wq + cfg.T * cfg.d * 6)
                              / (pk["hbm_gbs"] * 1e9))
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if cfg.fp8 else ("f32" if cfg.dtype == "f32" else "bf16"),
        "data": "synthetic",
        "config": config_block(cfg),
        "roofline": {"bound": "tensor",
                     "kernel": "gate_up (grouped SwiGLU GEMM, tcgen05 "
                               + ("kind::f8f6f4, E4M3)" if cfg.fp8 else "kind::f16, bf16)"),
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_source},
        "layer_roofline_frac": layer_roof_ms / ms,
        "kernels": kernels,
        "kernels_note": "per-stage times from a second replay of the K steps with events "
                        "between the stages; ms_per_step from the timed graph without them",
        "e2e": {"value": cfg.T * ws / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": u_host[0].numel() * u_host[0].element_size(),
                "d2h_bytes_per_step": h_host[0].numel() * h_host[0].element_size()
                + load_host[0].numel() * 4 + stat_host[0].numel() * 4,
                "api": "MoELayer.pipeline (copies overlap neighbouring steps' compute)"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if bwd is not None:
        line["backward"] = bwd
    if balance is not None:
        line["balance_run"] = balance
        line["decode"] = decode
    if ws == 1 and not args.no_cpu_baseline:
        layer = None
        del x, w
        torch.cuda.empty_cache()
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_tokens)
    print(json.dumps(line), flush=True)


def backward_pass(moe, cfg, x, dev, stream, steps: int = 10) -> dict:
    """The backward pass at the forward pass's selection (moe_backward, or
    moe_backward_fp8 for the FP8 layer: gradients of sum(dh * h') and of the balance loss
    with respect to u, e and every expert weight), timed over `steps` calls replayed from
    one CUDA graph after a forward step."""
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    lay = moe.MoELayer(T=cfg.T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I, G=cfg.G,
                       M=cfg.M, e=x["e"], b=x["b"].clone(), weights=w, n_seq=cfg.n_seq,
                       gamma=cfg.gamma, alpha=cfg.alpha, want_s=True, fp8=cfg.fp8)
    u, off = x["u"], x["seq_offsets"]
    lay.step(u, off, update_bias=False)
    g = torch.Generator(device=dev).manual_seed(5)
    dh = torch.randn(cfg.T, cfg.d, generator=g, device=dev)
    for _ in range(3):
        lay.backward(u, dh, off)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            lay.backward(u, dh, off)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if moe.device_error() != 0:
        raise RuntimeError("device error word set during the backward pass")
    ms = e0.elapsed_time(e1) / steps
    R = cfg.T * cfg.K_r + cfg.N_s * cfg.T
    ffn = 12.0 * R * cfg.d * cfg.I                    # dgrad + wgrad of the three expert GEMMs
    router = 4.0 * cfg.T * cfg.d * cfg.N_r            # du = dz e and de = dz^T u
    recompute = 4.0 * R * cfg.d * cfg.I               # the gate/up GEMM run again for a, c, h
    pk = peaks()
    del graph, lay
    torch.cuda.empty_cache()
    out = {"ms": ms, "tokens_per_s": cfg.T / (ms / 1e3),
           "flop_algorithmic": ffn + router, "flop_with_recompute": ffn + router + recompute,
           "TFLOP/s_algorithmic": (ffn + router) / (ms / 1e3) / 1e12,
           "TFLOP/s_executed": (ffn + router + recompute) / (ms / 1e3) / 1e12,
           "frac_of_bf16_burst_executed": (ffn + router + recompute) / (ms / 1e3) / 1e12 / pk["bf16_tflops"],
           "note": "at the forward pass's selection; the SwiGLU pre-activations are recomputed"}
    if cfg.fp8:
        # E4M3 expert GEMMs: their peak is twice the measured bf16 burst (the nominal
        # dense ratio, 4.5 / 2.25 PFLOP/s); the router GEMMs stay bf16
        out["frac_of_e4m3_peak_executed"] = out["TFLOP/s_executed"] / (2.0 * pk["bf16_tflops"])
        out["note"] += "; expert GEMMs in E4M3 (Fprop again, Dgrad, Wgrad)"
    return out


def balance_run(moe, cfg, layer, off, dev, stream, steps: int = 200) -> dict:
    """The skewed workload's balance run: `steps` steps of forward + load count + bias
    update, each on fresh mixture tokens (seed 1000 + step); reports max/mean expert
    load per step and the layer throughput over the run."""
    us = [synth.make_inputs(cfg, device=dev, u_seed=1000 + s, with_weights=False)["u"]
          for s in range(steps)]
    loads = torch.empty(steps, cfg.N_r, dtype=torch.int32, device=dev)
    u_buf = torch.empty_like(us[0])
    u_buf.copy_(us[0])
    g = layer.capture(u_buf, off, steps=1)
    layer.b.zero_()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_ in range(steps):
        u_buf.copy_(us[s_], non_blocking=True)
        g.replay()
        loads[s_].copy_(layer.load, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    mean = cfg.T * cfg.K_r / cfg.N_r
    ratio = (loads.max(dim=1).values.float() / mean).cpu().tolist()
    return {"steps": steps, "gamma": cfg.gamma, "tokens_per_s": cfg.T / (ms / 1e3),
            "ms_per_step": ms, "max_over_mean_load": [round(r, 4) for r in ratio],
            "first10_mean": sum(ratio[:10]) / 10, "last10_mean": sum(ratio[-10:]) / 10,
            "b_absmax_end": float(layer.b.abs().max())}


def decode_pass(moe, cfg, x, dev, stream, T: int = 128, steps: int = 50) -> dict:
    """A decode-sized batch (T tokens) through the same layer weights."""
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    lay = moe.MoELayer(T=T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I, G=cfg.G,
                       M=cfg.M, e=x["e"], b=x["b"].clone(), weights=w, n_seq=1,
                       gamma=cfg.gamma, alpha=cfg.alpha)
    u = synth.make_inputs(cfg.replace(T=T, n_seq=1), device=dev, u_seed=7, with_weights=False)["u"]
    off = synth.make_seq_offsets(T, 1).to(dev)
    for _ in range(3):
        lay.step(u, off)
    g = lay.capture(u, off, steps=steps)      # timed: no event nodes between the stages
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del g
    evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(6)]
           for _ in range(steps)]
    g = lay.capture(u, off, steps=steps, events=evs)   # per-stage times
    g.replay()
    torch.cuda.synchronize()
    stage_names = ["route", "dispatch", "gate_up", "down", "combine_bias_stat"]
    stages = {n: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(steps))
              for i, n in enumerate(stage_names)}
    wbytes = (cfg.N_r + cfg.N_s) * 3 * cfg.I * cfg.d * 2
    return {"T": T, "ms_per_step": ms, "tokens_per_s": T / (ms / 1e3),
            "weight_GB_per_s_if_all_read": wbytes / (ms / 1e3) / 1e9,
            "stages_ms": stages}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="v3", choices=sorted(synth.CONFIGS))
    ap.add_argument("--cpu-tokens", type=int, default=24)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward-pass measurement (reported beside the forward)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    cfg = synth.config(args.config)
    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        run_reference(args, cfg, ws, int(os.environ.get("RANK", "0")))
        return
    ws, rank, local = dist_setup()
    run_ours(args, cfg, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
