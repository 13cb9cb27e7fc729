"""Seeded synthetic inputs for the DeepSeekMoE layer with auxiliary-loss-free routing.

This module is shared by the CPU oracle's tests, the GPU parity tests, ``bench.py``
and ``__graft_entry__.smoke()``.  It only draws random numbers and lays them out in
the shapes the layer takes; it holds none of the layer's arithmetic (no affinity, no
selection, no gating, no FFN, no quantisation).

Shapes follow the notation of the DeepSeek-V3 reports: ``u`` [T, d] token inputs
u_t, ``e`` [N_r, d] expert centroids e_i, ``b`` [N_r] routing biases b_i, routed
SwiGLU weights ``w_gate``/``w_up`` [N_r, I, d] and ``w_down`` [N_r, d, I], shared
expert weights ``ws_*`` with N_s in place of N_r.  Every weight matrix is stored
K-major (the contraction dimension is contiguous).

Distributions: u_t ~ N(0, 1); e_i ~ N(0, 1/d); W ~ N(0, 1/fan_in) with fan_in = d
for gate/up and I for down; b_i ~ U[-0.01, 0.01] or 0.  The skewed workload draws
u_t from a 4-component Gaussian mixture whose component means are 3*sqrt(d) along
random orthonormal directions, so that each component shifts every expert logit
u_t.e_i by about N(0, 9) and a few experts dominate (see ``mixture_tokens``).

Every tensor has its own seeded random stream (``stream_seed``): u, e and b each,
and each expert's weights (gate, up, down drawn in that order), so one expert can be
drawn on its own.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["MoEConfig", "CONFIGS", "config", "make_inputs", "mixture_tokens",
           "make_seq_offsets", "expert_weights", "stream_seed"]


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens in the batch
    d: int            # hidden size
    N_r: int          # routed experts
    K_r: int          # routed experts active per token
    N_s: int          # shared experts
    I: int            # SwiGLU intermediate size
    G: int = 1        # expert groups (1 = no group limit)
    M: int = 1        # groups kept per token
    n_seq: int = 1    # sequences in the batch (equal lengths)
    dtype: str = "bf16"      # storage dtype of u, e and the weights: "f32" | "bf16"
    fp8: bool = False        # expert GEMMs in E4M3 with fp32 block scales
    bias: str = "uniform"    # "uniform" -> U[-0.01, 0.01]; "zero" -> 0
    gamma: float = 0.001     # bias update speed
    alpha: float = 0.0001    # sequence-wise balance factor
    seed: int = 0
    skew: bool = False       # tokens from the Gaussian mixture

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


# The five workloads: tiny fp32, mid bf16, DeepSeek-V3-shaped bf16 with group-limited
# routing, the skewed balance run (mid shapes, T=2048) and the FP8 variant of mid.
CONFIGS = {
    "tiny": MoEConfig("tiny", T=64, d=256, N_r=16, K_r=2, N_s=1, I=128,
                      dtype="f32", bias="uniform"),
    "mid": MoEConfig("mid", T=4096, d=2048, N_r=64, K_r=6, N_s=2, I=1408,
                     n_seq=4, dtype="bf16", bias="zero"),
    "v3": MoEConfig("v3", T=8192, d=7168, N_r=256, K_r=8, N_s=1, I=2048, G=8, M=4,
                    n_seq=2, dtype="bf16", bias="uniform"),
    "skew": MoEConfig("skew", T=2048, d=2048, N_r=64, K_r=6, N_s=2, I=1408,
                      n_seq=2, dtype="bf16", bias="zero", skew=True),
    "fp8": MoEConfig("fp8", T=4096, d=2048, N_r=64, K_r=6, N_s=2, I=1408,
                     n_seq=4, dtype="bf16", bias="zero", fp8=True),
    # a slice of the V3-shaped layer for hardware-counter captures: the same d, I, K_r
    # and mean expert load (256 tokens) with 32 experts in 8 groups, ~3 GB on the device
    "v3slice": MoEConfig("v3slice", T=1024, d=7168, N_r=32, K_r=8, N_s=1, I=2048, G=8, M=4,
                         n_seq=1, dtype="bf16", bias="uniform"),
}


def config(name: str, **overrides) -> MoEConfig:
    cfg = CONFIGS[name]
    return cfg.replace(**overrides) if overrides else cfg


def make_seq_offsets(T: int, n_seq: int) -> torch.Tensor:
    """Equal-length sequence boundaries [n_seq+1] (int32), the last one equal to T."""
    if n_seq < 1 or T % n_seq:
        raise ValueError("T must split into n_seq equal sequences")
    return torch.arange(0, T + 1, T // n_seq, dtype=torch.int32)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


_TAGS = {"u": 1, "e": 2, "b": 3, "shared": 4, "routed": 5}


def stream_seed(seed: int, tag: str, index: int = 0) -> int:
    """Seed of one named random stream: every tensor (and every expert's weights) has
    its own stream, so any single expert can be drawn without drawing the others."""
    return (seed * 1_000_003 + _TAGS[tag] * 7_919 + index * 104_729) % (2 ** 62)


def _normal(shape, std, g, device, dtype):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def mixture_tokens(T: int, d: int, seed: int, device="cpu", scale: float = 3.0,
                   n_comp: int = 4, dir_seed: int = 0) -> torch.Tensor:
    """Tokens from an n_comp-component Gaussian mixture (fp32, [T, d]).

    Component c has mean scale*sqrt(d)*q_c, with q_1..q_n orthonormal random
    directions drawn once from ``dir_seed``; each token picks its component
    uniformly (from ``seed``) and adds N(0, I) noise.
    """
    gd = _gen(dir_seed + 7919, "cpu")
    q, _ = torch.linalg.qr(torch.randn(d, n_comp, generator=gd, dtype=torch.float64))
    means = (scale * math.sqrt(d) * q.T).to(torch.float32).to(device)   # [n_comp, d]
    g = _gen(seed, device)
    comp = torch.randint(0, n_comp, (T,), generator=g, device=device)
    noise = torch.randn(T, d, generator=g, device=device, dtype=torch.float32)
    return noise + means[comp]


def expert_weights(cfg: MoEConfig, kind: str, i: int, device="cpu", seed=None):
    """(gate [I, d], up [I, d], down [d, I]) of routed (kind="routed") or shared
    (kind="shared") expert i, drawn from that expert's own stream."""
    seed = cfg.seed if seed is None else seed
    g = _gen(stream_seed(seed, kind, i), device)
    dt = cfg.torch_dtype
    sg, sd = 1.0 / math.sqrt(cfg.d), 1.0 / math.sqrt(cfg.I)
    return (_normal((cfg.I, cfg.d), sg, g, device, dt), _normal((cfg.I, cfg.d), sg, g, device, dt),
            _normal((cfg.d, cfg.I), sd, g, device, dt))


def make_inputs(cfg: MoEConfig, device="cpu", seed: Optional[int] = None,
                u_seed: Optional[int] = None, with_weights: bool = True) -> dict:
    """All layer inputs for ``cfg`` as torch tensors on ``device``.

    Storage dtype is ``cfg.torch_dtype`` (bf16 values are rounded once from the fp32
    draws).  ``b`` is always fp32.  ``u_seed`` redraws only the tokens (used by the
    skewed multi-step run, where step s uses seed 1000+s for u).  The values depend
    on the device's generator (CPU and CUDA streams differ), never on anything else.
    """
    seed = cfg.seed if seed is None else seed
    dt = cfg.torch_dtype
    T, d, N_r, N_s, I = cfg.T, cfg.d, cfg.N_r, cfg.N_s, cfg.I
    out = {}
    us = u_seed if u_seed is not None else seed
    if cfg.skew:
        out["u"] = mixture_tokens(T, d, seed=us, device=device).to(dt)
    else:
        out["u"] = _normal((T, d), 1.0, _gen(stream_seed(us, "u"), device), device, dt)
    out["e"] = _normal((N_r, d), 1.0 / math.sqrt(d), _gen(stream_seed(seed, "e"), device),
                       device, dt)
    if cfg.bias == "uniform":
        gb = _gen(stream_seed(seed, "b"), device)
        out["b"] = torch.rand(N_r, generator=gb, device=device, dtype=torch.float32) * 0.02 - 0.01
    else:
        out["b"] = torch.zeros(N_r, device=device, dtype=torch.float32)
    if with_weights:
        for prefix, kind, E in (("ws_", "shared", N_s), ("w_", "routed", N_r)):
            wg = torch.empty(E, I, d, dtype=dt, device=device)
            wu = torch.empty(E, I, d, dtype=dt, device=device)
            wd = torch.empty(E, d, I, dtype=dt, device=device)
            for i in range(E):
                wg[i], wu[i], wd[i] = expert_weights(cfg, kind, i, device, seed)
            out[prefix + "gate"], out[prefix + "up"], out[prefix + "down"] = wg, wu, wd
    out["seq_offsets"] = make_seq_offsets(T, cfg.n_seq).to(device)
    return out
