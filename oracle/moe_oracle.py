"""Plain CPU oracle of the DeepSeekMoE layer forward with auxiliary-loss-free routing.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``; never by the CUDA
library or its Python binding, and it imports nothing from them.  It is slow on
purpose: float64 NumPy, explicit per-token selection loops, no blocking or fusion.

Sources (untrusted web pages about the DeepSeek-V3 technical report; cited by site,
title and section):

* [P1] szhzxw.cn, DeepSeek-V3 解读 — sections "无辅助损失负载平衡的DeepSeekMoE",
  "互补序列级辅助损失", "节点限制路由", "无Token丢弃".
* [P3] pwwt.cn, "DeepSeek-V3 Technical Report" 笔记 — §一 (sigmoid + normalisation),
  §1.1.2 (three-step routing), §1.1.3 (bias update), §1.2 (sequence-wise loss),
  §1.3 (node-limited routing), §1.4 (no token dropping).
* [P4/P5] xyznot.com, "DeepSeek-V3 Technical Report" reading guide (ar / pt) —
  Method §2: the equations for h'_t, s_{i,t} and g'_{i,t}, and gamma = 0.001,
  alpha = 0.0001.

Readings taken where the pages are silent or garbled:

* gates are g = g' / sum_j g'_j over the selected experts ([P3] §一 "normalise all
  selected affinity scores"; [P4] Method §2 "normalising g'");
* the routing key is fp32(s + b) with one fp32 rounding; ties go to the lower
  expert index, and the selected list is ordered by descending key;
* a group's score is the fp32 sum, in descending key order, of its K_r/M largest
  keys ([P3] §1.3 "top K_r/M"); groups are contiguous blocks of N_r/G experts and
  are ranked on the biased keys; ties go to the lower group index;
* overloaded / underloaded means above / below the mean load T*K_r/N_r, compared in
  exact integers; equal load leaves b_i unchanged;
* the sequence statistic is alpha * sum_i f_i * P_i with
  f_i = N_r/(K_r*T_S) * #{t in S : i actually selected for t} and
  P_i = (1/T_S) * sum_{t in S} s_{i,t} / sum_j s_{j,t}; the pages give the product
  form and the word meanings of f_i and P_i ([P3] §1.2) but not the normalisation,
  so the normalisation of f_i and P_i is **parity unpinned** beyond the invariants
  sum_i f_i = N_r and sum_i P_i = 1 and the uniform closed form (stat = alpha);
* the expert FFN is SwiGLU without biases:
  FFN(x) = W_down (silu(W_gate x) * (W_up x)), silu(z) = z / (1 + exp(-z)).
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence

import numpy as np

from . import fp8 as _fp8

__all__ = [
    "affinity", "routing_keys", "group_scores", "select_experts", "gate_values",
    "route", "dispatch", "silu", "expert_ffn", "layer_output", "bias_update",
    "seq_p_sums", "seq_balance_stat", "moe_forward",
]


# ---------------------------------------------------------------- routing ---------

def affinity(u, e) -> np.ndarray:
    """s_{i,t} = Sigmoid(u_t^T e_i)  ([P4/P5] Method §2, equation for s_{i,t}).

    u [T, d] and e [N_r, d] hold the exact stored values (bf16 or fp32, upcast).  The
    product is formed in float64 and the sigmoid rounded once to fp32, the precision
    in which the routing decision is taken.
    """
    z = np.asarray(u, np.float64) @ np.asarray(e, np.float64).T
    return (1.0 / (1.0 + np.exp(-z))).astype(np.float32)


def routing_keys(s, b) -> np.ndarray:
    """k_{i,t} = s_{i,t} + b_i, the key Top-K ranks ([P4/P5] Method §2, g' equation;
    [P1] "偏置项仅用于路由").  One fp32 addition."""
    s = np.asarray(s, np.float32)
    b = np.asarray(b, np.float32)
    return (s + b[None, :]).astype(np.float32)


def _order_desc(values: Sequence, candidates: Sequence[int]) -> list[int]:
    """Candidates sorted by descending value, ties to the lower index."""
    return sorted(candidates, key=lambda i: (-float(values[i]), i))


def group_scores(keys_row, G: int, M: int, K_r: int) -> list[np.float32]:
    """Score of each of the G contiguous expert groups for one token.

    A group's score is the sum of its K_r/M largest keys ([P3] §1.3: nodes are chosen
    by the sum of the top K_r/M affinity scores of the experts on each node; [P1]
    "节点限制路由").  The sum is fp32, taken in descending key order.
    """
    N_r = len(keys_row)
    per, kg = N_r // G, K_r // M
    out = []
    for g in range(G):
        members = list(range(g * per, (g + 1) * per))
        acc = np.float32(0.0)
        for i in _order_desc(keys_row, members)[:kg]:
            acc = np.float32(acc + np.float32(keys_row[i]))
        out.append(acc)
    return out


def select_experts(s, b, K_r: int, G: int = 1, M: int = 1) -> np.ndarray:
    """Indices of the experts whose s+b is in TopK({s_j+b_j}, K_r), per token.

    ([P4/P5] Method §2, g' equation.)  With G > 1 only the M groups with the largest
    group scores are eligible (the node-limited routing of [P1]/[P3] §1.3, with nodes
    as contiguous expert groups).  Returns int32 [T, K_r], each row in descending key
    order with ties to the lower index.
    """
    keys = routing_keys(s, b)
    T, N_r = keys.shape
    idx = np.empty((T, K_r), dtype=np.int32)
    for t in range(T):
        row = keys[t]
        eligible = list(range(N_r))
        if G > 1:
            gs = group_scores(row, G, M, K_r)
            kept = set(_order_desc(gs, range(G))[:M])
            per = N_r // G
            eligible = [i for i in range(N_r) if i // per in kept]
        idx[t] = _order_desc(row, eligible)[:K_r]
    return idx


def gate_values(s, idx) -> np.ndarray:
    """g_{i,t} = g'_{i,t} / sum_j g'_{j,t} with g' the RAW s of the selected experts.

    ([P4/P5] Method §2: g computed by normalising g'; [P3] §一 and §1.1.2 step 3: the
    gate uses the original affinity, the bias only decides who is selected.)
    float64 arithmetic, rounded to fp32.
    """
    s = np.asarray(s, np.float64)
    sel = np.take_along_axis(s, np.asarray(idx, np.int64), axis=1)
    return (sel / sel.sum(axis=1, keepdims=True)).astype(np.float32)


def route(u, e, b, K_r: int, G: int = 1, M: int = 1, s=None) -> dict:
    """Affinities, selection and gates for a batch.  ``s`` overrides the affinities
    (used to take the routing decision on another implementation's fp32 scores)."""
    s = affinity(u, e) if s is None else np.asarray(s, np.float32)
    idx = select_experts(s, b, K_r, G, M)
    return {"s": s, "idx": idx, "gate": gate_values(s, idx)}


# --------------------------------------------------------------- dispatch ---------

def dispatch(idx, N_r: int) -> dict:
    """Per-expert token lists without dropping any token ([P3] §1.4, [P1] "无Token丢弃").

    load_i = #{(t, k) : idx[t, k] = i} over the whole batch ([P1]: the load of the
    entire batch is monitored each step; [P3] §1.1.3).  offset is the exclusive
    prefix sum of load; perm_token lists, expert by expert, the tokens routed there
    in ascending t; inv_row[t, k] is the position of (t, idx[t, k]) in that list.
    """
    idx = np.asarray(idx, np.int64)
    T, K_r = idx.shape
    load = np.zeros(N_r, dtype=np.int64)
    for i in idx.reshape(-1):
        load[i] += 1
    offset = np.zeros(N_r + 1, dtype=np.int64)
    offset[1:] = np.cumsum(load)
    perm_token = np.empty(T * K_r, dtype=np.int64)
    inv_row = np.empty((T, K_r), dtype=np.int64)
    fill = offset[:-1].copy()
    for t in range(T):                       # ascending t within every expert
        for k in range(K_r):
            i = idx[t, k]
            perm_token[fill[i]] = t
            inv_row[t, k] = fill[i]
            fill[i] += 1
    return {"load": load.astype(np.int32), "offset": offset.astype(np.int32),
            "perm_token": perm_token.astype(np.int32), "inv_row": inv_row.astype(np.int32)}


# ------------------------------------------------------------------- FFN ----------

def silu(z):
    z = np.asarray(z, np.float64)
    return z / (1.0 + np.exp(-z))


def expert_ffn(x, w_gate, w_up, w_down, h_quant: bool = False) -> np.ndarray:
    """FFN(x) = W_down (silu(W_gate x) * (W_up x)) for rows x [n, d]; float64.

    The pages name only "FFN" for the experts ([P4/P5] Method §2, h' equation); the
    SwiGLU form without biases is the reading taken.  Weights are K-major:
    w_gate, w_up [I, d], w_down [d, I].  With ``h_quant`` the intermediate is passed
    through the 1x128 E4M3 quantiser first, as the FP8 variant does.
    """
    x = np.asarray(x, np.float64)
    a = x @ np.asarray(w_gate, np.float64).T
    c = x @ np.asarray(w_up, np.float64).T
    h = silu(a) * c
    if h_quant:
        q, sc = _fp8.quantize_1x128(h.astype(np.float32))
        h = _fp8.dequantize_1x128(q, sc)
    return h @ np.asarray(w_down, np.float64).T


ExpertFn = Callable[[int], tuple]


def layer_output(u, idx, gate, routed: ExpertFn, shared: Sequence[tuple],
                 x=None, h_quant: bool = False) -> np.ndarray:
    """h'_t = u_t + sum_s FFN^(s)_s(u_t) + sum_k g_{k,t} FFN^(r)_{idx_k}(u_t).

    ([P4/P5] Method §2, equation for h'_t.)  ``routed(i)`` returns expert i's
    (w_gate, w_up, w_down); ``shared`` lists the shared experts' triples.  ``x`` is
    the FFN input when it differs from the residual u (the FP8 variant feeds the
    dequantised tokens).  float64; every token is processed (no dropping).
    """
    u = np.asarray(u, np.float64)
    x = u if x is None else np.asarray(x, np.float64)
    idx = np.asarray(idx, np.int64)
    gate = np.asarray(gate, np.float64)
    h = u.copy()
    for (wg, wu, wd) in shared:
        h += expert_ffn(x, wg, wu, wd, h_quant)
    for i in np.unique(idx):
        rows, ks = np.nonzero(idx == i)
        wg, wu, wd = routed(int(i))
        h[rows] += gate[rows, ks][:, None] * expert_ffn(x[rows], wg, wu, wd, h_quant)
    return h


# ------------------------------------------------------- end-of-step state ---------

def bias_update(b, load, T: int, K_r: int, gamma: float) -> np.ndarray:
    """b_i <- b_i - gamma if expert i is overloaded, + gamma if underloaded.

    ([P3] §1.1.3; [P1] "在每个步骤的末尾"; gamma = 0.001 in [P4/P5] Method §2.)
    Overloaded means load_i above the batch mean T*K_r/N_r, decided in exact
    integers as sign(T*K_r - N_r*load_i); the update is one fp32 addition.
    """
    load = np.asarray(load, np.int64)
    N_r = load.shape[0]
    sign = np.sign(T * K_r - N_r * load).astype(np.float32)
    return (np.asarray(b, np.float32) + np.float32(gamma) * sign).astype(np.float32)


def seq_p_sums(s, seq_offsets) -> np.ndarray:
    """sum_{t in S} s_{i,t} / sum_j s_{j,t} for each sequence S (float64 [n_seq, N_r])."""
    s = np.asarray(s, np.float64)
    sp = s / s.sum(axis=1, keepdims=True)
    off = np.asarray(seq_offsets, np.int64)
    return np.stack([sp[off[j]:off[j + 1]].sum(axis=0) for j in range(len(off) - 1)])


def seq_balance_stat(s, idx, seq_offsets, N_r: int, K_r: int, alpha: float):
    """Complementary sequence-wise balance statistic alpha * sum_i f_i * P_i.

    ([P3] §1.2: f_i is how often expert i is actually selected within the sequence,
    P_i the probability mass the gate assigns to it; alpha = 0.0001 in [P4/P5]
    Method §2.)  Normalisation as in the module docstring.  Returns
    (per-sequence values [n_seq] float64, their mean).
    """
    idx = np.asarray(idx, np.int64)
    off = np.asarray(seq_offsets, np.int64)
    psum = seq_p_sums(s, off)
    stats = []
    for j in range(len(off) - 1):
        a, z = off[j], off[j + 1]
        T_S = z - a
        counts = np.zeros(N_r, dtype=np.float64)
        for t in range(a, z):
            for i in idx[t]:
                counts[i] += 1.0
        f = counts * (N_r / (K_r * T_S))
        P = psum[j] / T_S
        stats.append(alpha * float(np.dot(f, P)))
    stats = np.asarray(stats, dtype=np.float64)
    return stats, float(stats.mean())


# ------------------------------------------------------------- whole layer ---------

def moe_forward(u, e, b, weights: dict, K_r: int, G: int = 1, M: int = 1, N_s: int = 0,
                s=None, fp8: bool = False, seq_offsets=None, gamma: float = 0.001,
                alpha: float = 0.0001) -> dict:
    """One forward pass of the layer plus the end-of-step quantities.

    ``weights`` holds numpy arrays "w_gate", "w_up" [N_r, I, d], "w_down" [N_r, d, I]
    and the shared "ws_*" arrays.  With ``fp8`` the FFN runs on the E4M3-dequantised
    tokens (1x128 tiles) and weights (128x128 blocks) and the SwiGLU output is
    quantised 1x128 before the down projection; routing stays on the unquantised u.
    """
    u = np.asarray(u, np.float32)
    T = u.shape[0]
    N_r = np.asarray(e).shape[0]
    r = route(u, e, b, K_r, G, M, s=s)
    dp = dispatch(r["idx"], N_r)

    def prep(w):
        w = np.asarray(w, np.float32)
        if not fp8:
            return w
        q, sc = _fp8.quantize_128x128(w)
        return _fp8.dequantize_128x128(q, sc)

    x = None
    if fp8:
        q, sc = _fp8.quantize_1x128(u)
        x = _fp8.dequantize_1x128(q, sc)

    def routed(i):
        return (prep(weights["w_gate"][i]), prep(weights["w_up"][i]),
                prep(weights["w_down"][i]))

    shared = [(prep(weights["ws_gate"][j]), prep(weights["ws_up"][j]),
               prep(weights["ws_down"][j])) for j in range(N_s)]
    h = layer_output(u, r["idx"], r["gate"], routed, shared, x=x, h_quant=fp8)
    out = dict(r, **dp, h=h, b_new=bias_update(b, dp["load"], T, K_r, gamma))
    if seq_offsets is not None:
        out["seq_stat"], out["seq_stat_mean"] = seq_balance_stat(
            r["s"], r["idx"], seq_offsets, N_r, K_r, alpha)
    return out
