"""Plain CPU oracle of the DeepSeekMoE layer's backward pass (gradients through the
layer with auxiliary-loss-free routing).

TEST INFRASTRUCTURE ONLY, like ``moe_oracle``: imported by ``tests/`` and by nothing
in the CUDA library or its binding.  float64 NumPy, per-expert loops, no fusion.

Sources: the same pages as ``moe_oracle`` — [P4/P5] Method §2 (h'_t, s_{i,t},
g'_{i,t}), [P3] §1.1.2–§1.1.3 (the bias only decides the selection and is moved by
the sign rule after each step) and §1.2 (the sequence-wise balance loss).

What is differentiated (readings taken where the pages are silent):

* the selection (Top-K_r of fp32(s + b) under the group limit) is piecewise
  constant in the inputs and passes no gradient; the bias b enters only the
  selection, so it receives none — it is moved by the sign rule instead ([P3] §1.1.3);
* the gates g = s_sel / sum(s_sel) are differentiated through the RAW affinities of
  the selected experts, whose normalisation couples them;
* s = sigmoid(z), z = u e^T: ds/dz = s (1 - s);
* the balance loss of a sequence S is alpha * sum_i f_i P_i with f_i the selection
  count scaled by N_r/(K_r T_S) (a count: no gradient) and P_i the mean over S of s
  normalised over all N_r experts; the objective adds the mean of the per-sequence
  losses, the quantity the forward reports;
* the experts are SwiGLU without biases, silu'(a) = sigma(a) (1 + a (1 - sigma(a))).

``forward64`` is the forward restated in float64 with the selection passed in (or
taken from ``moe_oracle.route``), so that finite differences of it, at a frozen
selection, measure exactly the function whose gradient ``layer_backward`` returns.
"""
from __future__ import annotations

import numpy as np

from . import moe_oracle as _fw

from . import fp8 as _fp8

__all__ = [
    "sigmoid64", "silu_grad", "expert_ffn_backward", "gate_backward", "balance_backward",
    "forward64", "layer_backward", "expert_ffn_backward_fp8", "layer_backward_fp8",
]


def sigmoid64(z) -> np.ndarray:
    z = np.asarray(z, np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def silu_grad(a) -> np.ndarray:
    """d/da [a * sigma(a)] = sigma(a) * (1 + a * (1 - sigma(a)))."""
    a = np.asarray(a, np.float64)
    sg = sigmoid64(a)
    return sg * (1.0 + a * (1.0 - sg))


def expert_ffn_backward(x, w_gate, w_up, w_down, dy):
    """Gradients of sum(dy * FFN(x)) for FFN(x) = W_down (silu(W_gate x) * (W_up x)).

    x [n, d], w_gate/w_up [I, d], w_down [d, I], dy [n, d].  Returns
    (dx [n, d], dw_gate [I, d], dw_up [I, d], dw_down [d, I]), float64.
    """
    x = np.asarray(x, np.float64)
    wg, wu, wd = (np.asarray(w, np.float64) for w in (w_gate, w_up, w_down))
    dy = np.asarray(dy, np.float64)
    a = x @ wg.T                    # gate pre-activation [n, I]
    c = x @ wu.T                    # up projection [n, I]
    h = _fw.silu(a) * c
    dh = dy @ wd                    # [n, I]
    dw_down = dy.T @ h              # [d, I]
    dc = dh * _fw.silu(a)
    da = dh * c * silu_grad(a)
    dx = da @ wg + dc @ wu
    return dx, da.T @ x, dc.T @ x, dw_down


def gate_backward(s, idx, dgate) -> np.ndarray:
    """ds [T, N_r] from dL/dg for g_k = s_{idx_k} / sum_j s_{idx_j} (raw s).

    dg_k/ds_{idx_j} = (delta_kj - g_k) / S, S = sum_j s_{idx_j}; so
    ds_{idx_j} = (dg_j - sum_k g_k dg_k) / S.  Unselected experts get zero.
    """
    s = np.asarray(s, np.float64)
    idx = np.asarray(idx, np.int64)
    dgate = np.asarray(dgate, np.float64)
    ds = np.zeros_like(s)
    for t in range(s.shape[0]):
        sel = s[t, idx[t]]
        S = sel.sum()
        g = sel / S
        inner = float(np.dot(g, dgate[t]))
        for j, i in enumerate(idx[t]):
            ds[t, i] += (dgate[t, j] - inner) / S
    return ds


def balance_backward(s, idx, seq_offsets, K_r: int, alpha: float) -> np.ndarray:
    """ds [T, N_r] of the mean over sequences of alpha * sum_i f_i P_i.

    P_i = (1/T_S) sum_{t in S} s_{i,t} / R_t with R_t = sum_j s_{j,t}, so
    dP_i/ds_{j,t} = (delta_ij - s_{i,t}/R_t) / (T_S R_t), and
    ds_{j,t} = alpha/n_seq * (f_j - sum_i f_i s_{i,t}/R_t) / (T_S R_t).
    """
    s = np.asarray(s, np.float64)
    idx = np.asarray(idx, np.int64)
    off = np.asarray(seq_offsets, np.int64)
    T, N_r = s.shape
    n_seq = len(off) - 1
    ds = np.zeros_like(s)
    for j in range(n_seq):
        a, z = off[j], off[j + 1]
        T_S = z - a
        if T_S == 0:
            continue
        counts = np.zeros(N_r)
        for t in range(a, z):
            for i in idx[t]:
                counts[i] += 1.0
        f = counts * (N_r / (K_r * T_S))
        for t in range(a, z):
            R = s[t].sum()
            sp = s[t] / R
            ds[t] += (alpha / n_seq) * (f - float(np.dot(f, sp))) / (T_S * R)
    return ds


def _weights64(weights: dict, N_s: int):
    routed = {k: np.asarray(weights[k], np.float64) for k in ("w_gate", "w_up", "w_down")}
    shared = [tuple(np.asarray(weights[k][j], np.float64) for k in ("ws_gate", "ws_up", "ws_down"))
              for j in range(N_s)]
    return routed, shared


def forward64(u, e, b, weights: dict, K_r: int, G: int = 1, M: int = 1, N_s: int = 0,
              seq_offsets=None, alpha: float = 0.0, idx=None) -> dict:
    """The layer forward in float64 (no fp32 rounding of s or of the gates).

    ``idx`` fixes the selection; by default it is the forward oracle's decision on
    fp32 keys.  Returns h' [T, d], s, idx, the gates, the per-expert outputs y[t, k]
    and (with ``seq_offsets``) the mean balance loss.
    """
    u = np.asarray(u, np.float64)
    e = np.asarray(e, np.float64)
    if idx is None:
        idx = _fw.route(u.astype(np.float32), e.astype(np.float32), b, K_r, G, M)["idx"]
    idx = np.asarray(idx, np.int64)
    s = sigmoid64(u @ e.T)
    sel = np.take_along_axis(s, idx, axis=1)
    gate = sel / sel.sum(axis=1, keepdims=True)
    routed, shared = _weights64(weights, N_s)
    h = u.copy()
    for (wg, wu, wd) in shared:
        h += _fw.expert_ffn(u, wg, wu, wd)
    y = np.zeros(idx.shape + (u.shape[1],))
    for i in np.unique(idx):
        rows, ks = np.nonzero(idx == i)
        y[rows, ks] = _fw.expert_ffn(u[rows], routed["w_gate"][i], routed["w_up"][i],
                                     routed["w_down"][i])
    h += np.einsum("tk,tkd->td", gate, y)
    out = {"h": h, "s": s, "idx": idx, "gate": gate, "y": y}
    if seq_offsets is not None:
        off = np.asarray(seq_offsets, np.int64)
        N_r = e.shape[0]
        losses = []
        for j in range(len(off) - 1):
            a, z = off[j], off[j + 1]
            T_S = z - a
            counts = np.zeros(N_r)
            for t in range(a, z):
                for i in idx[t]:
                    counts[i] += 1.0
            f = counts * (N_r / (K_r * T_S))
            P = (s[a:z] / s[a:z].sum(axis=1, keepdims=True)).sum(axis=0) / T_S
            losses.append(alpha * float(np.dot(f, P)))
        out["bal_mean"] = float(np.mean(losses))
    return out


def layer_backward(u, e, b, weights: dict, dh, K_r: int, G: int = 1, M: int = 1,
                   N_s: int = 0, seq_offsets=None, alpha: float = 0.0, idx=None) -> dict:
    """Gradients of J = sum(dh * h') (+ the mean balance loss when ``seq_offsets`` is
    given) with respect to u, e, b and every expert weight, at the selection of
    ``forward64``.  float64.  Keys: du, de, db (all zero), w_gate, w_up, w_down,
    ws_gate, ws_up, ws_down (arrays shaped like the weights)."""
    fw = forward64(u, e, b, weights, K_r, G, M, N_s, seq_offsets, alpha, idx)
    u = np.asarray(u, np.float64)
    e = np.asarray(e, np.float64)
    dh = np.asarray(dh, np.float64)
    s, idx, gate, y = fw["s"], fw["idx"], fw["gate"], fw["y"]
    routed, shared = _weights64(weights, N_s)
    du = dh.copy()                                    # residual
    grads = {k: np.zeros_like(v) for k, v in routed.items()}
    for k in ("ws_gate", "ws_up", "ws_down"):
        grads[k] = np.zeros((N_s,) + np.asarray(weights[k]).shape[1:])
    for j, (wg, wu, wd) in enumerate(shared):
        dx, dg_, du_, dd_ = expert_ffn_backward(u, wg, wu, wd, dh)
        du += dx
        grads["ws_gate"][j], grads["ws_up"][j], grads["ws_down"][j] = dg_, du_, dd_
    for i in np.unique(idx):
        rows, ks = np.nonzero(idx == i)
        dy = gate[rows, ks][:, None] * dh[rows]
        dx, dg_, du_, dd_ = expert_ffn_backward(u[rows], routed["w_gate"][i], routed["w_up"][i],
                                                routed["w_down"][i], dy)
        np.add.at(du, rows, dx)
        grads["w_gate"][i] += dg_
        grads["w_up"][i] += du_
        grads["w_down"][i] += dd_
    dgate = np.einsum("td,tkd->tk", dh, y)
    ds = gate_backward(s, idx, dgate)
    if seq_offsets is not None:
        ds += balance_backward(s, idx, seq_offsets, K_r, alpha)
    dz = ds * s * (1.0 - s)
    du += dz @ e
    de = dz.T @ u
    return dict(grads, du=du, de=de, db=np.zeros(np.asarray(b).shape))


# ----------------------------------------------------------------- FP8 backward -----
#
# The pages run all three GEMMs of a linear layer in E4M3 - Fprop, Dgrad (activation
# gradient) and Wgrad (weight gradient) - with fp32 outputs, fp32 scales per 1x128
# activation tile and per 128x128 weight block, promotion to fp32 every 128 elements
# of the contraction, and the activations that Wgrad needs kept in E4M3 from the
# forward pass (pwwt.cn notes §三; xyznot.com reading guide, Key ideas, FP8 bullet).
# Readings where the pages are silent:
#
# * an activation tile lies along the contraction axis of the GEMM that consumes it:
#   1x128 (one token, 128 features) in Fprop and Dgrad, 128x1 (one feature, 128 tokens
#   of an expert's segment, the last tile short) in Wgrad, whose contraction runs over
#   the tokens; the weights keep their 128x128 blocks (a block is a block of W^T too);
# * Wgrad takes the cached forward activations - the E4M3 tokens x and the E4M3 h the
#   forward's down GEMM consumed - and re-tiles them 128x1 (dequantise, quantise);
# * the gradients dY = g * dh, dA and dC are quantised for Dgrad (1x128) and for Wgrad
#   (128x1) each from its own value;
# * the router stays as in the FP8 forward: affinities, gates and the balance loss on
#   the unquantised bf16 tokens, their gradients in float64.
#
# Where a value is rounded before it is quantised, the oracle rounds it where the
# kernels do (bf16 a and c, dY, dH, and the dA / dC that Wgrad quantises), so that both
# sides decide every E4M3 code on the same number.  The products are float64 sums of
# dequantised operands: promotion every 128 with fp32 scales is this sum up to fp32
# rounding of the partial sums.

def _cached_activation(m) -> np.ndarray:
    """A forward activation as the FP8 layer keeps it: E4M3 per 1x128 tile."""
    return _fp8.dequantize_1x128(*_fp8.quantize_1x128(np.asarray(m, np.float32)))


def _dgrad_operand(m) -> np.ndarray:
    """An activation gradient entering a Dgrad GEMM: E4M3 per 1x128 tile (the
    contraction runs over the features)."""
    return _fp8.dequantize_1x128(*_fp8.quantize_1x128(np.asarray(m, np.float32)))


def _wgrad_operand(m) -> np.ndarray:
    """An operand of a Wgrad GEMM over one expert's tokens: E4M3 per 128x1 tile (the
    contraction runs over the tokens)."""
    return _fp8.dequantize_128x1(*_fp8.quantize_128x1(np.asarray(m, np.float32)))


def _cached_tokens(u) -> np.ndarray:
    """The FP8 layer's token rows: u in E4M3 per 1x128 tile."""
    return _fp8.dequantize_1x128(*_fp8.quantize_1x128(np.asarray(u, np.float32)))


def expert_ffn_backward_fp8(x, w_gate, w_up, w_down, dy):
    """FP8 gradients of one expert.  x [n, d]: the forward's dequantised E4M3 token
    rows; w_gate, w_up [I, d], w_down [d, I]: dequantised E4M3 weights; dy [n, d] fp32.
    Returns (dx [n, d], dw_gate [I, d], dw_up [I, d], dw_down [d, I]), float64."""
    x = np.asarray(x, np.float64)
    wg, wu, wd = (np.asarray(w, np.float64) for w in (w_gate, w_up, w_down))
    a64 = x @ wg.T
    c64 = x @ wu.T
    h = _cached_activation(_fw.silu(a64) * c64)      # what the forward's down GEMM read
    a = _fp8.bf16_round(a64).astype(np.float64)
    c = _fp8.bf16_round(c64).astype(np.float64)
    dY = _fp8.bf16_round(dy).astype(np.float64)
    # Dgrad: dH = dY W_down, the SwiGLU backward, dx = dA W_gate + dC W_up
    dH = _fp8.bf16_round(_dgrad_operand(dY) @ wd).astype(np.float64)
    dA = (dH * c * silu_grad(a)).astype(np.float32)
    dC = (dH * _fw.silu(a)).astype(np.float32)
    dx = _dgrad_operand(dA) @ wg + _dgrad_operand(dC) @ wu
    # Wgrad: contractions over the expert's tokens
    dw_down = _wgrad_operand(dY).T @ _wgrad_operand(h)
    xc = _wgrad_operand(x)
    dw_gate = _wgrad_operand(_fp8.bf16_round(dA)).T @ xc
    dw_up = _wgrad_operand(_fp8.bf16_round(dC)).T @ xc
    return dx, dw_gate, dw_up, dw_down


def layer_backward_fp8(u, e, b, weights: dict, dh, K_r: int, G: int = 1, M: int = 1,
                       N_s: int = 0, seq_offsets=None, alpha: float = 0.0, idx=None) -> dict:
    """``layer_backward`` for the FP8 layer: the forward with E4M3 tokens (1x128), E4M3
    weights (128x128) and the re-quantised h, and the expert gradients of
    ``expert_ffn_backward_fp8``; routing, gates, the balance loss and the affinity
    gradients stay in float64 on the unquantised u.  dy = fp32(g) * fp32(dh) for a
    routed slot, dh for a shared expert.  Same keys as ``layer_backward``."""
    fw = forward64(u, e, b, weights, K_r, G, M, N_s, seq_offsets, alpha, idx)
    u = np.asarray(u, np.float64)
    e = np.asarray(e, np.float64)
    dh = np.asarray(dh, np.float64)
    s, idx, gate = fw["s"], fw["idx"], fw["gate"]
    wq = lambda w: _fp8.dequantize_128x128(*_fp8.quantize_128x128(np.asarray(w, np.float32)))
    x = _cached_tokens(u)
    routed = {k: wq(weights[k]) for k in ("w_gate", "w_up", "w_down")}
    shared = [tuple(wq(np.asarray(weights[k])[j]) for k in ("ws_gate", "ws_up", "ws_down"))
              for j in range(N_s)]
    du = dh.copy()
    grads = {k: np.zeros_like(v) for k, v in routed.items()}
    for k in ("ws_gate", "ws_up", "ws_down"):
        grads[k] = np.zeros((N_s,) + np.asarray(weights[k]).shape[1:])
    dh32 = dh.astype(np.float32)
    for j, (wg, wu, wd) in enumerate(shared):
        dx, dg_, du_, dd_ = expert_ffn_backward_fp8(x, wg, wu, wd, dh32)
        du += dx
        grads["ws_gate"][j], grads["ws_up"][j], grads["ws_down"][j] = dg_, du_, dd_
    y = np.zeros(idx.shape + (u.shape[1],))
    for i in np.unique(idx):
        rows, ks = np.nonzero(idx == i)
        wg, wu, wd = routed["w_gate"][i], routed["w_up"][i], routed["w_down"][i]
        y[rows, ks] = _fw.expert_ffn(x[rows], wg, wu, wd, h_quant=True)
        dy = gate[rows, ks].astype(np.float32)[:, None] * dh32[rows]
        dx, dg_, du_, dd_ = expert_ffn_backward_fp8(x[rows], wg, wu, wd, dy)
        np.add.at(du, rows, dx)
        grads["w_gate"][i] += dg_
        grads["w_up"][i] += du_
        grads["w_down"][i] += dd_
    dgate = np.einsum("td,tkd->tk", dh, y)
    ds = gate_backward(s, idx, dgate)
    if seq_offsets is not None:
        ds += balance_backward(s, idx, seq_offsets, K_r, alpha)
    dz = ds * s * (1.0 - s)
    du += dz @ e
    de = dz.T @ u
    return dict(grads, du=du, de=de, db=np.zeros(np.asarray(b).shape))
