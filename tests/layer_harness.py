"""Shared test harness: run the CUDA layer through the C ABI on seeded inputs and
bring the results back to numpy; compare them with the CPU oracle.

Routing is compared bit-exactly by taking the oracle's decision on the library's own
fp32 affinities (both sides then decide on identical fp32 keys); the layer output is
compared with the oracle run on those same affinities.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import aux_loss_free_router_b300 as moe


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.cpu().numpy()


def run_layer(cfg: synth.MoEConfig, inputs: dict | None = None, device="cuda"):
    """Run route -> dispatch -> gate/up -> down -> combine -> bias update -> seq stat."""
    x = inputs if inputs is not None else synth.make_inputs(cfg, device=device)
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    b0 = x["b"].clone()
    layer = moe.MoELayer(T=cfg.T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I,
                         G=cfg.G, M=cfg.M, e=x["e"], b=x["b"].clone(), weights=w,
                         n_seq=cfg.n_seq, gamma=cfg.gamma, alpha=cfg.alpha, want_s=True,
                         fp8=cfg.fp8)
    out = layer.step(x["u"], x["seq_offsets"])
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    res = dict(layer=layer, inputs=x, b0=b0, out=out)
    for k in ("topk_idx", "topk_gate", "s_out", "seq_p_sum", "load", "expert_offset",
              "perm_token", "inv_row", "stat", "stat_mean"):
        res[k] = to_np(getattr(layer, k))
    res["h"] = to_np(out)
    res["b_new"] = to_np(layer.b)
    return res


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_routing(cfg, r):
    """Bit-exact routing, dispatch and bias update given the library's fp32 s."""
    s = r["s_out"]
    b = to_np(r["b0"])
    idx = oracle.select_experts(s, b, cfg.K_r, cfg.G, cfg.M)
    np.testing.assert_array_equal(r["topk_idx"], idx)
    np.testing.assert_allclose(r["topk_gate"], oracle.gate_values(s, idx), rtol=1e-6, atol=0)
    dp = oracle.dispatch(idx, cfg.N_r)
    for k in ("load", "perm_token", "inv_row"):
        np.testing.assert_array_equal(r[k], dp[k], err_msg=k)
    np.testing.assert_array_equal(r["expert_offset"], dp["offset"])
    np.testing.assert_array_equal(r["b_new"], oracle.bias_update(b, dp["load"], cfg.T, cfg.K_r, cfg.gamma))
    return idx, dp


def check_affinity(cfg, r, atol):
    x = r["inputs"]
    s_ref = oracle.affinity(to_np(x["u"]), to_np(x["e"]))
    err = np.abs(r["s_out"].astype(np.float64) - s_ref).max()
    assert err <= atol, f"affinity max abs error {err}"
    return s_ref


def check_seq_stat(cfg, r, idx):
    off = to_np(r["inputs"]["seq_offsets"]).astype(np.int64)
    ref_p = oracle.seq_p_sums(r["s_out"], off)
    np.testing.assert_allclose(r["seq_p_sum"], ref_p, rtol=1e-5, atol=1e-6)
    st, mean = oracle.seq_balance_stat(r["s_out"], idx, off, cfg.N_r, cfg.K_r, cfg.alpha)
    np.testing.assert_allclose(r["stat"], st, rtol=1e-5)
    np.testing.assert_allclose(r["stat_mean"][0], mean, rtol=1e-5)


def oracle_weights(x: dict) -> dict:
    return {k: to_np(x[k]) for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}


def check_output_full(cfg, r, rel_tol, abs_tol=None, abs_per_rms=False):
    """rel L2 and max-abs of h' against the oracle.  With ``abs_per_rms`` the max-abs
    bound scales with the reference's RMS when that exceeds 1 (inputs far from unit
    scale, as the Gaussian-mixture tokens are)."""
    x = r["inputs"]
    ref = oracle.moe_forward(to_np(x["u"]), to_np(x["e"]), to_np(r["b0"]), oracle_weights(x),
                             cfg.K_r, cfg.G, cfg.M, cfg.N_s, s=r["s_out"], fp8=cfg.fp8)
    err = rel_l2(r["h"], ref["h"])
    assert err <= rel_tol, f"rel L2 {err}"
    if abs_tol is not None:
        if abs_per_rms:
            abs_tol = abs_tol * max(1.0, float(np.sqrt(np.mean(ref["h"] ** 2))))
        mx = np.abs(r["h"] - ref["h"]).max()
        assert mx <= abs_tol, f"max abs {mx} (bound {abs_tol})"
    return ref


def check_output_sampled(cfg, r, tokens, rel_tol, abs_tol):
    """h' of selected tokens only: the oracle fetches just the experts they use."""
    x = r["inputs"]
    tokens = np.asarray(tokens)
    u = to_np(x["u"][torch.as_tensor(tokens, device=x["u"].device)])
    idx = r["topk_idx"][tokens]
    gate = oracle.gate_values(r["s_out"][tokens], idx)

    def routed(i):
        return tuple(to_np(x[k][i]) for k in ("w_gate", "w_up", "w_down"))

    shared = [tuple(to_np(x[k][j]) for k in ("ws_gate", "ws_up", "ws_down"))
              for j in range(cfg.N_s)]
    ref = oracle.layer_output(u, idx, gate, routed, shared)
    got = r["h"][tokens]
    err = rel_l2(got, ref)
    mx = np.abs(got - ref).max()
    assert err <= rel_tol and mx <= abs_tol, f"rel L2 {err}, max abs {mx}"
    return err, mx
