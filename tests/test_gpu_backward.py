"""GPU parity of the backward pass against the CPU oracle (marked gpu).

moe_backward returns the gradients of J = sum(dh * h') + mean over sequences of the
balance loss, at the forward pass's selection, with respect to u, the centroids e and
every expert weight.  The oracle (oracle/moe_backward.py, float64, pinned on the CPU by
finite differences) is run at the same selection (the kernels' topk_idx) on the same
bf16 values.  Every element of every gradient is compared.

Tolerance: the kernels keep dY = g*dh, the recomputed pre-activations a and c, dA, dC,
dX and dz in bf16 (one rounding each, relative 2^-9 = 2e-3) and accumulate in fp32; a
gradient passes through at most three such roundings, so its relative L2 error stays
well below 1e-2.  The bound is 2e-2 relative L2 per gradient (du is compared without
its residual term dh, which is exact).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import aux_loss_free_router_b300 as moe
from tests.layer_harness import rel_l2, to_np

pytestmark = pytest.mark.gpu

BWD_REL = 2e-2


def run_backward(cfg, x=None, with_balance=True, dh_seed=5, dh_scale=1.0):
    x = x if x is not None else synth.make_inputs(cfg, device="cuda")
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    layer = moe.MoELayer(T=cfg.T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I, G=cfg.G,
                         M=cfg.M, e=x["e"], b=x["b"].clone(), weights=w, n_seq=cfg.n_seq,
                         alpha=cfg.alpha, want_s=True)
    layer.step(x["u"], x["seq_offsets"], update_bias=False)
    g = torch.Generator(device="cuda").manual_seed(dh_seed)
    dh = torch.randn(cfg.T, cfg.d, generator=g, device="cuda") * dh_scale
    grads = layer.backward(x["u"], dh, x["seq_offsets"] if with_balance else None)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    got = {k: to_np(v) for k, v in grads.items()}
    ref = oracle.moe_backward.layer_backward(
        to_np(x["u"]), to_np(x["e"]), to_np(x["b"]),
        {k: to_np(v) for k, v in w.items()}, to_np(dh), cfg.K_r, cfg.G, cfg.M, cfg.N_s,
        seq_offsets=to_np(x["seq_offsets"]) if with_balance else None,
        alpha=cfg.alpha if with_balance else 0.0, idx=to_np(layer.topk_idx))
    return got, ref, to_np(dh), layer


def check_grads(cfg, got, ref, dh, tol=BWD_REL):
    errs = {"u": rel_l2(got["u"] - dh, ref["du"] - dh), "e": rel_l2(got["e"], ref["de"])}
    for k in ("w_gate", "w_up", "w_down"):
        errs[k] = rel_l2(got[k], ref[k])
    if cfg.N_s:
        for k in ("ws_gate", "ws_up", "ws_down"):
            errs[k] = rel_l2(got[k], ref[k])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, (bad, errs)
    return errs


@pytest.mark.parametrize("T,d,I,N_r,K_r,G,M,N_s,n_seq", [
    (256, 512, 256, 64, 4, 4, 2, 1, 2),     # group limit, two sequences
    (300, 320, 200, 64, 4, 1, 1, 1, 3),     # d and I not tile multiples, ragged segments
    (64, 256, 128, 64, 6, 1, 1, 0, 1),      # no shared expert, many experts without tokens
])
def test_backward_matches_oracle(T, d, I, N_r, K_r, G, M, N_s, n_seq):
    cfg = synth.MoEConfig("bwd", T=T, d=d, N_r=N_r, K_r=K_r, N_s=N_s, I=I, G=G, M=M, n_seq=n_seq,
                          dtype="bf16", bias="uniform", seed=T + d)
    got, ref, dh, _ = run_backward(cfg)
    check_grads(cfg, got, ref, dh)


def test_backward_balance_term():
    """The balance loss's gradient, made visible: with a small upstream gradient (dh at
    1e-5) the balance term dominates dz, so de and du change by far more than the
    tolerance when it is left out, and the kernels follow the oracle either way."""
    cfg = synth.MoEConfig("bwd-bal", T=256, d=256, N_r=64, K_r=4, N_s=1, I=128, n_seq=2,
                          dtype="bf16", bias="uniform", seed=9, alpha=1.0)
    x = synth.make_inputs(cfg, device="cuda")
    got, ref, dh, _ = run_backward(cfg, x=x, dh_scale=1e-5)
    check_grads(cfg, got, ref, dh)
    got0, ref_nb, dh0, _ = run_backward(cfg, x=x, with_balance=False, dh_scale=1e-5)
    assert rel_l2(ref["de"], ref_nb["de"]) > 5 * BWD_REL     # the term matters here
    assert rel_l2(got["e"], got0["e"]) > 5 * BWD_REL
    check_grads(cfg, got0, ref_nb, dh0)


def test_backward_empty_experts_get_zero_weight_gradients():
    cfg = synth.MoEConfig("bwd-zero", T=128, d=256, N_r=64, K_r=2, N_s=1, I=128, n_seq=1,
                          dtype="bf16", bias="zero", seed=3)
    x = synth.make_inputs(cfg, device="cuda")
    x["b"][:2] = 1.0                      # every token picks experts 0 and 1
    got, ref, dh, layer = run_backward(cfg, x=x)
    assert (to_np(layer.load)[2:] == 0).all()
    for k in ("w_gate", "w_up", "w_down"):
        assert (got[k][2:] == 0).all()
    check_grads(cfg, got, ref, dh)


def test_backward_mid_shape_every_element():
    """The mid workload (4096 tokens in 4 sequences, d=2048, 64 experts top-6, 2 shared,
    I=1408): every gradient element against the oracle."""
    cfg = synth.config("mid")
    got, ref, dh, _ = run_backward(cfg)
    errs = check_grads(cfg, got, ref, dh)
    print("backward mid shape rel L2:", {k: f"{v:.2e}" for k, v in errs.items()})
