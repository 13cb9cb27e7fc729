"""GPU parity of the FP8 backward pass against the CPU oracle (marked gpu).

moe_backward_fp8 runs the expert GEMMs' backward in E4M3 (Fprop again, Dgrad on 1x128
tiles, Wgrad on 128x1 tiles over each expert's tokens, reading the cached E4M3
activations); ``oracle.moe_backward.layer_backward_fp8`` (float64, pinned on the CPU)
computes the same gradients at the kernels' selection from the same bf16 inputs.  The
oracle rounds to bf16 where the kernels do before quantising (a, c, dY, dH and the dA,
dC that Wgrad reads), so both sides decide the E4M3 codes on the same values; what
remains is fp32 accumulation order, the kernels' bf16 dH / dX / dz, and the rare code
that an fp32-versus-float64 difference moves across a rounding boundary (each such
code moves one E4M3 step, 2^-3 relative).  The bound is 2e-2 relative L2 per gradient
(du without its exact residual term dh), as for the bf16 backward.
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


def run_backward_fp8(cfg, x=None, with_balance=True, dh_seed=5):
    x = x if x is not None else synth.make_inputs(cfg, device="cuda")
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    layer = moe.MoELayer(T=cfg.T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I, G=cfg.G,
                         M=cfg.M, e=x["e"], b=x["b"].clone(), weights=w, n_seq=cfg.n_seq,
                         alpha=cfg.alpha, want_s=True, fp8=True)
    layer.step(x["u"], x["seq_offsets"], update_bias=False)
    g = torch.Generator(device="cuda").manual_seed(dh_seed)
    dh = torch.randn(cfg.T, cfg.d, generator=g, device="cuda")
    grads = layer.backward(x["u"], dh, x["seq_offsets"] if with_balance else None)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    got = {k: to_np(v) for k, v in grads.items()}
    ref = oracle.moe_backward.layer_backward_fp8(
        to_np(x["u"]), to_np(x["e"]), to_np(x["b"]),
        {k: to_np(v) for k, v in w.items()}, to_np(dh), cfg.K_r, cfg.G, cfg.M, cfg.N_s,
        seq_offsets=to_np(x["seq_offsets"]) if with_balance else None,
        alpha=cfg.alpha if with_balance else 0.0, idx=to_np(layer.topk_idx))
    return got, ref, to_np(dh)


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
    (256, 256, 256, 64, 4, 4, 2, 1, 2),     # group limit, two sequences
    (300, 384, 256, 64, 4, 1, 1, 1, 3),     # d = 3 x 128, ragged segments
    (64, 256, 128, 64, 6, 1, 1, 0, 1),      # no shared expert, many experts without tokens
])
def test_backward_fp8_matches_oracle(T, d, I, N_r, K_r, G, M, N_s, n_seq):
    cfg = synth.MoEConfig("bwd8", T=T, d=d, N_r=N_r, K_r=K_r, N_s=N_s, I=I, G=G, M=M, n_seq=n_seq,
                          dtype="bf16", bias="uniform", seed=T + d)
    got, ref, dh = run_backward_fp8(cfg)
    errs = check_grads(cfg, got, ref, dh)
    print("fp8 backward rel L2:", {k: f"{v:.2e}" for k, v in errs.items()})


def test_backward_fp8_empty_experts_get_zero_weight_gradients():
    cfg = synth.MoEConfig("bwd8-zero", T=128, d=256, N_r=64, K_r=2, N_s=1, I=128, n_seq=1,
                          dtype="bf16", bias="zero", seed=3)
    x = synth.make_inputs(cfg, device="cuda")
    x["b"][:2] = 1.0                      # every token picks experts 0 and 1
    got, ref, dh = run_backward_fp8(cfg, x=x)
    for k in ("w_gate", "w_up", "w_down"):
        assert (got[k][2:] == 0).all()
    check_grads(cfg, got, ref, dh)


def test_backward_fp8_mid_shape_every_element():
    """The mid workload (4096 tokens in 4 sequences, d=2048, 64 experts top-6, 2 shared,
    I=1408 = 11 x 128): every gradient element against the oracle."""
    cfg = synth.config("mid")
    got, ref, dh = run_backward_fp8(cfg)
    errs = check_grads(cfg, got, ref, dh)
    print("fp8 backward mid shape rel L2:", {k: f"{v:.2e}" for k, v in errs.items()})
