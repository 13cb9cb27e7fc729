"""GPU parity of the FP8 (E4M3) variant against the CPU oracle (marked gpu).

DeepSeek-V3 Technical Report reading guide (xyznot.com), Key ideas, FP8 bullet:
E4M3 on all tensors, activations scaled per 1x128 tile, weights per 128x128 block.
The quantiser is integer-exact work once the scale is fixed (one fp32 division for
the scale, one for each code, then round-to-nearest-even into E4M3), so codes and
scales must match the oracle bit for bit.  The layer output is compared with the
oracle run on the dequantised tokens and weights, with the SwiGLU output quantised
1x128 as well, at 5e-2 relative L2.
"""
import numpy as np
import pytest
import torch

import synth
import aux_loss_free_router_b300 as moe
from oracle import fp8 as ofp8
from tests.layer_harness import (check_output_full, check_routing, check_seq_stat, run_layer,
                                 to_np)

pytestmark = pytest.mark.gpu

FP8_REL = 5e-2


def _codes_to_values(q: torch.Tensor) -> np.ndarray:
    return ofp8.e4m3_decode(q.cpu().numpy())


def test_quantize_tokens_1x128_bit_exact():
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn(300, 2048, device="cuda", generator=g).mul_(3.0).bfloat16()
    x[7].zero_()                                  # an all-zero row: scale 1, codes 0
    x[8, :128] = 1e-6                             # a tile of tiny values (subnormal codes)
    x[9, 5] = 300.0                               # a tile with one large outlier
    q = torch.empty(300, 2048, dtype=torch.uint8, device="cuda")
    sc = torch.empty(300, 16, dtype=torch.float32, device="cuda")
    moe.quantize_e4m3(x, 1, q, sc)
    torch.cuda.synchronize()
    ref_q, ref_sc = ofp8.quantize_1x128(to_np(x))
    np.testing.assert_array_equal(to_np(sc), ref_sc)
    np.testing.assert_array_equal(_codes_to_values(q), ref_q)
    assert (sc[7] == 1).all() and (q[7] == 0).all()


def test_quantize_weights_128x128_bit_exact():
    g = torch.Generator(device="cuda").manual_seed(12)
    w = (torch.randn(3, 256, 384, device="cuda", generator=g) * 0.02).bfloat16()
    w[1, :128, 128:256] = 0                        # an all-zero block
    qw = moe.quantize_weights({"w_gate": w})
    torch.cuda.synchronize()
    ref_q, ref_sc = ofp8.quantize_128x128(to_np(w))
    np.testing.assert_array_equal(to_np(qw["w_gate_scale"]), ref_sc)
    np.testing.assert_array_equal(_codes_to_values(qw["w_gate"]), ref_q)
    assert qw["w_gate_scale"][1, 0, 1].item() == 1.0


def test_fp8_layer_matches_oracle():
    """The FP8 workload at full size (4096 tokens in 4 sequences, d=2048, 64 experts
    top-6, 2 shared, I=1408), every output element."""
    cfg = synth.config("fp8")
    r = run_layer(cfg)
    idx, _ = check_routing(cfg, r)
    check_seq_stat(cfg, r, idx)
    check_output_full(cfg, r, rel_tol=FP8_REL)


@pytest.mark.parametrize("T,d,I,N_r,K_r,G,M,N_s", [
    (300, 256, 384, 32, 4, 4, 2, 1),     # ragged T, group limit
    (129, 512, 256, 64, 8, 8, 4, 0),     # no shared expert
    (1, 384, 128, 16, 2, 1, 1, 2),       # a single token, d = 3 K chunks
    (700, 1024, 640, 16, 2, 1, 1, 1),    # d = 4 x 256 output tiles, I = 5 x 128
])
def test_fp8_ragged_layers(T, d, I, N_r, K_r, G, M, N_s):
    cfg = synth.MoEConfig("fp8-ragged", T=T, d=d, N_r=N_r, K_r=K_r, N_s=N_s, I=I, G=G, M=M,
                          dtype="bf16", bias="uniform", fp8=True, seed=T + 1)
    r = run_layer(cfg)
    idx, _ = check_routing(cfg, r)
    check_output_full(cfg, r, rel_tol=FP8_REL)


def test_fp8_down_tile_past_d():
    """d = 384 is one and a half 256-column output tiles: the second half of the last
    tile reads another expert's rows (or nothing) and must not be stored."""
    cfg = synth.MoEConfig("fp8-d384", T=200, d=384, N_r=8, K_r=2, N_s=1, I=256, G=1, M=1,
                          dtype="bf16", bias="zero", fp8=True, seed=5)
    r = run_layer(cfg)
    check_routing(cfg, r)
    check_output_full(cfg, r, rel_tol=FP8_REL)


def test_fp8_layer_is_deterministic():
    cfg = synth.config("fp8", T=512, n_seq=1)
    x = synth.make_inputs(cfg, device="cuda")
    r1 = run_layer(cfg, {k: v.clone() for k, v in x.items()})
    r2 = run_layer(cfg, {k: v.clone() for k, v in x.items()})
    np.testing.assert_array_equal(r1["h"], r2["h"])


@pytest.mark.parametrize("fp8", [False, True])
def test_expert_ffn_call_equals_the_two_step_calls(fp8):
    """moe_expert_ffn (h in its workspace; for E4M3 also h's scales) gives the same y as
    moe_expert_gate_up followed by moe_expert_down."""
    cfg = synth.config("fp8" if fp8 else "mid", T=512, n_seq=1)
    r = run_layer(cfg)
    lay, x = r["layer"], r["inputs"]
    xin = lay.u_q if fp8 else x["u"]
    kw = dict(x_perm_scale=lay.x_perm_scale, u_scale=lay.u_scale) if fp8 else {}
    y = torch.empty_like(lay.y)
    moe.expert_ffn(lay.x_perm, xin, lay.expert_offset, lay.shape, lay.ffn_weights, y, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y, lay.y)


def test_quantize_wide_magnitudes_bit_exact():
    """Codes over 4 M values whose tiles span 2^-60 .. 2^60 and whose values sit down to
    2^-40 below their tile's largest: the library divides by the scale through a
    reciprocal and one correction step, and must still give the oracle's codes (its
    fp32 division) everywhere."""
    g = torch.Generator(device="cuda").manual_seed(21)
    rows, cols = 4096, 1024
    x = torch.randn(rows, cols, device="cuda", generator=g)
    mag = torch.exp2(torch.randint(-60, 60, (rows, cols // 128, 1), device="cuda", generator=g).float())
    spread = torch.exp2(-torch.randint(0, 40, (rows, cols), device="cuda", generator=g).float())
    x = (x.view(rows, cols // 128, 128) * mag).view(rows, cols) * spread
    q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    sc = torch.empty(rows, cols // 128, dtype=torch.float32, device="cuda")
    moe.quantize_e4m3(x, 1, q, sc)
    torch.cuda.synchronize()
    ref_q, ref_sc = ofp8.quantize_1x128(to_np(x))
    np.testing.assert_array_equal(to_np(sc), ref_sc)
    np.testing.assert_array_equal(_codes_to_values(q), ref_q)


def test_quantize_fp32_input_bit_exact():
    g = torch.Generator(device="cuda").manual_seed(13)
    x = torch.randn(64, 384, device="cuda", generator=g) * 10.0
    q = torch.empty(64, 384, dtype=torch.uint8, device="cuda")
    sc = torch.empty(64, 3, dtype=torch.float32, device="cuda")
    moe.quantize_e4m3(x, 1, q, sc)
    torch.cuda.synchronize()
    ref_q, ref_sc = ofp8.quantize_1x128(to_np(x))
    np.testing.assert_array_equal(to_np(sc), ref_sc)
    np.testing.assert_array_equal(_codes_to_values(q), ref_q)


def test_fp8_layer_on_the_hand_worked_token():
    """The FP8 kernels on the hand-worked single token of
    tests/golden/fp8_layer_single_token.json: routing on the unquantised u picks
    expert 0 (the dequantised token would pick expert 1), and h' equals the worked
    value up to the bf16 rounding of the experts' outputs y (|dh'| <= 2^-8 of the
    largest |y| that enters it)."""
    from tests.test_oracle_pins import fp8_golden_case
    g, u, e, b, w, h_ref = fp8_golden_case()
    cfg = synth.MoEConfig("fp8-golden", T=g["T"], d=g["d"], N_r=g["N_r"], K_r=g["K_r"],
                          N_s=g["N_s"], I=g["I"], dtype="bf16", bias="zero", fp8=True)
    dev = "cuda"
    x = {"u": torch.from_numpy(u).to(dev).bfloat16(), "e": torch.from_numpy(e).to(dev).bfloat16(),
         "b": torch.from_numpy(b).to(dev), "seq_offsets": synth.make_seq_offsets(1, 1).to(dev)}
    for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"):
        x[k] = torch.from_numpy(w[k]).to(dev).bfloat16()
    r = run_layer(cfg, x)
    assert r["topk_idx"].tolist() == g["idx"]
    np.testing.assert_array_equal(r["topk_gate"], np.array(g["gate"], np.float32))
    np.testing.assert_allclose(r["s_out"], g["s"], rtol=2e-6)
    err = np.abs(r["h"].astype(np.float64) - h_ref)
    assert err.max() <= 2.0 ** -8 * 29.0, err.max()          # |y| <= 29 in this case
    assert err[:, 2:].max() == 0.0
