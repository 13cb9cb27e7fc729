"""CPU pins of the FP8 backward oracle (``oracle.moe_backward.layer_backward_fp8``).

A two-token, one-expert layer (d = I = 256) built so that every E4M3 step is exact
except the ones a pin is about, where a tile holds one value 2^20 times larger than
another: the small value then falls below half the smallest E4M3 subnormal and
quantises to zero.  Which values vanish says which way each tile runs and which
tensor each GEMM reads; every expected value below is worked out by hand.

  u:  token 0 = e_0 + 2^-22 e_1, token 1 = e_0 + e_130 (2^-22 vanishes in the cached
      E4M3 tokens);
  W_gate rows: 0 -> e_0, 1 -> e_0, 3 -> e_0 + e_5, 2 -> 16 e_130;
  W_up rows:   0 -> e_0, 1 -> 0.5 e_0, 3 -> 2^-12 e_0, 2 -> 2^16 e_130;
  W_down: [0,0] = 1, [1,1] = 1, [0,3] = 2^-8 (every 128x128 block is exact in E4M3);
  dh: token 0 = 2^20 e_0 + e_1, token 1 = e_1; one expert, top-1: the gate is 1.

With s1 = silu(1) and p1 = silu'(1):
  a = (1, 1, 0|16, 1) and c = (1, 0.5, 0|2^16, 2^-12) at features 0..3 (token 0|1);
  the cached h of token 1 keeps only h[1,2] = silu(16) 2^16 (its other entries vanish);
  Dgrad (1x128 along d): dY[0,1] = 1 vanishes beside 2^20, so dH[0] = 2^20 e_0 + 2^12 e_3
  and dH[1] = e_1; dA[0,3] = p1 vanishes beside dA[0,0] = 2^20 p1 in its 1x128 tile;
  Wgrad (128x1 along the tokens): columns of dY, h, dA, dC over the two tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import moe_backward as mb

S1 = 1.0 / (1.0 + np.exp(-1.0))                 # silu(1) = sigma(1)
P1 = S1 * (1.0 + (1.0 - S1))                     # silu'(1)
SILU16 = 16.0 / (1.0 + np.exp(-16.0))
REL = 1e-5


def bf16(v: float) -> float:
    return float(torch.tensor(v, dtype=torch.float32).bfloat16().float())


def case():
    d = I = 256
    u = np.zeros((2, d), np.float32)
    u[0, 0], u[0, 1] = 1.0, 2.0 ** -22
    u[1, 0], u[1, 130] = 1.0, 1.0
    wg = np.zeros((1, I, d), np.float32)
    wu = np.zeros((1, I, d), np.float32)
    wd = np.zeros((1, d, I), np.float32)
    wg[0, 0, 0] = wg[0, 1, 0] = wg[0, 3, 0] = wg[0, 3, 5] = 1.0
    wg[0, 2, 130] = 16.0
    wu[0, 0, 0], wu[0, 1, 0], wu[0, 3, 0], wu[0, 2, 130] = 1.0, 0.5, 2.0 ** -12, 2.0 ** 16
    wd[0, 0, 0], wd[0, 1, 1], wd[0, 0, 3] = 1.0, 1.0, 2.0 ** -8
    dh = np.zeros((2, d), np.float32)
    dh[0, 0], dh[0, 1], dh[1, 1] = 2.0 ** 20, 1.0, 1.0
    weights = {"w_gate": wg, "w_up": wu, "w_down": wd,
               "ws_gate": np.zeros((0, I, d), np.float32), "ws_up": np.zeros((0, I, d), np.float32),
               "ws_down": np.zeros((0, d, I), np.float32)}
    e = np.zeros((1, d), np.float32)
    b = np.zeros(1, np.float32)
    return u, e, b, weights, dh


def run():
    u, e, b, w, dh = case()
    return mb.layer_backward_fp8(u, e, b, w, dh, K_r=1, N_s=0, idx=np.zeros((2, 1), np.int64))


def close(got, want):
    return abs(got - want) <= REL * abs(want)


def test_wgrad_tiles_run_along_tokens_and_read_the_cached_h():
    """dW_down[1,0] = dY[0,1] h[0,0] + dY[1,1] h[1,0] = s1 + 0: dY's column 1 (1, 1) is
    exact in its 128x1 tile, while h[1,0] vanished in the forward's 1x128 cache."""
    g = run()["w_down"][0]
    assert close(g[1, 0], S1), g[1, 0]
    assert close(g[0, 0], 2.0 ** 20 * S1), g[0, 0]
    assert close(g[1, 2], SILU16 * 2.0 ** 16), g[1, 2]


def test_dgrad_tiles_run_along_features():
    """dY[0,1] vanishes in token 0's 1x128 tile, so dH[0,1] = dC[0,1] = 0 and
    dW_up[1,0] = bf16(dC[1,1]) x[1,0] = bf16(s1) (not twice that)."""
    g = run()
    assert close(g["w_up"][0][1, 0], bf16(S1)), g["w_up"][0][1, 0]
    assert close(g["w_up"][0][0, 0], bf16(2.0 ** 20 * S1)), g["w_up"][0][0, 0]
    assert close(g["w_gate"][0][0, 0], bf16(2.0 ** 20 * P1)), g["w_gate"][0][0, 0]


def test_dgrad_quantises_the_swiglu_gradients():
    """dA[0,3] = p1 vanishes beside 2^20 p1 in the Dgrad operand, so feature 5 (reached
    only through W_gate row 3) gets nothing in dx[0]; Wgrad quantises dA on its own:
    dW_gate[3,0] = bf16(p1)."""
    g = run()
    assert g["du"][0, 5] == 0.0, g["du"][0, 5]
    assert close(g["w_gate"][0][3, 0], bf16(P1)), g["w_gate"][0][3, 0]
    want0 = 2.0 ** 20 * (1.0 + P1 + S1) + S1             # dh + 2^20 p1 + 2^20 s1 + s1
    assert close(g["du"][0, 0], want0), g["du"][0, 0]
    assert close(g["du"][1, 0], 0.5 * P1 + 0.5 * S1), g["du"][1, 0]


def test_wgrad_reads_the_cached_tokens():
    """u[0,1] = 2^-22 vanished in the E4M3 tokens, so dW_gate[:,1] is exactly zero."""
    g = run()["w_gate"][0]
    assert not g[:, 1].any()


# ------------------------------------------------------------- planted mistakes ----

PINS = [test_wgrad_tiles_run_along_tokens_and_read_the_cached_h, test_dgrad_tiles_run_along_features,
        test_dgrad_quantises_the_swiglu_gradients, test_wgrad_reads_the_cached_tokens]


def _some_pin_fails():
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    return failed > 0


def _rows(m):
    return oracle.fp8.dequantize_1x128(*oracle.fp8.quantize_1x128(np.asarray(m, np.float32)))


def _cols(m):
    return oracle.fp8.dequantize_128x1(*oracle.fp8.quantize_128x1(np.asarray(m, np.float32)))


def _fp32(m):
    return np.asarray(m, np.float32).astype(np.float64)


@pytest.mark.parametrize("name,fn", [
    ("_wgrad_operand", _rows),         # Wgrad tiles along the features
    ("_dgrad_operand", _cols),         # Dgrad tiles along the tokens
    ("_cached_activation", _fp32),     # Wgrad reads the fp32 h, not the cached E4M3 one
    ("_dgrad_operand", _fp32),         # Dgrad operands left unquantised
    ("_cached_tokens", _fp32),         # the FFNs read u, not the E4M3 tokens
])
def test_planted_mistake_is_caught(monkeypatch, name, fn):
    assert not _some_pin_fails()
    monkeypatch.setattr(mb, name, fn)
    assert _some_pin_fails()


def test_close_to_the_float64_backward():
    """On a random layer the FP8 gradients stay within E4M3's precision of the float64
    ones (3 mantissa bits: a few per cent in relative L2), and no further."""
    import synth
    cfg = synth.MoEConfig("fp8-bwd-pin", T=96, d=256, N_r=8, K_r=2, N_s=1, I=256, n_seq=2,
                          dtype="bf16", bias="uniform", seed=4)
    x = synth.make_inputs(cfg, device="cpu")
    f = lambda t: t.float().numpy()
    w = {k: f(x[k]) for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    dh = np.random.default_rng(1).standard_normal((cfg.T, cfg.d)).astype(np.float32)
    args = (f(x["u"]), f(x["e"]), f(x["b"]), w, dh, cfg.K_r, cfg.G, cfg.M, cfg.N_s, f(x["seq_offsets"]), 1e-4)
    r8 = mb.layer_backward_fp8(*args)
    r = mb.layer_backward(*args)
    for k in ("du", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"):
        err = np.linalg.norm(r8[k] - r[k]) / np.linalg.norm(r[k])
        assert 5e-3 < err < 0.15, (k, err)


def test_quantize_128x1_matches_torch_e4m3():
    """128x1 tiles from the first row, the last one short: codes are torch's E4M3 cast of
    x / scale (scale = amax / 448 in fp32, 1 for an all-zero tile)."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((300, 6)) * np.exp(rng.standard_normal((300, 6)) * 3)).astype(np.float32)
    x[256:, 2] = 0.0                                   # an all-zero short tile
    q, sc = oracle.fp8.quantize_128x1(x)
    assert sc.shape == (3, 6) and sc[2, 2] == 1.0
    for t in range(3):
        rows = slice(128 * t, min(300, 128 * (t + 1)))
        amax = np.abs(x[rows]).max(axis=0)
        want_sc = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
        assert np.array_equal(sc[t], want_sc)
        codes = torch.tensor(x[rows] / want_sc).to(torch.float8_e4m3fn).float().numpy()
        assert np.array_equal(q[rows], codes.astype(np.float64))
    assert np.allclose(oracle.fp8.dequantize_128x1(q, sc), q * np.repeat(sc, 128, axis=0)[:300])
