"""The seeded input generator: shapes, dtypes, determinism and the stated
distributions (no layer arithmetic here)."""
import math

import pytest
import torch

import synth


def test_tiny_inputs_shapes_and_determinism():
    cfg = synth.config("tiny")
    a = synth.make_inputs(cfg)
    b = synth.make_inputs(cfg)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert a["u"].shape == (64, 256) and a["u"].dtype == torch.float32
    assert a["e"].shape == (16, 256)
    assert a["w_gate"].shape == (16, 128, 256) and a["w_down"].shape == (16, 256, 128)
    assert a["ws_gate"].shape == (1, 128, 256)
    assert a["b"].abs().max() <= 0.01 and a["b"].dtype == torch.float32
    assert a["seq_offsets"].tolist() == [0, 64]


def test_distributions():
    cfg = synth.config("tiny", T=512, d=512, I=256)
    x = synth.make_inputs(cfg)
    assert abs(x["u"].std().item() - 1.0) < 0.02
    assert abs(x["e"].std().item() * math.sqrt(512) - 1.0) < 0.05
    assert abs(x["w_down"].std().item() * math.sqrt(256) - 1.0) < 0.02
    assert abs(x["w_gate"].std().item() * math.sqrt(512) - 1.0) < 0.02


def test_bf16_storage_and_zero_bias():
    cfg = synth.config("mid", T=64, d=128, N_r=8, K_r=2, I=128, n_seq=4)
    x = synth.make_inputs(cfg)
    assert x["u"].dtype == torch.bfloat16 and x["w_up"].dtype == torch.bfloat16
    assert (x["b"] == 0).all()
    assert x["seq_offsets"].tolist() == [0, 16, 32, 48, 64]


def test_mixture_is_skewed():
    u = synth.mixture_tokens(256, 64, seed=1000)
    # component means have norm 3*sqrt(d): tokens are far from the origin
    assert u.norm(dim=1).mean() > 2.5 * math.sqrt(64)
    with pytest.raises(ValueError):
        synth.make_seq_offsets(10, 3)
