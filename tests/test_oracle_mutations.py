"""Planted mistakes in the CPU oracle must be caught by its pins.

Each case swaps one oracle function for a plausible wrong variant (on the CPU, in
this process only) and checks that at least one pin of ``test_oracle_pins`` fails.
"""
import numpy as np
import pytest

import oracle
from oracle import moe_oracle as mo
import tests.test_oracle_pins as pins


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(mo, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def _fails(test, *args):
    with pytest.raises(AssertionError):
        test(*args)


def test_gate_from_biased_keys_is_caught(monkeypatch):
    orig = mo.gate_values

    def bad(s, idx, _b=np.array([-0.25, 0.0, 0.0, 0.5], np.float32)):
        s = np.asarray(s, np.float32)
        return orig(s + _b[: s.shape[1]] if s.shape[1] == 4 else s, idx)
    _patch(monkeypatch, "gate_values", bad)
    _fails(pins.test_golden_bias_routing)


def test_ties_to_higher_index_is_caught(monkeypatch):
    monkeypatch.setattr(mo, "_order_desc",
                        lambda v, c: sorted(c, key=lambda i: (-float(v[i]), -i)))
    _fails(pins.test_topk_brute_force, 8, 2)


def test_group_score_over_all_members_is_caught(monkeypatch):
    def bad(keys_row, G, M, K_r):
        per = len(keys_row) // G
        return [np.float32(sum(keys_row[g * per:(g + 1) * per])) for g in range(G)]
    monkeypatch.setattr(mo, "group_scores", bad)
    _fails(pins.test_group_limited_brute_force, 12, 3, 1, 2)


def test_bias_update_sign_flip_is_caught(monkeypatch):
    orig = mo.bias_update
    _patch(monkeypatch, "bias_update",
           lambda b, load, T, K_r, g: orig(b, load, T, K_r, -g))
    _fails(pins.test_golden_bias_update)


def test_sigmoid_instead_of_silu_is_caught(monkeypatch):
    monkeypatch.setattr(mo, "silu", lambda z: 1.0 / (1.0 + np.exp(-np.asarray(z))))
    _fails(pins.test_golden_ffn_single_token)


def test_transposed_down_projection_is_caught(monkeypatch):
    def bad(x, w_gate, w_up, w_down, h_quant=False):
        x = np.asarray(x, np.float64)
        h = mo.silu(x @ np.asarray(w_gate).T) * (x @ np.asarray(w_up).T)
        wd = np.asarray(w_down)
        return h @ (wd.T if wd.shape[0] == wd.shape[1] else wd.T[:, ::-1])
    monkeypatch.setattr(mo, "expert_ffn", bad)
    _fails(pins.test_golden_ffn_single_token)


def test_dropped_shared_expert_is_caught(monkeypatch):
    orig = mo.layer_output
    monkeypatch.setattr(mo, "layer_output",
                        lambda u, idx, gate, routed, shared, **kw: orig(u, idx, gate, routed, [], **kw))
    _fails(pins.test_identical_experts_closed_form)


def test_p_normalised_over_selected_only_is_caught(monkeypatch):
    def bad(s, seq_offsets):
        s = np.asarray(s, np.float64)
        off = np.asarray(seq_offsets)
        top = np.sort(s, 1)[:, -2:].sum(1, keepdims=True)
        sp = s / top
        return np.stack([sp[off[j]:off[j + 1]].sum(0) for j in range(len(off) - 1)])
    monkeypatch.setattr(mo, "seq_p_sums", bad)
    monkeypatch.setattr(oracle, "seq_p_sums", bad)
    _fails(pins.test_seq_stat_uniform_closed_form_and_sums)


def test_e4m3_round_half_away_is_caught(monkeypatch):
    from oracle import fp8

    def bad(x):
        x = np.asarray(x, np.float64)
        a = np.abs(x)
        _, ex = np.frexp(a)
        q = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
        return np.copysign(np.minimum(np.floor(a / q + 0.5) * q, 448.0), x)
    monkeypatch.setattr(fp8, "e4m3_round", bad)
    monkeypatch.setattr(pins.ofp8, "e4m3_round", bad)
    _fails(pins.test_e4m3_matches_torch_cast_in_range)


# --------------------------------------------------- the FP8 layer's composition --

def test_fp8_routing_on_dequantised_tokens_is_caught(monkeypatch):
    from oracle import fp8
    orig = mo.route

    def bad(u, e, b, K_r, G=1, M=1, s=None):
        q, sc = fp8.quantize_1x128(np.asarray(u, np.float32))
        return orig(fp8.dequantize_1x128(q, sc).astype(np.float32), e, b, K_r, G, M, s=s)
    monkeypatch.setattr(mo, "route", bad)
    _fails(pins.test_golden_fp8_layer_single_token)


def test_fp8_skipped_h_quantisation_is_caught(monkeypatch):
    orig = mo.expert_ffn
    monkeypatch.setattr(mo, "expert_ffn",
                        lambda x, wg, wu, wd, h_quant=False: orig(x, wg, wu, wd, False))
    _fails(pins.test_golden_fp8_layer_single_token)


def test_fp8_shared_expert_on_unquantised_tokens_is_caught(monkeypatch):
    orig = mo.layer_output

    def bad(u, idx, gate, routed, shared, x=None, h_quant=False):
        h = orig(u, idx, gate, routed, [], x=x, h_quant=h_quant)
        for (wg, wu, wd) in shared:
            h += mo.expert_ffn(u, wg, wu, wd, h_quant)
        return h
    monkeypatch.setattr(mo, "layer_output", bad)
    _fails(pins.test_golden_fp8_layer_single_token)
