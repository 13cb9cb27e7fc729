"""Pins of the backward-pass oracle (CPU).

The gradients in ``oracle.moe_backward`` are pinned to central finite differences of
the float64 forward at a frozen selection (the forward itself is pinned in
``test_oracle_pins.py``, and ``forward64`` is checked against it here), to the
invariances the normalisations imply, and to closed forms; each planted mistake in
the backward must make a pin fail.
"""
import numpy as np
import pytest

import oracle
from oracle import moe_backward as mb

SHAPE = dict(T=6, d=5, N_r=6, K_r=2, G=3, M=1, N_s=1, I=4)
SEQ = np.array([0, 3, 6])
ALPHA = 0.3
WKEYS = ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")


def _inputs(seed=0, T=6, d=5, N_r=6, K_r=2, G=3, M=1, N_s=1, I=4):
    rng = np.random.default_rng(seed)
    u = rng.standard_normal((T, d))
    e = rng.standard_normal((N_r, d)) / np.sqrt(d)
    b = rng.uniform(-0.01, 0.01, N_r).astype(np.float32)
    w = {"w_gate": rng.standard_normal((N_r, I, d)) / np.sqrt(d),
         "w_up": rng.standard_normal((N_r, I, d)) / np.sqrt(d),
         "w_down": rng.standard_normal((N_r, d, I)) / np.sqrt(I),
         "ws_gate": rng.standard_normal((N_s, I, d)) / np.sqrt(d),
         "ws_up": rng.standard_normal((N_s, I, d)) / np.sqrt(d),
         "ws_down": rng.standard_normal((N_s, d, I)) / np.sqrt(I)}
    dh = rng.standard_normal((T, d))
    return u, e, b, w, dh


def _objective(u, e, b, w, dh, idx, seq=SEQ, alpha=ALPHA, sh=SHAPE):
    fw = mb.forward64(u, e, b, w, sh["K_r"], sh["G"], sh["M"], sh["N_s"], seq, alpha, idx)
    return float(np.sum(dh * fw["h"])) + (fw["bal_mean"] if seq is not None else 0.0)


def _fd_mismatch(seed=0, eps=1e-6, seq=SEQ, alpha=ALPHA):
    """Largest |analytic - finite difference| / max(1, |analytic|) over every input."""
    sh = SHAPE
    u, e, b, w, dh = _inputs(seed)
    idx = mb.forward64(u, e, b, w, sh["K_r"], sh["G"], sh["M"], sh["N_s"])["idx"]
    g = mb.layer_backward(u, e, b, w, dh, sh["K_r"], sh["G"], sh["M"], sh["N_s"], seq, alpha, idx)
    worst = 0.0
    params = {"du": ("u", u), "de": ("e", e)}
    params.update({k: (k, w[k]) for k in WKEYS})
    for gk, (name, arr) in params.items():
        for pos in np.ndindex(arr.shape):
            def J(delta):
                a2 = arr.copy()
                a2[pos] += delta
                uu = a2 if name == "u" else u
                ee = a2 if name == "e" else e
                ww = dict(w, **{name: a2}) if name in WKEYS else w
                return _objective(uu, ee, b, ww, dh, idx, seq, alpha)
            fd = (J(eps) - J(-eps)) / (2 * eps)
            an = g[gk][pos]
            worst = max(worst, abs(an - fd) / max(1.0, abs(an)))
    return worst


def test_gradients_match_finite_differences():
    """Every gradient (tokens, centroids, routed and shared weights), with the
    group limit and the balance loss on, against central differences."""
    assert _fd_mismatch(seed=0) < 1e-7
    assert _fd_mismatch(seed=1, seq=None, alpha=0.0) < 1e-7


def test_forward64_agrees_with_the_forward_oracle():
    sh = SHAPE
    u, e, b, w, dh = _inputs(2)
    u32, e32 = u.astype(np.float32), e.astype(np.float32)
    w32 = {k: v.astype(np.float32) for k, v in w.items()}
    ref = oracle.moe_forward(u32, e32, b, w32, sh["K_r"], sh["G"], sh["M"], sh["N_s"],
                             seq_offsets=SEQ, alpha=ALPHA)
    fw = mb.forward64(u32, e32, b, w32, sh["K_r"], sh["G"], sh["M"], sh["N_s"], SEQ, ALPHA)
    np.testing.assert_array_equal(fw["idx"], ref["idx"])
    np.testing.assert_allclose(fw["h"], ref["h"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(fw["bal_mean"], ref["seq_stat_mean"], rtol=1e-6)


def test_silu_grad_matches_finite_differences():
    a = np.linspace(-8.0, 8.0, 161)
    fd = (oracle.silu(a + 1e-6) - oracle.silu(a - 1e-6)) / 2e-6
    np.testing.assert_allclose(mb.silu_grad(a), fd, rtol=1e-8, atol=1e-9)
    assert mb.silu_grad(0.0) == 0.5


def test_gate_gradient_is_scale_free():
    """g = s_sel / sum(s_sel) does not change when the selected s scale together, so
    sum over the selected experts of s * ds vanishes for any upstream dg."""
    rng = np.random.default_rng(3)
    s = rng.uniform(0.05, 0.95, (7, 9))
    idx = np.stack([rng.choice(9, 3, replace=False) for _ in range(7)])
    ds = mb.gate_backward(s, idx, rng.standard_normal((7, 3)))
    for t in range(7):
        mask = np.zeros(9, bool)
        mask[idx[t]] = True
        assert (ds[t, ~mask] == 0).all()
        assert abs(np.dot(s[t, mask], ds[t, mask])) < 1e-12


def test_balance_gradient_is_scale_free():
    """P uses s normalised over all experts of the token, so sum_j s_j ds_j = 0 per token."""
    rng = np.random.default_rng(4)
    s = rng.uniform(0.05, 0.95, (8, 6))
    idx = np.stack([rng.choice(6, 2, replace=False) for _ in range(8)])
    ds = mb.balance_backward(s, idx, np.array([0, 5, 8]), 2, 0.7)
    np.testing.assert_allclose((s * ds).sum(axis=1), 0.0, atol=1e-13)
    assert np.abs(ds).max() > 1e-3


def test_zero_experts_pass_the_gradient_straight():
    """All expert weights zero: h' = u, so du = dh and every other gradient is zero
    (the experts output 0, the gates see dg = 0; no balance loss)."""
    sh = SHAPE
    u, e, b, w, dh = _inputs(5)
    w = {k: np.zeros_like(v) for k, v in w.items()}
    g = mb.layer_backward(u, e, b, w, dh, sh["K_r"], sh["G"], sh["M"], sh["N_s"])
    np.testing.assert_array_equal(g["du"], dh)
    assert not g["de"].any()
    for k in WKEYS:
        assert not g[k].any()


def test_single_expert_gate_has_no_gradient():
    """With one routed expert the gate is identically 1: the centroid gets no gradient."""
    u, e, b, w, dh = _inputs(6, N_r=1, K_r=1, G=1, M=1)
    g = mb.layer_backward(u, e, b, w, dh, 1, 1, 1, 1)
    assert not g["de"].any()


def test_bias_gets_no_gradient():
    """b only decides the selection: at a fixed selection h' does not depend on it."""
    sh = SHAPE
    u, e, b, w, dh = _inputs(7)
    fw = mb.forward64(u, e, b, w, sh["K_r"], sh["G"], sh["M"], sh["N_s"])
    fw2 = mb.forward64(u, e, b + np.float32(0.5), w, sh["K_r"], sh["G"], sh["M"], sh["N_s"],
                       idx=fw["idx"])
    np.testing.assert_array_equal(fw["h"], fw2["h"])
    g = mb.layer_backward(u, e, b, w, dh, sh["K_r"], sh["G"], sh["M"], sh["N_s"])
    assert g["db"].shape == b.shape and not g["db"].any()


def _bad_gate_backward(s, idx, dgate):
    """Mistake: drops the normalisation's coupling term (- sum_k g_k dg_k)."""
    s = np.asarray(s, np.float64)
    ds = np.zeros_like(s)
    for t in range(s.shape[0]):
        S = s[t, idx[t]].sum()
        for j, i in enumerate(idx[t]):
            ds[t, i] += dgate[t, j] / S
    return ds


def _bad_silu_grad(a):
    """Mistake: sigma(a) in place of silu'(a)."""
    return mb.sigmoid64(a)


def _bad_balance_backward(s, idx, seq_offsets, K_r, alpha):
    """Mistake: treats R_t = sum_j s_{j,t} as a constant (drops the coupling term
    - sum_i f_i s_{i,t} / R_t of the normalisation)."""
    s = np.asarray(s, np.float64)
    off = np.asarray(seq_offsets, np.int64)
    N_r, n_seq = s.shape[1], len(off) - 1
    ds = np.zeros_like(s)
    for j in range(n_seq):
        a, z = off[j], off[j + 1]
        counts = np.bincount(np.asarray(idx[a:z]).reshape(-1), minlength=N_r).astype(float)
        f = counts * (N_r / (K_r * (z - a)))
        for t in range(a, z):
            ds[t] += (alpha / n_seq) * f / ((z - a) * s[t].sum())
    return ds


_good_ffn_backward = mb.expert_ffn_backward


def _bad_ffn_backward(x, w_gate, w_up, w_down, dy):
    """Mistake: the gate and up weight gradients swapped."""
    dx, dwg, dwu, dwd = _good_ffn_backward(x, w_gate, w_up, w_down, dy)
    return dx, dwu, dwg, dwd


@pytest.mark.parametrize("name,bad", [
    ("gate_backward", _bad_gate_backward),
    ("silu_grad", _bad_silu_grad),
    ("balance_backward", _bad_balance_backward),
    ("expert_ffn_backward", _bad_ffn_backward),
])
def test_planted_backward_mistakes_are_caught(monkeypatch, name, bad):
    monkeypatch.setattr(mb, name, bad)
    assert _fd_mismatch(seed=0) > 1e-4
