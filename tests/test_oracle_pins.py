"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU.  Each test checks the oracle against something other than itself: values
worked out by hand from the pages' definitions (tests/golden/*.json), closed forms,
brute-force enumeration on tiny inputs, invariants the pages state in words, and
special cases that reduce to a library routine.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import fp8 as ofp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ worked examples --

def test_golden_bias_routing():
    g = golden("routing_bias.json")
    s, b = np.array(g["s"], np.float32), np.array(g["b"], np.float32)
    idx = oracle.select_experts(s, b, g["K_r"])
    assert idx.tolist() == g["idx"]
    np.testing.assert_allclose(oracle.gate_values(s, idx), g["gate"], rtol=1e-7)
    idx0 = oracle.select_experts(s, np.zeros_like(b), g["K_r"])
    assert idx0.tolist() == g["idx_b0"]
    np.testing.assert_allclose(oracle.gate_values(s, idx0), g["gate_b0"], rtol=1e-7)


def test_golden_group_routing():
    g = golden("routing_groups.json")
    s, b = np.array(g["s"], np.float32), np.array(g["b"], np.float32)
    keys = oracle.routing_keys(s, b)[0]
    assert [float(x) for x in oracle.group_scores(keys, g["G"], g["M"], g["K_r"])] \
        == g["group_scores"]
    assert oracle.select_experts(s, b, g["K_r"], g["G"], g["M"]).tolist() == g["idx"]
    assert oracle.select_experts(s, b, g["K_r"]).tolist() == g["idx_ungrouped"]


def test_golden_bias_update():
    g = golden("bias_update.json")
    out = oracle.bias_update(np.array(g["b"], np.float32), np.array(g["load"]),
                             g["T"], g["K_r"], g["gamma"])
    assert out.dtype == np.float32
    np.testing.assert_array_equal(out, np.array(g["b_new"], np.float32))


def test_golden_seq_stat():
    g = golden("seq_stat.json")
    st, mean = oracle.seq_balance_stat(np.array(g["s"], np.float32), np.array(g["idx"]),
                                       g["seq_offsets"], g["N_r"], g["K_r"], g["alpha"])
    np.testing.assert_allclose(st, g["stat"], rtol=1e-12)
    assert mean == pytest.approx(g["stat"][0], rel=1e-12)


def test_golden_ffn_single_token():
    g = golden("ffn_single_token.json")
    u = np.array(g["u"])
    wg, wu, wd = (np.array(g[k]) for k in ("w_gate", "w_up", "w_down"))
    h = oracle.layer_output(u, np.array([[0]]), np.array([[1.0]]),
                            lambda i: (wg, wu, wd),
                            [(np.zeros_like(wg), np.zeros_like(wu), np.zeros_like(wd))])
    np.testing.assert_allclose(h, g["h"], rtol=1e-14)


# ------------------------------------------------------------- closed forms ----

def test_affinity_closed_forms():
    rng = np.random.default_rng(1)
    d = 16
    u = rng.standard_normal((3, d))
    # e_i chosen so that u_0 . e_i is exactly a chosen logit z_i.
    z = np.array([0.0, math.log(3.0), -math.log(3.0), 2.0])
    e = np.stack([zi * u[0] / np.dot(u[0], u[0]) for zi in z])
    s = oracle.affinity(u, e)
    want = np.array([0.5, 0.75, 0.25, 1.0 / (1.0 + math.exp(-2.0))], np.float32)
    np.testing.assert_allclose(s[0], want, rtol=2e-7)
    # u = 0 gives sigmoid(0) = 1/2 for every expert.
    assert (oracle.affinity(np.zeros((2, d)), rng.standard_normal((5, d))) == 0.5).all()


def test_routing_keys_single_fp32_rounding():
    s = np.array([[np.float32(0.1), np.float32(0.3)]], np.float32)
    b = np.array([np.float32(0.2), np.float32(-0.1)], np.float32)
    k = oracle.routing_keys(s, b)
    assert k.dtype == np.float32
    # The fp32 sum of two fp32 values is the correctly rounded exact sum.
    exact = np.float64(s[0, 0]) + np.float64(b[0])
    assert k[0, 0] == np.float32(exact)


# -------------------------------------------------------------- brute force ----

def _dominates(keys, S):
    """S is the Top-K set under 'larger key first, ties to the lower index' iff every
    member beats every non-member."""
    out = [j for j in range(len(keys)) if j not in S]
    return all(keys[i] > keys[j] or (keys[i] == keys[j] and i < j)
               for i in S for j in out)


@pytest.mark.parametrize("N_r,K_r", [(4, 1), (5, 2), (6, 3), (8, 2), (8, 5)])
def test_topk_brute_force(N_r, K_r):
    rng = np.random.default_rng(N_r * 10 + K_r)
    for _ in range(60):
        # coarse grid -> many exact ties
        s = (rng.integers(0, 6, size=(1, N_r)) / 8.0).astype(np.float32)
        b = (rng.integers(-2, 3, size=N_r) / 16.0).astype(np.float32)
        keys = (s[0] + b).astype(np.float32)
        winners = [S for S in itertools.combinations(range(N_r), K_r)
                   if _dominates(keys, set(S))]
        assert len(winners) == 1
        idx = oracle.select_experts(s, b, K_r)[0]
        assert sorted(idx.tolist()) == list(winners[0])
        # descending key order, ties to the lower index
        for a, c in zip(idx[:-1], idx[1:]):
            assert keys[a] > keys[c] or (keys[a] == keys[c] and a < c)


@pytest.mark.parametrize("N_r,G,M,K_r", [(8, 4, 2, 2), (8, 4, 2, 4), (12, 3, 1, 2),
                                         (12, 4, 3, 3), (12, 6, 2, 4)])
def test_group_limited_brute_force(N_r, G, M, K_r):
    rng = np.random.default_rng(N_r + G * 7 + M * 13 + K_r)
    per, kg = N_r // G, K_r // M
    for _ in range(40):
        s = (rng.integers(0, 5, size=(1, N_r)) / 8.0).astype(np.float32)
        b = (rng.integers(-1, 2, size=N_r) / 16.0).astype(np.float32)
        keys = (s[0] + b).astype(np.float32)
        # group score: sum of the kg largest member keys (all values on a 1/16 grid,
        # so every partial sum is exact and the order of summation is irrelevant)
        gsc = [float(np.sort(keys[g * per:(g + 1) * per])[::-1][:kg].sum())
               for g in range(G)]
        win_g = [S for S in itertools.combinations(range(G), M) if _dominates(gsc, set(S))]
        assert len(win_g) == 1
        eligible = [i for i in range(N_r) if i // per in win_g[0]]
        masked = np.where(np.isin(np.arange(N_r), eligible), keys, -np.inf)
        win = [S for S in itertools.combinations(eligible, K_r) if _dominates(masked, set(S))]
        assert len(win) == 1
        idx = oracle.select_experts(s, b, K_r, G, M)[0]
        assert sorted(idx.tolist()) == list(win[0])
        assert len({i // per for i in idx}) <= M


# ---------------------------------------------------------------- invariants ---

def _rand_route(T=50, N_r=16, K_r=4, G=1, M=1, seed=0):
    rng = np.random.default_rng(seed)
    s = (1 / (1 + np.exp(-rng.standard_normal((T, N_r))))).astype(np.float32)
    b = rng.uniform(-0.05, 0.05, N_r).astype(np.float32)
    return s, b, oracle.select_experts(s, b, K_r, G, M)


def test_gates_sum_to_one_over_exactly_K_r_distinct():
    s, b, idx = _rand_route(K_r=6)
    g = oracle.gate_values(s, idx)
    assert all(len(set(r)) == 6 for r in idx.tolist())
    np.testing.assert_allclose(g.astype(np.float64).sum(1), 1.0, atol=1e-6)
    assert (g > 0).all()


def test_bias_changes_selection_not_gate_values():
    s, b, idx = _rand_route(T=200, K_r=3, seed=3)
    # A bias that changes the selection: gates are still the raw s renormalised.
    g = oracle.gate_values(s, idx)
    sel = np.take_along_axis(s.astype(np.float64), idx.astype(np.int64), 1)
    np.testing.assert_allclose(g, sel / sel.sum(1, keepdims=True), rtol=1e-7)
    # Two biases giving the same selection give identical gates.
    b2 = (b + np.float32(0.5)).astype(np.float32)
    idx2 = oracle.select_experts(s, b2, 3)
    same = (np.sort(idx, 1) == np.sort(idx2, 1)).all(1)
    assert same.mean() > 0.9
    g2 = oracle.gate_values(s, idx2)
    np.testing.assert_array_equal(np.sort(g[same], 1), np.sort(g2[same], 1))
    # and the bias did change some selections relative to b = 0
    idx0 = oracle.select_experts(s, np.zeros_like(b), 3)
    assert (np.sort(idx0, 1) != np.sort(idx, 1)).any()


def test_zero_bias_is_plain_sigmoid_topk():
    rng = np.random.default_rng(5)
    u = rng.standard_normal((40, 32))
    e = rng.standard_normal((16, 32)) / math.sqrt(32)
    s = oracle.affinity(u, e)
    idx = oracle.select_experts(s, np.zeros(16, np.float32), 4)
    ref = np.argsort(-s, axis=1, kind="stable")[:, :4]   # library sort, stable ties
    np.testing.assert_array_equal(idx, ref)


@pytest.mark.parametrize("G,M", [(1, 1), (4, 4)])
def test_group_limit_degenerate_cases_match_ungrouped(G, M):
    s, b, idx = _rand_route(N_r=16, K_r=4, seed=11)
    np.testing.assert_array_equal(oracle.select_experts(s, b, 4, G, M), idx)


def test_group_limit_touches_at_most_M_groups():
    s, b, idx = _rand_route(T=300, N_r=32, K_r=8, G=8, M=4, seed=2)
    per = 4
    assert max(len(set((r // per).tolist())) for r in idx) <= 4
    s, b, idx = _rand_route(T=300, N_r=32, K_r=4, G=8, M=2, seed=4)
    assert max(len(set((r // per).tolist())) for r in idx) <= 2


def test_dispatch_invariants():
    s, b, idx = _rand_route(T=123, N_r=16, K_r=4, seed=9)
    dp = oracle.dispatch(idx, 16)
    load, off, perm, inv = dp["load"], dp["offset"], dp["perm_token"], dp["inv_row"]
    assert load.sum() == 123 * 4
    np.testing.assert_array_equal(load, np.bincount(idx.reshape(-1), minlength=16))
    assert off[0] == 0 and off[-1] == 123 * 4 and (np.diff(off) == load).all()
    assert sorted(perm.tolist()) == sorted(np.repeat(np.arange(123), 4).tolist())
    for i in range(16):
        seg = perm[off[i]:off[i + 1]]
        assert (np.diff(seg) > 0).all()                     # ascending t, no repeats
        assert all(i in idx[t] for t in seg)
    for t in range(123):
        for k in range(4):
            r = inv[t, k]
            assert perm[r] == t and off[idx[t, k]] <= r < off[idx[t, k] + 1]


def test_bias_update_steps_are_plus_minus_gamma_or_zero():
    rng = np.random.default_rng(0)
    T, K_r, N_r, gamma = 96, 6, 64, 0.001
    b = rng.uniform(-0.01, 0.01, N_r).astype(np.float32)
    load = rng.multinomial(T * K_r, np.ones(N_r) / N_r)
    load[0] = T * K_r // N_r                                # exactly at the mean
    nb = oracle.bias_update(b, load, T, K_r, gamma)
    d = nb.astype(np.float64) - b.astype(np.float64)
    mean = T * K_r / N_r
    for i in range(N_r):
        want = -gamma if load[i] > mean else (gamma if load[i] < mean else 0.0)
        assert d[i] == pytest.approx(want, abs=2e-9)
    assert nb[0] == b[0]


def test_seq_stat_uniform_closed_form_and_sums():
    # Every expert with equal affinity and exactly equal counts -> f_i = 1,
    # P_i = 1/N_r, so sum_i f_i P_i = 1 and the statistic is alpha.
    N_r, K_r, T = 8, 2, 16
    s = np.full((T, N_r), 0.3, np.float32)
    idx = np.array([[(2 * t) % N_r, (2 * t + 1) % N_r] for t in range(T)])
    st, mean = oracle.seq_balance_stat(s, idx, [0, 8, 16], N_r, K_r, 1e-4)
    np.testing.assert_allclose(st, [1e-4, 1e-4], rtol=1e-12)
    # sum_i P_i = 1 per sequence and sum_i f_i = N_r
    s2, b2, idx2 = _rand_route(T=40, N_r=16, K_r=4, seed=8)
    ps = oracle.seq_p_sums(s2, [0, 25, 40])
    np.testing.assert_allclose(ps.sum(1), [25, 15], rtol=1e-12)
    counts = np.bincount(idx2[:25].reshape(-1), minlength=16)
    assert (counts * (16 / (4 * 25))).sum() == pytest.approx(16)


# ------------------------------------------------------------------ layer ------

def _weights(rng, E, I, d, scale=1.0):
    # fp32-representable values: the oracle takes stored (fp32 / bf16) weights
    f = lambda a: a.astype(np.float32).astype(np.float64)
    return (f(rng.standard_normal((E, I, d)) * scale / math.sqrt(d)),
            f(rng.standard_normal((E, I, d)) * scale / math.sqrt(d)),
            f(rng.standard_normal((E, d, I)) * scale / math.sqrt(I)))


def test_identical_experts_closed_form():
    # All routed experts equal -> the normalised gates sum to 1 and
    # h' = u + shared(u) + FFN(u), whatever the routing.
    rng = np.random.default_rng(0)
    T, d, I, N_r, K_r = 30, 24, 10, 8, 3
    u = rng.standard_normal((T, d)).astype(np.float32).astype(np.float64)
    e = rng.standard_normal((N_r, d)) / math.sqrt(d)
    wg, wu, wd = _weights(rng, 1, I, d)
    sg, su, sd = _weights(rng, 1, I, d)
    w = {"w_gate": np.repeat(wg, N_r, 0), "w_up": np.repeat(wu, N_r, 0),
         "w_down": np.repeat(wd, N_r, 0), "ws_gate": sg, "ws_up": su, "ws_down": sd}
    out = oracle.moe_forward(u, e, rng.uniform(-.01, .01, N_r).astype(np.float32), w,
                             K_r, N_s=1)

    def ffn(x, a, c, o):
        hid = (x @ a.T) / (1 + np.exp(-(x @ a.T))) * (x @ c.T)
        return hid @ o.T
    want = u + ffn(u, sg[0], su[0], sd[0]) + ffn(u, wg[0], wu[0], wd[0])
    np.testing.assert_allclose(out["h"], want, rtol=1e-6, atol=1e-6)


def test_zero_weights_give_residual():
    rng = np.random.default_rng(1)
    T, d, I, N_r = 10, 16, 8, 4
    u = rng.standard_normal((T, d)).astype(np.float32)
    z = lambda E: (np.zeros((E, I, d)), np.zeros((E, I, d)), np.zeros((E, d, I)))
    wg, wu, wd = z(N_r)
    sg, su, sd = z(2)
    w = dict(w_gate=wg, w_up=wu, w_down=wd, ws_gate=sg, ws_up=su, ws_down=sd)
    out = oracle.moe_forward(u, rng.standard_normal((N_r, d)), np.zeros(N_r, np.float32),
                             w, 2, N_s=2)
    np.testing.assert_array_equal(out["h"], u.astype(np.float64))


def test_single_selected_expert_matches_direct_formula():
    # K_r = 1: the only gate is 1 and h' = u + FFN_idx(u).
    rng = np.random.default_rng(2)
    T, d, I, N_r = 12, 8, 4, 3
    u = rng.standard_normal((T, d)).astype(np.float32).astype(np.float64)
    wg, wu, wd = _weights(rng, N_r, I, d)
    w = dict(w_gate=wg, w_up=wu, w_down=wd, ws_gate=wg[:0], ws_up=wu[:0], ws_down=wd[:0])
    e = rng.standard_normal((N_r, d))
    out = oracle.moe_forward(u, e, np.zeros(N_r, np.float32), w, 1, N_s=0)
    np.testing.assert_allclose(out["gate"], 1.0)
    for t in range(T):
        i = out["idx"][t, 0]
        a = wg[i] @ u[t]
        hid = a / (1 + np.exp(-a)) * (wu[i] @ u[t])
        np.testing.assert_allclose(out["h"][t], u[t] + wd[i] @ hid, rtol=1e-12)


# --------------------------------------------------------------------- FP8 -----

def test_e4m3_matches_torch_cast_in_range():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    finite = codes[(codes & 0x7F) != 0x7F]
    vals = ofp8.e4m3_decode(finite)
    tv = torch.from_numpy(finite.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(vals, tv)
    # round trip of every finite code (both zeros decode to 0, encode back to +0/-0)
    np.testing.assert_array_equal(ofp8.e4m3_encode(vals), finite)
    # grid points, midpoints (ties to even) and random values inside +-448
    grid = np.unique(np.abs(vals))
    mids = (grid[:-1] + grid[1:]) / 2
    rng = np.random.default_rng(0)
    xs = np.concatenate([grid, -grid, mids, -mids, rng.uniform(-448, 448, 20000),
                         rng.standard_normal(20000) * 0.01]).astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(ofp8.e4m3_round(xs), want)


def test_e4m3_saturates():
    np.testing.assert_array_equal(ofp8.e4m3_round([448.0, 463.9, 464.0, 500.0, 1e6, -1e6]),
                                  [448, 448, 448, 448, 448, -448])


def test_quantize_1x128_scale_rule():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 256)).astype(np.float32)
    x[1, :128] = 0.0
    q, sc = ofp8.quantize_1x128(x)
    assert sc.shape == (3, 2) and sc.dtype == np.float32
    assert sc[1, 0] == 1.0 and (q[1, :128] == 0).all()
    amax = np.abs(x.reshape(3, 2, 128)).max(-1)
    np.testing.assert_array_equal(sc[amax > 0], (amax / np.float32(448)).astype(np.float32)[amax > 0])
    # the tile maximum lands on (or next to) the format's largest value
    assert np.abs(q.reshape(3, 2, 128)).max(-1)[amax > 0].min() >= 416
    deq = ofp8.dequantize_1x128(q, sc)
    assert np.abs(deq - x).max() <= np.abs(x).max() * 2 ** -4


def test_quantize_128x128_blocks():
    rng = np.random.default_rng(1)
    w = rng.standard_normal((2, 256, 128)).astype(np.float32)
    q, sc = ofp8.quantize_128x128(w)
    assert sc.shape == (2, 2, 1)
    blk = w[1, 128:, :]
    assert sc[1, 1, 0] == np.float32(np.abs(blk).max() / np.float32(448))
    np.testing.assert_array_equal(q[1, 128:, :], ofp8.e4m3_round((blk / sc[1, 1, 0]).astype(np.float32)))


# ----------------------------------------------------- the FP8 layer composed ----

def _sparse(entries, shape):
    a = np.zeros(shape, np.float32)
    for *ix, v in entries:
        a[tuple(ix)] = v
    return a


def fp8_golden_case():
    g = golden("fp8_layer_single_token.json")
    T, d, I, N_r, N_s = g["T"], g["d"], g["I"], g["N_r"], g["N_s"]
    w = {"w_gate": _sparse(g["w_gate"], (N_r, I, d)), "w_up": _sparse(g["w_up"], (N_r, I, d)),
         "w_down": _sparse(g["w_down"], (N_r, d, I)), "ws_gate": _sparse(g["ws_gate"], (N_s, I, d)),
         "ws_up": _sparse(g["ws_up"], (N_s, I, d)), "ws_down": _sparse(g["ws_down"], (N_s, d, I))}
    u = _sparse(g["u"], (T, d))
    e = _sparse(g["e"], (N_r, d))
    h = _sparse(g["h_nonzero"], (T, d)).astype(np.float64)
    h[0, 0], h[0, 1] = g["h_nonzero"][0][2], g["h_nonzero"][1][2]   # exact float64 values
    return g, u, e, np.array(g["b"], np.float32), w, h


def test_golden_fp8_layer_single_token():
    """The FP8 composition worked by hand: 1x128 token scales, 128x128 weight scales,
    routing on the unquantised u, the dequantised tokens into both the routed and the
    shared expert, and the SwiGLU output re-quantised 1x128 before the down
    projection (xyznot.com reading guide, Key ideas FP8 bullet; Method §2)."""
    g, u, e, b, w, h = fp8_golden_case()
    out = oracle.moe_forward(u, e, b, w, g["K_r"], 1, 1, g["N_s"], fp8=True)
    assert out["idx"].tolist() == g["idx"]
    np.testing.assert_allclose(out["gate"], g["gate"], rtol=0)
    np.testing.assert_allclose(out["s"], g["s"], rtol=1e-7)
    np.testing.assert_allclose(out["h"], h, rtol=1e-12, atol=1e-12)
