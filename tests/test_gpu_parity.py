"""GPU parity of the whole path against the CPU oracle (marked gpu).

Sizes: the tiny fp32 layer and the mid bf16 layer are compared element by element;
the DeepSeek-V3-shaped layer is compared at full size: routing, dispatch and the bias
update on every token, h' on 66 sampled tokens, and the expert GEMMs' output on every
row of four whole segments (largest, smallest, one of 257-512 rows, the shared
expert); a 65536-token batch at the mid sizes is compared the same way on sampled
tokens.  Edge cases: ragged token counts and hidden sizes that are not tile multiples,
an empty batch, a single token, experts with no tokens and an expert with every token.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import aux_loss_free_router_b300 as moe
from tests.layer_harness import (check_affinity, check_output_full, check_output_sampled,
                                 check_routing, check_seq_stat, rel_l2, run_layer, to_np)

pytestmark = pytest.mark.gpu

# bf16 layer outputs: 2e-2 max-abs and 1e-2 relative L2 against the float64 oracle
BF16_ABS, BF16_REL = 2e-2, 1e-2


def test_tiny_fp32_layer_matches_oracle():
    cfg = synth.config("tiny")
    r = run_layer(cfg)
    check_affinity(cfg, r, atol=2e-6)
    idx, _ = check_routing(cfg, r)
    check_seq_stat(cfg, r, idx)
    check_output_full(cfg, r, rel_tol=1e-5)


def test_mid_bf16_layer_matches_oracle():
    cfg = synth.config("mid")
    r = run_layer(cfg)
    check_affinity(cfg, r, atol=2e-5)
    idx, _ = check_routing(cfg, r)
    check_seq_stat(cfg, r, idx)
    check_output_full(cfg, r, rel_tol=BF16_REL, abs_tol=BF16_ABS)


def test_v3_layer_full_size_sampled():
    cfg = synth.config("v3")
    r = run_layer(cfg)
    # affinities on a token sample (the oracle's float64 GEMM over all tokens is slow)
    x = r["inputs"]
    sample = np.random.default_rng(0).choice(cfg.T, 64, replace=False)
    sample = np.concatenate([sample, [0, cfg.T - 1]])
    s_ref = oracle.affinity(to_np(x["u"][torch.as_tensor(sample, device="cuda")]), to_np(x["e"]))
    assert np.abs(r["s_out"][sample] - s_ref).max() <= 5e-5
    idx, _ = check_routing(cfg, r)
    per = cfg.N_r // cfg.G
    assert max(len(set((row // per).tolist())) for row in r["topk_idx"]) <= cfg.M
    check_seq_stat(cfg, r, idx)
    check_output_sampled(cfg, r, sample, BF16_REL, BF16_ABS)
    check_segments_full(cfg, r)


def test_largest_batch_sampled():
    """65536 tokens in 8 sequences at the mid layer's sizes (d=2048, 64 experts top-6, 2
    shared, I=1408): 512 router clusters, about 6 k rows per expert segment (24 token
    tiles of gate/up, 12 of down), 393 k rows in the FFN row space.  Routing, dispatch,
    the bias update and the statistic on every token; h' on 66 sampled tokens."""
    cfg = synth.MoEConfig("large", T=65536, d=2048, N_r=64, K_r=6, N_s=2, I=1408, n_seq=8,
                          dtype="bf16", bias="uniform", seed=11)
    r = run_layer(cfg)
    idx, _ = check_routing(cfg, r)
    check_seq_stat(cfg, r, idx)
    sample = np.random.default_rng(1).choice(cfg.T, 64, replace=False)
    sample = np.concatenate([sample, [0, cfg.T - 1]])
    check_output_sampled(cfg, r, sample, BF16_REL, BF16_ABS)


def check_segments_full(cfg, r):
    """Every row of the expert GEMMs' output y for four segments of the V3-shaped
    batch: the largest routed segment, the smallest non-empty one, one of 257-512 rows
    (two token tiles sharing each weight slab) and the shared expert (all T tokens),
    each against the oracle's FFN on the same token rows (K = 7168 and I = 2048 loop
    counts, every gate/up feature tile, every down output tile)."""
    x, lay = r["inputs"], r["layer"]
    off, perm, load = r["expert_offset"], r["perm_token"], r["load"]
    nonempty = np.nonzero(load > 0)[0]
    picks = {"largest": int(np.argmax(load)),
             "smallest": int(nonempty[np.argmin(load[nonempty])])}
    mid = np.nonzero((load > 256) & (load <= 512))[0]
    assert len(mid) > 0
    picks["257-512 rows"] = int(mid[0])
    dev = x["u"].device
    for name, i in picks.items():
        rows = slice(int(off[i]), int(off[i + 1]))
        tok = torch.as_tensor(perm[rows].astype(np.int64), device=dev)
        ref = oracle.expert_ffn(to_np(x["u"][tok]), *(to_np(x[k][i]) for k in ("w_gate", "w_up", "w_down")))
        got = to_np(lay.y[rows])
        err, mx = rel_l2(got, ref), np.abs(got - ref).max()
        assert err <= BF16_REL and mx <= BF16_ABS, (name, i, int(load[i]), err, mx)
    R0 = cfg.T * cfg.K_r
    for j in range(cfg.N_s):
        ref = oracle.expert_ffn(to_np(x["u"]), *(to_np(x[k][j]) for k in ("ws_gate", "ws_up", "ws_down")))
        got = to_np(lay.y[R0 + j * cfg.T:R0 + (j + 1) * cfg.T])
        err, mx = rel_l2(got, ref), np.abs(got - ref).max()
        assert err <= BF16_REL and mx <= BF16_ABS, ("shared", j, err, mx)


def test_routing_with_own_scores_differs_only_at_near_ties():
    """Full oracle routing (its own float64-derived s) against the library's: any
    disagreement must sit where the competing keys are closer than the affinity
    error bound."""
    cfg = synth.config("mid", T=1024, n_seq=1)
    r = run_layer(cfg)
    x = r["inputs"]
    s_ref = oracle.affinity(to_np(x["u"]), to_np(x["e"]))
    b = to_np(r["b0"])
    idx_ref = oracle.select_experts(s_ref, b, cfg.K_r)
    keys = oracle.routing_keys(s_ref, b).astype(np.float64)
    bad = np.nonzero((np.sort(idx_ref, 1) != np.sort(r["topk_idx"], 1)).any(1))[0]
    for t in bad:
        kth = np.sort(keys[t])[::-1]
        gap = kth[cfg.K_r - 1] - kth[cfg.K_r]
        assert gap <= 4e-5, (t, gap)
    assert len(bad) <= cfg.T // 100


@pytest.mark.parametrize("T,d,I,N_r,K_r,G,M,N_s", [
    (300, 320, 200, 32, 4, 4, 2, 1),     # ragged T, d not a multiple of 64, I not of 128
    (1, 256, 128, 64, 6, 1, 1, 2),       # a single token
    (129, 512, 384, 64, 8, 8, 4, 0),     # no shared expert, group limit
    (257, 1024, 256, 128, 8, 8, 2, 1),
])
def test_ragged_bf16_layers(T, d, I, N_r, K_r, G, M, N_s):
    cfg = synth.MoEConfig("ragged", T=T, d=d, N_r=N_r, K_r=K_r, N_s=N_s, I=I, G=G, M=M,
                          dtype="bf16", bias="uniform", seed=T)
    r = run_layer(cfg)
    check_affinity(cfg, r, atol=2e-5)
    idx, _ = check_routing(cfg, r)
    check_seq_stat(cfg, r, idx)
    check_output_full(cfg, r, rel_tol=BF16_REL, abs_tol=BF16_ABS)


@pytest.mark.parametrize("T,d,I,N_r,K_r,G,M,N_s", [
    (100, 64, 64, 1, 1, 1, 1, 1),         # one routed expert: every token picks it
    (96, 128, 64, 256, 32, 1, 1, 0),      # the largest K_r: 32 of 256 experts
    (64, 128, 64, 256, 32, 32, 32, 1),    # 32 groups of 8 experts, all kept, one key each
])
def test_extreme_bf16_shapes(T, d, I, N_r, K_r, G, M, N_s):
    cfg = synth.MoEConfig("extreme", T=T, d=d, N_r=N_r, K_r=K_r, N_s=N_s, I=I, G=G, M=M,
                          dtype="bf16", bias="uniform", seed=T + N_r)
    r = run_layer(cfg)
    idx, _ = check_routing(cfg, r)
    check_seq_stat(cfg, r, idx)
    check_output_full(cfg, r, rel_tol=BF16_REL, abs_tol=BF16_ABS)


@pytest.mark.parametrize("T,d,I,N_r,K_r,N_s", [
    (150, 264, 200, 16, 3, 1),   # K steps and output tiles that end part-way
    (77, 136, 72, 24, 4, 2),
])
def test_ragged_fp32_layers(T, d, I, N_r, K_r, N_s):
    cfg = synth.MoEConfig("ragged-f32", T=T, d=d, N_r=N_r, K_r=K_r, N_s=N_s, I=I, G=1, M=1,
                          dtype="f32", bias="uniform", seed=T + 2)
    r = run_layer(cfg)
    idx, _ = check_routing(cfg, r)
    check_seq_stat(cfg, r, idx)
    check_output_full(cfg, r, rel_tol=1e-5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_empty_and_concentrated_experts(dtype):
    # a bias of +1 on experts 0..K_r-1 sends every token there: the other experts get
    # zero rows and the chosen ones all T rows
    cfg = synth.MoEConfig("skewed", T=200, d=256, N_r=32, K_r=2, N_s=1, I=128,
                          dtype=dtype, bias="zero", seed=3)
    x = synth.make_inputs(cfg, device="cuda")
    x["b"][:2] = 1.0
    r = run_layer(cfg, x)
    assert r["load"][:2].tolist() == [200, 200] and (r["load"][2:] == 0).all()
    idx, _ = check_routing(cfg, r)
    check_output_full(cfg, r, rel_tol=1e-5 if dtype == "f32" else BF16_REL)
    # overloaded experts move down by gamma, the idle ones up
    assert (r["b_new"][:2] < to_np(r["b0"])[:2]).all() and (r["b_new"][2:] > 0).all()


def test_empty_batch():
    cfg = synth.MoEConfig("empty", T=0, d=256, N_r=16, K_r=2, N_s=1, I=128, dtype="bf16")
    sh = moe.make_shape(0, 256, 16, 2, 1, 128)
    dev = "cuda"
    e = torch.randn(16, 256, device=dev).bfloat16()
    b = torch.zeros(16, device=dev)
    idx = torch.empty(0, 2, dtype=torch.int32, device=dev)
    gate = torch.empty(0, 2, device=dev)
    load = torch.full((16,), 7, dtype=torch.int32, device=dev)
    off = torch.full((17,), 7, dtype=torch.int32, device=dev)
    u = torch.empty(0, 256, device=dev).bfloat16()
    moe.route(u, e, b, sh, idx, gate)
    moe.dispatch(idx, sh, load, off, torch.empty(0, dtype=torch.int32, device=dev),
                 torch.empty(0, 2, dtype=torch.int32, device=dev))
    moe.bias_update(b, load, sh, 0.001)
    torch.cuda.synchronize()
    assert (load == 0).all() and (off == 0).all()
    assert (b == 0).all()        # zero load equals the zero mean: no change


def test_layer_is_deterministic():
    cfg = synth.config("mid", T=1024, n_seq=2)
    x = synth.make_inputs(cfg, device="cuda")
    r1 = run_layer(cfg, {k: v.clone() for k, v in x.items()})
    r2 = run_layer(cfg, {k: v.clone() for k, v in x.items()})
    for k in ("h", "topk_idx", "topk_gate", "perm_token", "inv_row", "stat", "b_new"):
        np.testing.assert_array_equal(r1[k], r2[k], err_msg=k)


def test_layer_reading_rows_from_u_is_bit_identical():
    """MoELayer(gather_rows=True): gate/up reads the routed rows straight from u and the
    dispatch writes no x_perm.  h' equals the default layer's bit for bit, and backward()
    (which then gathers x_perm itself) gives the same gradients."""
    cfg = synth.config("mid", T=512, n_seq=2)
    x = synth.make_inputs(cfg, device="cuda")
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    outs = []
    for gather in (False, True):
        lay = moe.MoELayer(T=cfg.T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I,
                           G=cfg.G, M=cfg.M, e=x["e"], b=x["b"].clone(), weights=w,
                           n_seq=cfg.n_seq, alpha=cfg.alpha, want_s=True, gather_rows=gather)
        h = lay.step(x["u"], x["seq_offsets"], update_bias=False).clone()
        g = torch.Generator(device="cuda").manual_seed(3)
        dh = torch.randn(cfg.T, cfg.d, generator=g, device="cuda")
        grads = {k: v.clone() for k, v in lay.backward(x["u"], dh, x["seq_offsets"]).items()}
        torch.cuda.synchronize()
        assert moe.device_error() == 0
        outs.append((h, grads))
    assert torch.equal(outs[0][0], outs[1][0])
    for k in outs[0][1]:
        assert torch.equal(outs[0][1][k], outs[1][1][k]), k


def test_gathered_rows_are_token_rows():
    """The dispatch's row gather writes x_perm = u[perm_token]."""
    cfg = synth.config("mid", T=512, n_seq=1)
    r = run_layer(cfg)
    layer, u = r["layer"], r["inputs"]["u"]
    xp = torch.empty_like(layer.x_perm)
    moe.dispatch(layer.topk_idx, layer.shape, layer.load, layer.expert_offset, layer.perm_token,
                 layer.inv_row, u, xp)
    torch.cuda.synchronize()
    assert torch.equal(xp, u[layer.perm_token.long()])


def test_bias_update_moves_toward_balance_over_steps():
    cfg = synth.config("skew", T=1024, n_seq=1)
    x = synth.make_inputs(cfg, device="cuda")
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    layer = moe.MoELayer(T=cfg.T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I,
                         G=1, M=1, e=x["e"], b=x["b"].clone(), weights=w, n_seq=1,
                         gamma=0.01)
    ratios = []
    for step in range(40):
        u = synth.make_inputs(cfg, device="cuda", u_seed=1000 + step, with_weights=False)["u"]
        b_before = layer.b.clone()
        layer.step(u, x["seq_offsets"])
        load = layer.load.clone()
        torch.cuda.synchronize()
        ref = oracle.bias_update(to_np(b_before), to_np(load), cfg.T, cfg.K_r, 0.01)
        np.testing.assert_array_equal(to_np(layer.b), ref)
        ratios.append(load.max().item() / (cfg.T * cfg.K_r / cfg.N_r))
    assert np.mean(ratios[-5:]) < np.mean(ratios[:5])


def test_skewed_balance_run_200_steps():
    """The skewed workload: 200 steps of forward + load count + bias update with
    gamma = 0.001 on Gaussian-mixture tokens.  Every step's update equals the oracle's
    update of that step's loads, routing is bit-exact at sampled steps, and the
    imbalance falls."""
    cfg = synth.config("skew")
    x = synth.make_inputs(cfg, device="cuda")
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    layer = moe.MoELayer(T=cfg.T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I,
                         G=1, M=1, e=x["e"], b=x["b"].clone(), weights=w, n_seq=cfg.n_seq,
                         gamma=cfg.gamma, want_s=True)
    mean = cfg.T * cfg.K_r / cfg.N_r
    ratios = []
    for step in range(200):
        u = synth.make_inputs(cfg, device="cuda", u_seed=1000 + step, with_weights=False)["u"]
        b_before = to_np(layer.b)
        layer.step(u, x["seq_offsets"])
        torch.cuda.synchronize()
        load = to_np(layer.load)
        np.testing.assert_array_equal(
            to_np(layer.b), oracle.bias_update(b_before, load, cfg.T, cfg.K_r, cfg.gamma))
        if step in (0, 99, 199):
            idx = oracle.select_experts(to_np(layer.s_out), b_before, cfg.K_r)
            np.testing.assert_array_equal(to_np(layer.topk_idx), idx)
        ratios.append(load.max() / mean)
    assert ratios[0] > 1.5                     # the mixture does skew the routing
    assert np.mean(ratios[-20:]) < np.mean(ratios[:20])


def test_decode_sized_pass():
    """The decode-sized batch (128 mixture tokens through the skewed workload's layer):
    routing bit-exact, h' within 1e-2 relative L2, and its max-abs error reported."""
    cfg = synth.config("skew", T=128, n_seq=1)
    r = run_layer(cfg)
    idx, _ = check_routing(cfg, r)
    ref = check_output_full(cfg, r, rel_tol=BF16_REL)
    mx = float(np.abs(r["h"] - ref["h"]).max())
    rms = float(np.sqrt(np.mean(ref["h"] ** 2)))
    print(f"decode pass: max-abs error {mx:.4g}, RMS(h') {rms:.4g}, "
          f"rel L2 {rel_l2(r['h'], ref['h']):.3g}")
    assert mx <= BF16_ABS * max(1.0, rms), mx


def test_pipelined_host_batches_match_steps():
    """MoELayer.pipeline (copies overlapped with compute on three streams) gives, batch
    by batch, exactly what step() gives on the same batches in the same order."""
    cfg = synth.config("mid", T=512, n_seq=2)
    x = synth.make_inputs(cfg, device="cuda")
    w = {k: x[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")}
    batches = [synth.make_inputs(cfg, device="cuda", u_seed=50 + k, with_weights=False)["u"]
               for k in range(5)]

    def layer():
        return moe.MoELayer(T=cfg.T, d=cfg.d, N_r=cfg.N_r, K_r=cfg.K_r, N_s=cfg.N_s, I=cfg.I,
                            G=cfg.G, M=cfg.M, e=x["e"], b=x["b"].clone(), weights=w,
                            n_seq=cfg.n_seq, gamma=0.01)

    ref = layer()
    want, want_load = [], []
    for u in batches:
        want.append(ref.step(u, x["seq_offsets"]).clone())
        want_load.append(ref.load.clone())
    lay = layer()
    u_host = [u.cpu().pin_memory() for u in batches]
    out_host = [torch.empty(lay.out.shape, dtype=lay.out.dtype).pin_memory() for _ in batches]
    load_host = [torch.empty(cfg.N_r, dtype=torch.int32).pin_memory() for _ in batches]
    lay.pipeline(u_host, out_host, x["seq_offsets"], load_host)
    torch.cuda.synchronize()
    for k in range(len(batches)):
        assert torch.equal(out_host[k], want[k].cpu()), k
        assert torch.equal(load_host[k], want_load[k].cpu()), k
    assert torch.equal(lay.b, ref.b)


def test_sequence_statistic_with_many_short_sequences():
    """64 sequences of 16 tokens (shorter than a P-sum window, many per window)."""
    cfg = synth.config("mid", T=1024, n_seq=64)
    r = run_layer(cfg)
    idx, _ = check_routing(cfg, r)
    check_seq_stat(cfg, r, idx)
