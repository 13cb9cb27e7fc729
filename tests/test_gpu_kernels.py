"""Single-call parity at the DeepSeek-V3 layer's full sizes (marked gpu): the router,
the dispatch and the combine on their own, each against the CPU oracle.  These are
also the small, weight-free cases used for detailed kernel profiles."""
import numpy as np
import pytest
import torch

import oracle
import synth
import aux_loss_free_router_b300 as moe
from tests.layer_harness import to_np

pytestmark = pytest.mark.gpu

V3 = synth.config("v3")


def _route(cfg, x, with_stat=True):
    dev = "cuda"
    sh = moe.make_shape(cfg.T, cfg.d, cfg.N_r, cfg.K_r, cfg.N_s, cfg.I, cfg.G, cfg.M)
    idx = torch.empty(cfg.T, cfg.K_r, dtype=torch.int32, device=dev)
    gate = torch.empty(cfg.T, cfg.K_r, dtype=torch.float32, device=dev)
    s = torch.empty(cfg.T, cfg.N_r, dtype=torch.float32, device=dev)
    psum = torch.empty(cfg.n_seq, cfg.N_r, dtype=torch.float32, device=dev) if with_stat else None
    moe.route(x["u"], x["e"], x["b"], sh, idx, gate, s, x["seq_offsets"], cfg.n_seq, psum)
    torch.cuda.synchronize()
    return sh, idx, gate, s, psum


def test_router_v3_shape_bit_exact():
    x = synth.make_inputs(V3, device="cuda", with_weights=False)
    for _ in range(3):                      # repeated launches: same bits every time
        sh, idx, gate, s, psum = _route(V3, x)
    s_np, b = to_np(s), to_np(x["b"])
    idx_ref = oracle.select_experts(s_np, b, V3.K_r, V3.G, V3.M)
    np.testing.assert_array_equal(to_np(idx), idx_ref)
    np.testing.assert_allclose(to_np(gate), oracle.gate_values(s_np, idx_ref), rtol=1e-6)
    np.testing.assert_allclose(to_np(psum), oracle.seq_p_sums(s_np, to_np(x["seq_offsets"])),
                               rtol=1e-5)
    rows = np.random.default_rng(1).choice(V3.T, 64, replace=False)
    s_ref = oracle.affinity(to_np(x["u"][torch.as_tensor(rows, device="cuda")]), to_np(x["e"]))
    assert np.abs(s_np[rows] - s_ref).max() < 5e-5


def test_dispatch_v3_shape_bit_exact():
    rng = np.random.default_rng(0)
    # random distinct experts per token with a skewed popularity
    p = rng.dirichlet(np.ones(V3.N_r) * 0.3)
    idx = np.stack([rng.choice(V3.N_r, V3.K_r, replace=False, p=p) for _ in range(V3.T)])
    dev = "cuda"
    sh = moe.make_shape(V3.T, V3.d, V3.N_r, V3.K_r, V3.N_s, V3.I, V3.G, V3.M)
    t_idx = torch.as_tensor(idx, dtype=torch.int32, device=dev)
    u = synth.make_inputs(V3, device=dev, with_weights=False)["u"]
    load = torch.empty(V3.N_r, dtype=torch.int32, device=dev)
    off = torch.empty(V3.N_r + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(V3.T * V3.K_r, dtype=torch.int32, device=dev)
    inv = torch.empty(V3.T, V3.K_r, dtype=torch.int32, device=dev)
    xp = torch.empty(V3.T * V3.K_r, V3.d, dtype=torch.bfloat16, device=dev)
    moe.dispatch(t_idx, sh, load, off, perm, inv, u, xp)
    torch.cuda.synchronize()
    ref = oracle.dispatch(idx, V3.N_r)
    np.testing.assert_array_equal(to_np(load), ref["load"])
    np.testing.assert_array_equal(to_np(off), ref["offset"])
    np.testing.assert_array_equal(to_np(perm), ref["perm_token"])
    np.testing.assert_array_equal(to_np(inv), ref["inv_row"])
    assert torch.equal(xp, u[perm.long()])


def test_combine_v3_shape_sampled():
    dev = "cuda"
    T, d, K_r, N_s = V3.T, V3.d, V3.K_r, V3.N_s
    g = torch.Generator(device=dev).manual_seed(5)
    u = torch.randn(T, d, device=dev, generator=g).bfloat16()
    R = T * K_r + N_s * T
    y = torch.randn(R, d, device=dev, generator=g).bfloat16()
    gate = torch.rand(T, K_r, device=dev, generator=g)
    gate /= gate.sum(1, keepdim=True)
    inv = torch.randperm(T * K_r, device=dev, generator=g).int().view(T, K_r)
    out = torch.empty(T, d, device=dev)
    sh = moe.make_shape(T, d, V3.N_r, K_r, N_s, V3.I, V3.G, V3.M)
    moe.combine(u, y, gate, inv, sh, out)
    torch.cuda.synchronize()
    rows = np.random.default_rng(2).choice(T, 32, replace=False)
    for t in rows:
        ref = to_np(u[t]).astype(np.float64)
        ref = ref + sum(to_np(y[T * K_r + s * T + t]).astype(np.float64) for s in range(N_s))
        for k in range(K_r):
            ref = ref + float(gate[t, k]) * to_np(y[int(inv[t, k])]).astype(np.float64)
        np.testing.assert_allclose(to_np(out[t]), ref, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("N_r,K_r,G,M,T,d,n_seq", [
    (64, 4, 2, 2, 700, 256, 7),      # two groups of 32, top-2 per group; 100-token sequences
    (128, 8, 4, 4, 333, 512, 3),     # four groups of 32
    (128, 6, 4, 3, 257, 256, 1),
    (256, 8, 8, 8, 129, 384, 3),     # eight groups, one key each
    (256, 8, 1, 1, 96, 256, 3),      # no group limit; sequences of one window
    (64, 1, 1, 1, 50, 128, 5),       # K_r = 1; sequences shorter than a window
    # shapes outside the one-warp and eight-thread kernels: the general selection kernel
    (16, 2, 1, 1, 100, 256, 2),      # 16 experts: one warp per token
    (48, 5, 3, 1, 130, 128, 2),      # three groups of 16, the best group keeps all five
    (96, 6, 3, 3, 164, 256, 4),      # three groups of 32: one thread per token
    (200, 10, 1, 1, 77, 256, 1),     # ten of 200 experts
    # 256 experts, batches of 2048 tokens or more: the fused router's CTA-pair launches
    (256, 8, 8, 4, 2200, 384, 4),    # last 256-token tile partly past T, four slices of d
    (256, 6, 1, 1, 2100, 256, 2),    # the last tile's odd CTA holds no token
    (256, 8, 4, 2, 2048, 256, 1),    # two slices of d, two 64-wide blocks each
    (256, 8, 8, 4, 12288, 512, 3),   # 48 tiles: more clusters than fit in one wave
])
def test_router_shapes_bit_exact(N_r, K_r, G, M, T, d, n_seq):
    cfg = synth.MoEConfig("route", T=T, d=d, N_r=N_r, K_r=K_r, N_s=0, I=128, G=G, M=M,
                          dtype="bf16", bias="uniform", seed=N_r + T, n_seq=n_seq)
    x = synth.make_inputs(cfg, device="cuda", with_weights=False)
    sh, idx, gate, s, psum = _route(cfg, x)
    s_np, b = to_np(s), to_np(x["b"])
    idx_ref = oracle.select_experts(s_np, b, K_r, G, M)
    np.testing.assert_array_equal(to_np(idx), idx_ref)
    np.testing.assert_allclose(to_np(gate), oracle.gate_values(s_np, idx_ref), rtol=1e-6)
    np.testing.assert_allclose(to_np(psum), oracle.seq_p_sums(s_np, to_np(x["seq_offsets"])),
                               rtol=1e-5)


@pytest.mark.parametrize("T,offsets,N_r,G,M", [
    (100, [0, 0, 40, 40, 100], 128, 4, 2),           # one cluster: empty first and middle sequences
    (300, [0, 128, 128, 129, 300, 300], 128, 4, 2),  # several clusters: empty sequences at a boundary and at the end
    (2300, [0, 256, 256, 1000, 2300, 2300], 256, 8, 4),  # CTA-pair launch
])
def test_router_p_sums_with_empty_sequences(T, offsets, N_r, G, M):
    """The fused router's P sums where some sequences hold no token: those rows are zero,
    the others match the oracle (a batch of <= 128 tokens adds its sums inside one
    cluster, a larger one through the fixed-point accumulators)."""
    n_seq = len(offsets) - 1
    cfg = synth.MoEConfig("route-empty", T=T, d=256, N_r=N_r, K_r=8, N_s=0, I=128, G=G, M=M,
                          dtype="bf16", bias="uniform", seed=T, n_seq=1)
    x = synth.make_inputs(cfg, device="cuda", with_weights=False)
    x["seq_offsets"] = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    cfg = cfg.replace(n_seq=n_seq)
    sh, idx, gate, s, psum = _route(cfg, x)
    assert moe.device_error() == 0
    s_np = to_np(s)
    ref = oracle.seq_p_sums(s_np, np.array(offsets))
    np.testing.assert_allclose(to_np(psum), ref, rtol=1e-5, atol=1e-6)
    for j in range(n_seq):
        if offsets[j + 1] == offsets[j]:
            assert (to_np(psum)[j] == 0).all()


@pytest.mark.parametrize("N_r,K_r,G,M", [(256, 8, 8, 4), (64, 6, 1, 1), (128, 8, 4, 2)])
def test_router_exact_ties_go_to_lower_index(N_r, K_r, G, M):
    """Zero centroids give s = 0.5 for every expert, and biases repeat in steps of three,
    so most keys (and group scores) tie exactly: the lower index must win each tie."""
    T, d = 200, 256
    cfg = synth.MoEConfig("ties", T=T, d=d, N_r=N_r, K_r=K_r, N_s=0, I=128, G=G, M=M,
                          dtype="bf16", bias="zero", seed=1, n_seq=1)
    x = synth.make_inputs(cfg, device="cuda", with_weights=False)
    x["e"].zero_()
    x["b"].copy_(torch.tensor([(i % 3) * 0.25 for i in range(N_r)], device="cuda"))
    sh, idx, gate, s, psum = _route(cfg, x)
    s_np, b = to_np(s), to_np(x["b"])
    assert (s_np == 0.5).all()
    idx_ref = oracle.select_experts(s_np, b, K_r, G, M)
    np.testing.assert_array_equal(to_np(idx), idx_ref)
    np.testing.assert_allclose(to_np(gate), np.full((T, K_r), 1.0 / K_r), rtol=1e-6)


def test_expert_gemms_every_token_tile_size():
    """The bf16 gate/up and down GEMMs on hand-made expert segments of 0 to 700 rows:
    token tiles of every height from 1 to 256 rows (so every token-row box the
    kernels load, 16 to 128 rows a CTA), segments cut into two or three tiles, empty
    segments, and an output width (d = 320) that ends inside a 256-column tile.  Each
    segment's y rows are compared with the oracle's expert FFN of the same rows."""
    counts = [0, 1, 8, 15, 16, 17, 31, 32, 33, 47, 64, 65, 80, 100, 127, 128, 129, 150,
              176, 200, 239, 241, 255, 256, 257, 300, 400, 511, 513, 700, 0, 3]
    N_r, K_r, N_s, d, I = len(counts), 4, 1, 320, 384
    counts[-1] += -sum(counts) % K_r
    T = sum(counts) // K_r
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(21)
    rnd = lambda *shape, std=1.0: (torch.randn(*shape, device=dev, generator=g) * std).bfloat16()
    x_perm, u = rnd(T * K_r, d), rnd(T, d)
    w = {"w_gate": rnd(N_r, I, d, std=d ** -0.5), "w_up": rnd(N_r, I, d, std=d ** -0.5),
         "w_down": rnd(N_r, d, I, std=I ** -0.5), "ws_gate": rnd(N_s, I, d, std=d ** -0.5),
         "ws_up": rnd(N_s, I, d, std=d ** -0.5), "ws_down": rnd(N_s, d, I, std=I ** -0.5)}
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=dev)
    sh = moe.make_shape(T, d, N_r, K_r, N_s, I)
    h = torch.empty(T * K_r + N_s * T, I, dtype=torch.bfloat16, device=dev)
    y = torch.empty(T * K_r + N_s * T, d, dtype=torch.bfloat16, device=dev)
    moe.expert_gate_up(x_perm, u, off, sh, w, h)
    moe.expert_down(h, off, sh, w, y)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    yg, xn, un = to_np(y), to_np(x_perm), to_np(u)
    wn = {k: to_np(v) for k, v in w.items()}
    segs = [(xn[a:a + c], wn["w_gate"][i], wn["w_up"][i], wn["w_down"][i], a)
            for i, (a, c) in enumerate(zip(np.cumsum([0] + counts[:-1]), counts)) if c]
    segs.append((un, wn["ws_gate"][0], wn["ws_up"][0], wn["ws_down"][0], T * K_r))
    for xs, wg, wu, wd, r0 in segs:
        ref = oracle.expert_ffn(xs, wg, wu, wd)
        got = yg[r0:r0 + len(xs)].astype(np.float64)
        assert np.abs(got - ref).max() <= 2e-2, (r0, len(xs))
        assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref), (r0, len(xs))


def test_expert_gemms_small_batch_tiles():
    """Batches of at most 128 tokens (the down GEMM's small-batch ring: tiles of up to 128
    tokens, one MMA each): segments of every token-tile height up to 128 rows, one of 200
    rows (two tiles), empty segments and d = 320, against the oracle's expert FFN."""
    counts = [0, 1, 8, 15, 16, 17, 31, 32, 33, 47, 64, 65, 80, 100, 127, 128, 200, 0, 3]
    N_r, K_r, N_s, d, I = len(counts), 8, 1, 320, 384
    counts[-1] += -sum(counts) % K_r
    T = sum(counts) // K_r
    assert T <= 128
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(23)
    rnd = lambda *shape, std=1.0: (torch.randn(*shape, device=dev, generator=g) * std).bfloat16()
    x_perm, u = rnd(T * K_r, d), rnd(T, d)
    w = {"w_gate": rnd(N_r, I, d, std=d ** -0.5), "w_up": rnd(N_r, I, d, std=d ** -0.5),
         "w_down": rnd(N_r, d, I, std=I ** -0.5), "ws_gate": rnd(N_s, I, d, std=d ** -0.5),
         "ws_up": rnd(N_s, I, d, std=d ** -0.5), "ws_down": rnd(N_s, d, I, std=I ** -0.5)}
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=dev)
    sh = moe.make_shape(T, d, N_r, K_r, N_s, I)
    h = torch.empty(T * K_r + N_s * T, I, dtype=torch.bfloat16, device=dev)
    y = torch.empty(T * K_r + N_s * T, d, dtype=torch.bfloat16, device=dev)
    moe.expert_gate_up(x_perm, u, off, sh, w, h)
    moe.expert_down(h, off, sh, w, y)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    yg, xn, un = to_np(y), to_np(x_perm), to_np(u)
    wn = {k: to_np(v) for k, v in w.items()}
    segs = [(xn[a:a + c], wn["w_gate"][i], wn["w_up"][i], wn["w_down"][i], a)
            for i, (a, c) in enumerate(zip(np.cumsum([0] + counts[:-1]), counts)) if c]
    segs.append((un, wn["ws_gate"][0], wn["ws_up"][0], wn["ws_down"][0], T * K_r))
    for xs, wg, wu, wd, r0 in segs:
        ref = oracle.expert_ffn(xs, wg, wu, wd)
        got = yg[r0:r0 + len(xs)].astype(np.float64)
        assert np.abs(got - ref).max() <= 2e-2, (r0, len(xs))
        assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref), (r0, len(xs))


@pytest.mark.parametrize("d,I,seed", [(320, 384, 31), (2048, 1408, 32)])
def test_gate_up_gather_matches_x_perm_bit_for_bit(d, I, seed):
    """Gate/up reading the routed rows straight from u (row r = u[perm[r]]) against gate/up
    on x_perm = u[perm]: the MMAs see the same operands in the same order, so h is
    identical bit for bit.  Segments of every token-tile height as above, a d that ends
    inside a 64-wide K step (the gathered pieces past d are zeros), tokens repeated and
    in any order."""
    counts = [0, 1, 8, 15, 16, 17, 31, 32, 33, 47, 64, 65, 80, 100, 127, 128, 129, 150,
              176, 200, 239, 241, 255, 256, 257, 300, 400, 511, 513, 700, 0, 3]
    N_r, K_r, N_s = len(counts), 4, 1
    counts[-1] += -sum(counts) % K_r
    T = sum(counts) // K_r
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(seed)
    rnd = lambda *shape, std=1.0: (torch.randn(*shape, device=dev, generator=g) * std).bfloat16()
    u = rnd(T, d)
    perm = torch.randint(0, T, (T * K_r,), device=dev, generator=g, dtype=torch.int32)
    x_perm = u[perm.long()].contiguous()
    w = {"w_gate": rnd(N_r, I, d, std=d ** -0.5), "w_up": rnd(N_r, I, d, std=d ** -0.5),
         "w_down": rnd(N_r, d, I, std=I ** -0.5), "ws_gate": rnd(N_s, I, d, std=d ** -0.5),
         "ws_up": rnd(N_s, I, d, std=d ** -0.5), "ws_down": rnd(N_s, d, I, std=I ** -0.5)}
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=dev)
    sh = moe.make_shape(T, d, N_r, K_r, N_s, I)
    h_ref = torch.empty(T * K_r + N_s * T, I, dtype=torch.bfloat16, device=dev)
    h = torch.full_like(h_ref, float("nan"))
    moe.expert_gate_up(x_perm, u, off, sh, w, h_ref)
    moe.expert_gate_up_gather(u, perm, off, sh, w, h)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    assert torch.equal(h, h_ref)


def test_gate_up_gather_bad_token_is_a_zero_row_and_reported():
    """A perm entry outside [0, T) is read as a zero row (its h row is that of a zero
    token), the other rows are untouched, and the device error word reads
    MOE_ERR_INVALID_ARG."""
    T, d, I, N_r, K_r = 64, 256, 128, 4, 2
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(41)
    rnd = lambda *shape, std=1.0: (torch.randn(*shape, device=dev, generator=g) * std).bfloat16()
    u = rnd(T, d)
    perm = torch.arange(T * K_r, device=dev, dtype=torch.int32) % T
    perm[5], perm[77] = -3, T
    x_perm = u[perm.long().clamp(0, T - 1)].contiguous()
    x_perm[5].zero_()
    x_perm[77].zero_()
    w = {"w_gate": rnd(N_r, I, d, std=d ** -0.5), "w_up": rnd(N_r, I, d, std=d ** -0.5),
         "w_down": rnd(N_r, d, I, std=I ** -0.5)}
    off = torch.tensor([0, 40, 90, 100, T * K_r], dtype=torch.int32, device=dev)
    sh = moe.make_shape(T, d, N_r, K_r, 0, I)
    h_ref = torch.empty(T * K_r, I, dtype=torch.bfloat16, device=dev)
    h = torch.empty_like(h_ref)
    moe.expert_gate_up(x_perm, u, off, sh, w, h_ref)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    moe.expert_gate_up_gather(u, perm, off, sh, w, h)
    torch.cuda.synchronize()
    assert moe.STATUS[moe.device_error()] == "MOE_ERR_INVALID_ARG"   # read and cleared
    assert torch.equal(h, h_ref)


def test_out_of_range_expert_index_is_skipped_and_reported():
    """One topk_idx entry outside [0, N_r): dispatch skips it (no count, inv_row = -1,
    no gathered row), combine leaves it out, the device error word reads
    MOE_ERR_INVALID_ARG, and nothing is written past the output buffers."""
    T, d, N_r, K_r = 96, 256, 16, 2
    dev = "cuda"
    sh = moe.make_shape(T, d, N_r, K_r, 0, 128)
    g = torch.Generator(device=dev).manual_seed(3)
    idx = torch.stack([torch.randperm(N_r, generator=g, device=dev)[:K_r] for _ in range(T)]).int()
    idx[40, 1] = N_r + 5                                  # the bad entry
    u = torch.randn(T, d, device=dev, generator=g).bfloat16()
    guard = 64
    load = torch.empty(N_r, dtype=torch.int32, device=dev)
    off = torch.empty(N_r + 1, dtype=torch.int32, device=dev)
    perm = torch.full((T * K_r + guard,), -7, dtype=torch.int32, device=dev)
    inv = torch.full((T * K_r + guard,), -7, dtype=torch.int32, device=dev)
    xp = torch.full((T * K_r + guard, d), 3.0, device=dev).bfloat16()
    moe.device_error(clear=True)
    moe.dispatch(idx, sh, load, off, perm[:T * K_r], inv[:T * K_r].view(T, K_r), u=u,
                 x_perm=xp[:T * K_r])
    torch.cuda.synchronize()
    assert moe.device_error(clear=True) == 1              # MOE_ERR_INVALID_ARG
    assert int(load.sum()) == T * K_r - 1 and int(off[N_r]) == T * K_r - 1
    assert int(inv[40 * K_r + 1]) == -1
    assert (perm[T * K_r:] == -7).all() and (inv[T * K_r:] == -7).all()
    assert (xp[T * K_r:] == 3.0).all()
    valid = [(t, k) for t in range(T) for k in range(K_r) if (t, k) != (40, 1)]
    rows = inv[:T * K_r].view(T, K_r)
    for t, k in valid[::17]:
        assert torch.equal(xp[int(rows[t, k])], u[t])
    # combine: the skipped slot adds nothing
    y = torch.randn(T * K_r, d, device=dev, generator=g).bfloat16()
    gate = torch.full((T, K_r), 0.5, device=dev)
    h = torch.empty(T, d, device=dev)
    moe.combine(u, y, gate, rows.contiguous(), sh, h)
    torch.cuda.synchronize()
    assert moe.device_error(clear=True) == 1
    want = u[40].float() + 0.5 * y[int(rows[40, 0])].float()
    torch.testing.assert_close(h[40], want, rtol=1e-6, atol=1e-6)


def test_bad_sequence_offsets_are_reported():
    """seq_offsets that are not 0 <= ... <= T: the statistic records
    MOE_ERR_INVALID_ARG, treats the out-of-order sequence as empty and reads nothing
    outside topk_idx and seq_p_sum."""
    T, N_r, K_r = 256, 32, 4
    dev = "cuda"
    sh = moe.make_shape(T, 256, N_r, K_r, 0, 128)
    g = torch.Generator(device=dev).manual_seed(4)
    idx = torch.stack([torch.randperm(N_r, generator=g, device=dev)[:K_r] for _ in range(T)]).int()
    psum = torch.rand(3, N_r, device=dev, generator=g)
    stat = torch.full((3,), -1.0, device=dev)
    mean = torch.empty(1, device=dev)
    ok_off = torch.tensor([0, 100, 180, T], dtype=torch.int32, device=dev)
    moe.device_error(clear=True)
    moe.seq_balance_stat(psum, idx, ok_off, 3, sh, 1e-4, stat, mean)
    torch.cuda.synchronize()
    assert moe.device_error(clear=True) == 0
    good = stat.clone()
    bad_off = torch.tensor([0, 180, 100, T], dtype=torch.int32, device=dev)   # 180 > 100
    moe.seq_balance_stat(psum, idx, bad_off, 3, sh, 1e-4, stat, mean)
    torch.cuda.synchronize()
    assert moe.device_error(clear=True) == 1
    assert float(stat[1]) == 0.0                         # [180, 100) counts as empty
    short_off = torch.tensor([0, 100, 180, T - 1], dtype=torch.int32, device=dev)
    moe.seq_balance_stat(psum, idx, short_off, 3, sh, 1e-4, stat, mean)
    torch.cuda.synchronize()
    assert moe.device_error(clear=True) == 1             # does not end at T
    assert float(stat[0]) == float(good[0])
