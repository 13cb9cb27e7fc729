"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate device memory
(an application whose allocator owns the whole device, or a runtime whose buffers
are all fixed before it starts).  It keeps its chunk counts in a device array built
into the library instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row, on different routings, and
checks each result against moe_dispatch with a caller workspace: both are integer
work (loads, offsets, permutation, inverse rows) plus a row copy, so they must agree
bit for bit.  The second call shows that what the first call left in the shared
array does not leak into the next one.

This file is named to be collected last, so a run that stops at the first failure
has already run every other test; it passes alone in a fresh process too.
"""
import numpy as np
import pytest
import torch

import synth
import aux_loss_free_router_b300 as moe
from aux_loss_free_router_b300 import build as moe_build
from tests.layer_harness import run_layer


def _routing(rng, T, N_r, K_r, conc):
    p = rng.dirichlet(np.ones(N_r) * conc)
    return np.stack([rng.choice(N_r, K_r, replace=False, p=p) for _ in range(T)])


def _dispatch_pair(idx, u, sh, T, N_r, K_r, d):
    dev = u.device
    t_idx = torch.as_tensor(idx, dtype=torch.int32, device=dev)
    outs = []
    for fn in (moe.dispatch, moe.dispatch_noalloc):
        load = torch.full((N_r,), -7, dtype=torch.int32, device=dev)
        off = torch.full((N_r + 1,), -7, dtype=torch.int32, device=dev)
        perm = torch.full((T * K_r,), -7, dtype=torch.int32, device=dev)
        inv = torch.full((T, K_r), -7, dtype=torch.int32, device=dev)
        xp = torch.zeros(T * K_r, d, dtype=u.dtype, device=dev)
        fn(t_idx, sh, load, off, perm, inv, u, xp)
        torch.cuda.synchronize()
        outs.append((load, off, perm, inv, xp))
    return outs


@pytest.mark.gpu
def test_noalloc_dispatch_matches_workspace_dispatch_twice():
    cfg = synth.config("v3")
    T, N_r, K_r, d = cfg.T, cfg.N_r, cfg.K_r, cfg.d
    sh = moe.make_shape(T, d, N_r, K_r, cfg.N_s, cfg.I, cfg.G, cfg.M)
    u = synth.make_inputs(cfg, device="cuda", with_weights=False)["u"]
    rng = np.random.default_rng(5)
    # two different routings back to back: a skewed one, then a near-uniform one
    for conc in (0.2, 50.0):
        idx = _routing(rng, T, N_r, K_r, conc)
        ref, got = _dispatch_pair(idx, u, sh, T, N_r, K_r, d)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
        assert int(got[0].sum()) == T * K_r
    assert moe.device_error() == 0


@pytest.mark.gpu
def test_noalloc_dispatch_at_its_largest_batch():
    """65536 tokens with 256 experts: ceil(T/32) * N_r fills the built-in scratch exactly."""
    T, N_r, K_r, d = 65536, 256, 8, 128
    sh = moe.make_shape(T, d, N_r, K_r, 0, 128, 1, 1)
    g = torch.Generator(device="cuda").manual_seed(9)
    u = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    idx = _routing(np.random.default_rng(9), T, N_r, K_r, 1.0)
    ref, got = _dispatch_pair(idx, u, sh, T, N_r, K_r, d)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    assert int(got[0].sum()) == T * K_r
    assert moe.device_error() == 0


def test_noalloc_dispatch_rejects_batches_beyond_its_scratch():
    moe_build.build()
    lib = moe.load_library()
    fake = 1 << 20   # aligned, never dereferenced: the size check fails first
    # ceil(T/32) * N_r above 524288 counts: T = 65568 tokens with 256 experts
    sh = moe.make_shape(65568, 256, 256, 8, 0, 128, 1, 1)
    code = lib.moe_dispatch_noalloc(fake, sh, None, moe.BF16, None, fake, fake, fake, fake,
                                    None, None, None)
    assert code == 1


@pytest.mark.gpu
def test_noalloc_dispatch_gathers_e4m3_rows_and_scales():
    """The allocation-free dispatch on E4M3 tokens: codes and their 1x128 scales are
    gathered exactly like the workspace dispatch does."""
    cfg = synth.config("fp8", T=1024, n_seq=1)
    r = run_layer(cfg)
    lay = r["layer"]
    dev = "cuda"
    sh = lay.shape
    out = []
    for fn in (moe.dispatch, moe.dispatch_noalloc):
        load = torch.empty(cfg.N_r, dtype=torch.int32, device=dev)
        off = torch.empty(cfg.N_r + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(cfg.T * cfg.K_r, dtype=torch.int32, device=dev)
        inv = torch.empty(cfg.T, cfg.K_r, dtype=torch.int32, device=dev)
        xp = torch.empty_like(lay.x_perm)
        xs = torch.empty_like(lay.x_perm_scale)
        fn(lay.topk_idx, sh, load, off, perm, inv, lay.u_q, xp, lay.u_scale, xs)
        torch.cuda.synchronize()
        out.append((load, off, perm, inv, xp, xs))
    for a, b in zip(*out):
        assert torch.equal(a, b)
    assert torch.equal(out[0][4], lay.x_perm) and torch.equal(out[0][5], lay.x_perm_scale)
