"""The C ABI without a GPU: the library loads, exports every call include/moe.h
declares, answers workspace queries, and rejects invalid arguments before launching
anything (so these calls never reach the device)."""
import ctypes
import os
import re

import pytest

import aux_loss_free_router_b300 as moe
from aux_loss_free_router_b300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load_library()


def _declared():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe._SIGS), "binding and header disagree"


def test_status_strings_and_version(lib):
    assert lib.moe_abi_version() == 1
    for code in range(6):
        assert lib.moe_status_string(code)
    assert lib.moe_status_string(0) == b"ok"


FAKE = 1 << 20      # aligned, never dereferenced: validation fails first


def shape(**kw):
    base = dict(T=64, d=256, N_r=16, K_r=2, N_s=1, I=128, G=1, M=1)
    base.update(kw)
    return moe.make_shape(**base)


@pytest.mark.parametrize("bad", [
    dict(K_r=0), dict(K_r=17), dict(N_r=257), dict(N_r=300, K_r=2), dict(G=3),
    dict(G=4, M=3), dict(G=4, M=5), dict(G=16, M=1, K_r=2), dict(d=12), dict(I=100),
    dict(T=-1), dict(N_s=33), dict(K_r=33, N_r=64)])
def test_route_rejects_bad_shapes(lib, bad):
    code = lib.moe_route(FAKE, FAKE, moe.BF16, FAKE, shape(**bad), None, 0, FAKE, FAKE, None,
                         None, None, 0, None)
    assert code == 1


def test_route_rejects_bad_pointers_and_dtype(lib):
    sh = shape()
    assert lib.moe_route(None, FAKE, moe.BF16, FAKE, sh, None, 0, FAKE, FAKE, None, None, None, 0, None) == 1
    assert lib.moe_route(FAKE + 4, FAKE, moe.BF16, FAKE, sh, None, 0, FAKE, FAKE, None, None, None, 0, None) == 1
    assert lib.moe_route(FAKE, FAKE, moe.E4M3, FAKE, sh, None, 0, FAKE, FAKE, None, None, None, 0, None) == 2
    # statistics requested without sequences, then without workspace
    assert lib.moe_route(FAKE, FAKE, moe.BF16, FAKE, sh, None, 0, FAKE, FAKE, None, FAKE, None, 0, None) == 1
    assert lib.moe_route(FAKE, FAKE, moe.BF16, FAKE, sh, FAKE, 1, FAKE, FAKE, None, FAKE, None, 0, None) == 3
    need = lib.moe_route_workspace(sh, 1)
    assert lib.moe_route(FAKE, FAKE, moe.BF16, FAKE, sh, FAKE, 1, FAKE, FAKE, None, FAKE, FAKE,
                         need - 1, None) == 3


def test_workspace_queries(lib):
    sh = shape(T=8192, d=7168, N_r=256, K_r=8, I=2048, G=8, M=4)
    assert lib.moe_route_workspace(sh, 2) >= 8192 * 256 * 4
    assert lib.moe_route_workspace(sh, 0) >= 8192 * 256 * 4      # split-K partials
    assert lib.moe_route_workspace(sh, 2) > lib.moe_route_workspace(sh, 0)
    assert lib.moe_dispatch_workspace(sh) >= (8192 // 32) * 256 * 4
    assert lib.moe_expert_ffn_workspace(sh, moe.BF16) >= (8192 * 8 + 8192) * 2048 * 2
    assert lib.moe_dispatch_workspace(shape(T=0)) == 0


def test_dispatch_and_ffn_reject_bad_args(lib):
    sh = shape()
    ws = lib.moe_dispatch_workspace(sh)
    assert lib.moe_dispatch(FAKE, sh, FAKE, moe.BF16, None, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, ws, None) == 1
    assert lib.moe_dispatch(FAKE, sh, FAKE, moe.BF16, None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, ws, None) == 1
    assert lib.moe_dispatch(FAKE, sh, None, moe.BF16, None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, ws - 4, None) == 3
    # E4M3 gather without scales
    assert lib.moe_dispatch(FAKE, sh, FAKE, moe.E4M3, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, ws, None) == 1
    w = moe._Weights(moe.BF16, FAKE, FAKE, None, None, None, None, FAKE, FAKE, FAKE, None, None, None)
    assert lib.moe_expert_gate_up(FAKE, None, FAKE, None, FAKE, sh, ctypes.byref(w), FAKE, None, None) == 1
    # gate/up reading rows from u: every pointer needed, u 16-byte aligned, bf16 weights only
    w.down = FAKE
    assert lib.moe_expert_gate_up_gather(None, FAKE, FAKE, sh, ctypes.byref(w), FAKE, None) == 1
    assert lib.moe_expert_gate_up_gather(FAKE + 8, FAKE, FAKE, sh, ctypes.byref(w), FAKE, None) == 1
    assert lib.moe_expert_gate_up_gather(FAKE, None, FAKE, sh, ctypes.byref(w), FAKE, None) == 1
    assert lib.moe_expert_gate_up_gather(FAKE, FAKE, FAKE, sh, ctypes.byref(w), None, None) == 1
    assert lib.moe_expert_gate_up_gather(None, None, None, shape(T=0), ctypes.byref(w), None, None) == 0
    w.dtype = moe.F32
    assert lib.moe_expert_gate_up_gather(FAKE, FAKE, FAKE, sh, ctypes.byref(w), FAKE, None) == 1
    w.dtype, w.down = moe.BF16, None
    assert lib.moe_expert_ffn(FAKE, None, FAKE, None, FAKE, sh, None, FAKE, FAKE, 1 << 30, None) == 1
    w.down = FAKE
    assert lib.moe_expert_ffn(FAKE, None, FAKE, None, FAKE, sh, ctypes.byref(w), FAKE, FAKE, 16, None) == 3


def test_quant_combine_balance_reject_bad_args(lib):
    assert lib.moe_quantize_e4m3(FAKE, moe.BF16, 4, 100, 1, FAKE, FAKE, None) == 1
    assert lib.moe_quantize_e4m3(FAKE, moe.BF16, 100, 128, 128, FAKE, FAKE, None) == 1
    assert lib.moe_quantize_e4m3(FAKE, moe.BF16, 128, 128, 2, FAKE, FAKE, None) == 1
    assert lib.moe_quantize_e4m3(FAKE, moe.E4M3, 128, 128, 1, FAKE, FAKE, None) == 2
    sh = shape()
    assert lib.moe_combine(FAKE, FAKE, moe.E4M3, FAKE, FAKE, sh, FAKE, moe.BF16, None) == 2
    assert lib.moe_combine(FAKE, None, moe.BF16, FAKE, FAKE, sh, FAKE, moe.BF16, None) == 1
    assert lib.moe_bias_update(None, FAKE, sh, 0.001, None) == 1
    assert lib.moe_bias_update(FAKE, FAKE, sh, -1.0, None) == 1
    assert lib.moe_seq_balance_stat(FAKE, FAKE, FAKE, 0, sh, 1e-4, FAKE, FAKE, None) == 1
    assert lib.moe_device_error(None, 0) == 1


def test_expert_calls_check_weights_and_empty_batches(lib):
    """E4M3 weights need their block scales and d, I multiples of 128; an unknown
    weight dtype is unsupported; an empty batch is accepted and enqueues nothing."""
    sh = shape()
    w = moe._Weights(moe.E4M3, FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, FAKE, None, None, None)
    assert lib.moe_expert_gate_up(FAKE, FAKE, FAKE, FAKE, FAKE, sh, ctypes.byref(w), FAKE, FAKE, None) == 1
    w.gate_scale = w.up_scale = w.down_scale = FAKE
    w.s_gate_scale = w.s_up_scale = w.s_down_scale = FAKE
    assert lib.moe_expert_down(FAKE, FAKE, FAKE, shape(I=200), ctypes.byref(w), FAKE, None) == 1
    assert lib.moe_expert_down(FAKE, FAKE, FAKE, shape(d=264), ctypes.byref(w), FAKE, None) == 1
    w.dtype = 7
    assert lib.moe_expert_down(FAKE, None, FAKE, sh, ctypes.byref(w), FAKE, None) == 2
    w.dtype = moe.BF16
    assert lib.moe_expert_down(FAKE, None, FAKE, sh, ctypes.byref(w), None, None) == 1
    assert lib.moe_expert_down(FAKE, None, FAKE, sh, ctypes.byref(w), FAKE + 8, None) == 1
    empty = shape(T=0)
    assert lib.moe_expert_gate_up(None, None, None, None, None, empty, ctypes.byref(w), None, None, None) == 0
    assert lib.moe_expert_ffn(None, None, None, None, None, empty, ctypes.byref(w), None, None, 0, None) == 0
    assert lib.moe_combine(None, None, moe.BF16, None, None, empty, None, moe.F32, None) == 0


def test_combine_route_and_statistic_argument_checks(lib):
    sh = shape()
    assert lib.moe_combine(FAKE, FAKE, moe.BF16, FAKE, FAKE, sh, FAKE, moe.E4M3, None) == 2
    assert lib.moe_combine(FAKE, FAKE, moe.BF16, FAKE, FAKE, sh, FAKE + 4, moe.F32, None) == 1
    assert lib.moe_route(FAKE, FAKE, moe.BF16, FAKE, sh, FAKE, -1, FAKE, FAKE, None, None, None, 0, None) == 1
    assert lib.moe_route(FAKE, FAKE, moe.BF16, FAKE, sh, None, 0, FAKE, FAKE, FAKE + 4, None, None, 0, None) == 1
    assert lib.moe_seq_balance_stat(None, FAKE, FAKE, 2, sh, 1e-4, FAKE, FAKE, None) == 1
    assert lib.moe_seq_balance_stat(FAKE, None, FAKE, 2, sh, 1e-4, FAKE, FAKE, None) == 1
    assert lib.moe_seq_balance_stat(FAKE, FAKE, FAKE, 2, sh, 1e-4, FAKE, FAKE + 4, None) == 1
    assert lib.moe_bias_update(FAKE, FAKE, shape(G=3), 0.001, None) == 1
