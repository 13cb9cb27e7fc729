"""Python binding of ``libmoe.so``: the B300 forward pass of a DeepSeekMoE layer with
auxiliary-loss-free load balancing.

Every function here only marshals arguments (device pointers, sizes, the current
CUDA stream) and calls the C ABI declared in ``include/moe.h`` of the same name; all
arithmetic runs in the library's CUDA kernels.  There is no CPU or PyTorch fallback:
if the library is missing or a call fails, a ``MoEError`` is raised.

Tensors are ``torch.Tensor`` on a CUDA device, contiguous, in the layouts of moe.h.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

__all__ = [
    "MoEError", "Shape", "load_library", "route", "dispatch", "dispatch_noalloc", "quantize_e4m3",
    "expert_gate_up", "expert_gate_up_gather", "expert_down", "expert_ffn", "combine", "bias_update",
    "seq_balance_stat", "device_error", "quantize_weights", "route_workspace_bytes",
    "backward", "backward_workspace_bytes",
    "dispatch_workspace_bytes", "expert_ffn_workspace_bytes", "MoELayer",
    "LIB_PATH", "STATUS", "launch_counter", "launch_counter_reset", "make_shape",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT"}
F32, BF16, E4M3 = 0, 1, 2


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "d", "N_r", "K_r", "N_s", "I", "G", "M")]


class _Weights(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int)] + [
        (n, ctypes.c_void_p) for n in (
            "gate", "up", "down", "gate_scale", "up_scale", "down_scale",
            "s_gate", "s_up", "s_down", "s_gate_scale", "s_up_scale", "s_down_scale")]


class _DgradWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "wdt", "wdt_scale", "wgut", "wgut_scale", "s_wdt", "s_wdt_scale", "s_wgut", "s_wgut_scale")]


_P, _S, _I32, _I64, _F = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_abi_version": (ctypes.c_int, []),
    "moe_route_workspace": (_S, [Shape, _I32]),
    "moe_route": (ctypes.c_int, [_P, _P, ctypes.c_int, _P, Shape, _P, _I32, _P, _P, _P, _P, _P, _S, _P]),
    "moe_dispatch_workspace": (_S, [Shape]),
    "moe_dispatch": (ctypes.c_int, [_P, Shape, _P, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_dispatch_noalloc": (ctypes.c_int, [_P, Shape, _P, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_quantize_e4m3": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _I32, _P, _P, _P]),
    "moe_expert_ffn_workspace": (_S, [Shape, ctypes.c_int]),
    "moe_expert_gate_up": (ctypes.c_int, [_P, _P, _P, _P, _P, Shape, ctypes.POINTER(_Weights), _P, _P, _P]),
    "moe_expert_gate_up_gather": (ctypes.c_int, [_P, _P, _P, Shape, ctypes.POINTER(_Weights), _P, _P]),
    "moe_expert_down": (ctypes.c_int, [_P, _P, _P, Shape, ctypes.POINTER(_Weights), _P, _P]),
    "moe_expert_ffn": (ctypes.c_int, [_P, _P, _P, _P, _P, Shape, ctypes.POINTER(_Weights), _P, _P, _S, _P]),
    "moe_combine": (ctypes.c_int, [_P, _P, ctypes.c_int, _P, _P, Shape, _P, ctypes.c_int, _P]),
    "moe_bias_update": (ctypes.c_int, [_P, _P, Shape, _F, _P]),
    "moe_seq_balance_stat": (ctypes.c_int, [_P, _P, _P, _I32, Shape, _F, _P, _P, _P]),
    "moe_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), _I32]),
    "moe_backward_workspace": (_S, [Shape, _I32]),
    "moe_backward": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(_Weights),
                                    Shape, _P, _I32, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _S, _P]),
    "moe_fp8_dgrad_weights_make": (ctypes.c_int, [ctypes.POINTER(_Weights), Shape,
                                                  ctypes.POINTER(_DgradWeights), _P]),
    "moe_backward_fp8_workspace": (_S, [Shape, _I32]),
    "moe_backward_fp8": (ctypes.c_int, [_P] * 12 + [ctypes.POINTER(_Weights), ctypes.POINTER(_DgradWeights),
                                                    Shape, _P, _I32, _F] + [_P] * 10 + [_S, _P]),
}

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (once).  Raises ``OSError`` if it is missing:
    build it with ``python -m aux_loss_free_router_b300.build``."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise OSError(f"{path} not found: run `python -m aux_loss_free_router_b300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


# Kernels each call enqueues for a non-empty batch (the launch count of a step).
_KERNELS = {"moe_route": 2, "moe_dispatch": 3, "moe_dispatch_noalloc": 3, "moe_quantize_e4m3": 1, "moe_expert_gate_up": 1,
            "moe_expert_gate_up_gather": 1,
            "moe_expert_down": 1, "moe_expert_ffn": 2, "moe_combine": 1, "moe_bias_update": 1,
            "moe_seq_balance_stat": 1,
            # gate/up recompute, per-token prep, six GEMMs, combine (+ counts with the
            # balance term)
            "moe_backward": 9,
            # weight transposes: W_down^T, W_gate^T, W_up^T (routed; again for shared)
            "moe_fp8_dgrad_weights_make": 3,
            # gate/up recompute, prep, dY quantisation, two Dgrad GEMMs, SwiGLU backward,
            # five Wgrad operand quantisations, three Wgrad GEMMs, two router GEMMs, combine
            "moe_backward_fp8": 17}
_launches = 0


def launch_counter_reset() -> None:
    global _launches
    _launches = 0


def launch_counter() -> int:
    """Kernels launched through this binding since the last reset."""
    return _launches


def _call(name: str, *args, extra_kernels: int = 0) -> None:
    global _launches
    code = getattr(load_library(), name)(*args)
    if code != 0:
        raise MoEError(name, code)
    _launches += _KERNELS.get(name, 0) + extra_kernels


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the MoE library must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return E4M3
    raise ValueError(f"unsupported dtype {t.dtype}")


def make_shape(T, d, N_r, K_r, N_s, I, G=1, M=1) -> Shape:
    return Shape(T, d, N_r, K_r, N_s, I, G, M)


# ----------------------------------------------------------------- workspaces -----

def route_workspace_bytes(sh: Shape, n_seq: int) -> int:
    return load_library().moe_route_workspace(sh, n_seq)


def dispatch_workspace_bytes(sh: Shape) -> int:
    return load_library().moe_dispatch_workspace(sh)


def expert_ffn_workspace_bytes(sh: Shape, w_dtype: int) -> int:
    return load_library().moe_expert_ffn_workspace(sh, w_dtype)


def _workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device) if nbytes else None


# ------------------------------------------------------------------ the calls -----

def route(u, e, b, sh: Shape, topk_idx, topk_gate, s_out=None, seq_offsets=None, n_seq=0,
          seq_p_sum=None, workspace=None, stream=None):
    ws = workspace
    if ws is None:
        ws = _workspace(route_workspace_bytes(sh, n_seq if seq_p_sum is not None else 0), u.device)
    _call("moe_route", _ptr(u), _ptr(e), _dt(u), _ptr(b), sh, _ptr(seq_offsets), n_seq,
          _ptr(topk_idx), _ptr(topk_gate), _ptr(s_out), _ptr(seq_p_sum), _ptr(ws),
          ws.numel() if ws is not None else 0, _stream(stream),
          extra_kernels=_route_kernels(sh, _dt(u), seq_p_sum is not None) - _KERNELS["moe_route"])


def _route_kernels(sh: Shape, dt: int, with_stat: bool) -> int:
    """Kernels one moe_route call launches: one for the fused bf16 path (64/128/256
    experts, K_r <= 8, groups of whole 32-expert blocks keeping <= 2 keys, d >= 128),
    else the affinity GEMM and the selection, plus the P-sum kernel with statistics."""
    grouped_ok = sh.G == 1 or ((sh.N_r // 32) % sh.G == 0 and sh.K_r // sh.M <= 2)
    if dt == BF16 and sh.N_r in (64, 128, 256) and sh.K_r <= 8 and grouped_ok and sh.d >= 128:
        return 1
    return 2 + (1 if with_stat else 0)


def dispatch(topk_idx, sh: Shape, load, expert_offset, perm_token, inv_row, u=None,
             x_perm=None, u_scale=None, x_perm_scale=None, workspace=None, stream=None):
    ws = workspace if workspace is not None else _workspace(dispatch_workspace_bytes(sh), topk_idx.device)
    _call("moe_dispatch", _ptr(topk_idx), sh, _ptr(u), _dt(u) if u is not None else BF16,
          _ptr(u_scale), _ptr(load), _ptr(expert_offset), _ptr(perm_token), _ptr(inv_row),
          _ptr(x_perm), _ptr(x_perm_scale), _ptr(ws), ws.numel() if ws is not None else 0,
          _stream(stream), extra_kernels=_dispatch_kernels(sh, x_perm is not None) - 3)


def dispatch_noalloc(topk_idx, sh: Shape, load, expert_offset, perm_token, inv_row, u=None,
                     x_perm=None, u_scale=None, x_perm_scale=None, stream=None):
    """``dispatch`` for callers that cannot allocate device memory: the chunk counts
    live in the library's built-in device array (T <= 65536 at 256 experts), which all
    calls on a device share, so calls must not overlap on the GPU."""
    _call("moe_dispatch_noalloc", _ptr(topk_idx), sh, _ptr(u), _dt(u) if u is not None else BF16,
          _ptr(u_scale), _ptr(load), _ptr(expert_offset), _ptr(perm_token), _ptr(inv_row),
          _ptr(x_perm), _ptr(x_perm_scale), _stream(stream),
          extra_kernels=_dispatch_kernels(sh, x_perm is not None) - 3)


def _dispatch_kernels(sh: Shape, gather: bool) -> int:
    """Kernels one dispatch launches: count, scan and scatter (one kernel while each 32nd
    of the tokens holds at most 512 (token, slot) entries, three above), plus the row
    gather."""
    if sh.T == 0:
        return 0
    small = ((sh.T + 31) // 32) * sh.K_r <= 512
    return (1 if small else 3) + (1 if gather else 0)


def quantize_e4m3(x, block_rows: int, q, scale, stream=None):
    rows, cols = x.shape[0] if x.dim() == 2 else x.numel() // x.shape[-1], x.shape[-1]
    _call("moe_quantize_e4m3", _ptr(x), _dt(x), rows, cols, block_rows, _ptr(q), _ptr(scale),
          _stream(stream))


def _weights(w: dict) -> _Weights:
    g = w["w_gate"]
    dt = E4M3 if g.dtype in (torch.uint8, torch.float8_e4m3fn) else _dt(g)
    get = lambda k: _ptr(w.get(k))
    return _Weights(dt, get("w_gate"), get("w_up"), get("w_down"), get("w_gate_scale"),
                    get("w_up_scale"), get("w_down_scale"), get("ws_gate"), get("ws_up"),
                    get("ws_down"), get("ws_gate_scale"), get("ws_up_scale"), get("ws_down_scale"))


def expert_gate_up(x_perm, u, expert_offset, sh: Shape, weights: dict, h, x_perm_scale=None,
                   u_scale=None, h_scale=None, stream=None):
    wt = _weights(weights)
    _call("moe_expert_gate_up", _ptr(x_perm), _ptr(x_perm_scale), _ptr(u), _ptr(u_scale),
          _ptr(expert_offset), sh, ctypes.byref(wt), _ptr(h), _ptr(h_scale), _stream(stream))


def expert_gate_up_gather(u, perm_token, expert_offset, sh: Shape, weights: dict, h, stream=None):
    """bf16 gate/up reading the routed rows' tokens straight from u (row r is
    u[perm_token[r]]): the dispatch can skip writing x_perm."""
    wt = _weights(weights)
    _call("moe_expert_gate_up_gather", _ptr(u), _ptr(perm_token), _ptr(expert_offset), sh,
          ctypes.byref(wt), _ptr(h), _stream(stream))


def expert_down(h, expert_offset, sh: Shape, weights: dict, y, h_scale=None, stream=None):
    wt = _weights(weights)
    _call("moe_expert_down", _ptr(h), _ptr(h_scale), _ptr(expert_offset), sh, ctypes.byref(wt),
          _ptr(y), _stream(stream))


def expert_ffn(x_perm, u, expert_offset, sh: Shape, weights: dict, y, workspace=None,
               x_perm_scale=None, u_scale=None, stream=None):
    wt = _weights(weights)
    ws = workspace if workspace is not None else _workspace(
        expert_ffn_workspace_bytes(sh, wt.dtype), u.device)
    _call("moe_expert_ffn", _ptr(x_perm), _ptr(x_perm_scale), _ptr(u), _ptr(u_scale),
          _ptr(expert_offset), sh, ctypes.byref(wt), _ptr(y), _ptr(ws),
          ws.numel() if ws is not None else 0, _stream(stream))


def combine(u, y, topk_gate, inv_row, sh: Shape, h_out, stream=None):
    _call("moe_combine", _ptr(u), _ptr(y), _dt(u), _ptr(topk_gate), _ptr(inv_row), sh,
          _ptr(h_out), _dt(h_out), _stream(stream))


def bias_update(b, load, sh: Shape, gamma: float, stream=None):
    _call("moe_bias_update", _ptr(b), _ptr(load), sh, gamma, _stream(stream))


def seq_balance_stat(seq_p_sum, topk_idx, seq_offsets, n_seq: int, sh: Shape, alpha: float,
                     stat_per_seq, stat_mean=None, stream=None):
    _call("moe_seq_balance_stat", _ptr(seq_p_sum), _ptr(topk_idx), _ptr(seq_offsets), n_seq, sh,
          alpha, _ptr(stat_per_seq), _ptr(stat_mean), _stream(stream),
          extra_kernels=1 if (stat_mean is not None and n_seq > 1) else 0)


def backward_workspace_bytes(sh: Shape, n_seq: int) -> int:
    return load_library().moe_backward_workspace(sh, n_seq)


def backward(u, e, s, topk_idx, topk_gate, expert_offset, inv_row, x_perm, y, sh: Shape,
             weights: dict, dh, grads: dict, seq_offsets=None, n_seq: int = 0,
             alpha: float = 0.0, workspace=None, stream=None):
    """moe_backward: gradients of sum(dh * h') (+ the mean balance loss) at the forward
    pass's selection.  ``grads`` holds the fp32 outputs "u", "e", "w_gate", "w_up",
    "w_down" and, with shared experts, "ws_gate", "ws_up", "ws_down"."""
    wt = _weights(weights)
    ws = workspace if workspace is not None else _workspace(backward_workspace_bytes(sh, n_seq), u.device)
    g = lambda k: _ptr(grads.get(k))
    balance = n_seq > 0 and alpha != 0.0
    _call("moe_backward", _ptr(u), _ptr(e), _ptr(s), _ptr(topk_idx), _ptr(topk_gate),
          _ptr(expert_offset), _ptr(inv_row), _ptr(x_perm), _ptr(y), ctypes.byref(wt), sh,
          _ptr(seq_offsets), n_seq, alpha, _ptr(dh), g("u"), g("e"), g("w_gate"), g("w_up"),
          g("w_down"), g("ws_gate"), g("ws_up"), g("ws_down"), _ptr(ws),
          ws.numel() if ws is not None else 0, _stream(stream),
          extra_kernels=1 if balance else 0)


def fp8_dgrad_weights(weights8: dict, sh: Shape, stream=None) -> dict:
    """moe_fp8_dgrad_weights_make: the transposed E4M3 weights of the FP8 Dgrad GEMMs
    ("wdt" [E, I, d], "wgut" [E, d, 2I] with their "_scale" grids; "s_*" for the shared
    experts) from the E4M3 weights of ``quantize_weights``."""
    wq = weights8["w_gate"]
    dev, N_r, I, d = wq.device, sh.N_r, sh.I, sh.d
    out = {}
    for pre, E in (("", N_r), ("s_", sh.N_s)):
        out[pre + "wdt"] = torch.empty(E, I, d, dtype=torch.uint8, device=dev)
        out[pre + "wdt_scale"] = torch.empty(E, I // 128, d // 128, dtype=torch.float32, device=dev)
        out[pre + "wgut"] = torch.empty(E, d, 2 * I, dtype=torch.uint8, device=dev)
        out[pre + "wgut_scale"] = torch.empty(E, d // 128, 2 * I // 128, dtype=torch.float32, device=dev)
    st = _DgradWeights(*[_ptr(out[k]) if out[k].numel() else None for k in (
        "wdt", "wdt_scale", "wgut", "wgut_scale", "s_wdt", "s_wdt_scale", "s_wgut", "s_wgut_scale")])
    wt = _weights(weights8)
    _call("moe_fp8_dgrad_weights_make", ctypes.byref(wt), sh, ctypes.byref(st), _stream(stream),
          extra_kernels=3 if sh.N_s else 0)
    out["_struct"] = st
    return out


def backward_fp8_workspace_bytes(sh: Shape, n_seq: int) -> int:
    return load_library().moe_backward_fp8_workspace(sh, n_seq)


def backward_fp8(u, u_q, u_scale, e, s, topk_idx, topk_gate, expert_offset, inv_row, x_perm_q,
                 x_perm_scale, y, sh: Shape, weights8: dict, dgrad_weights: dict, dh, grads: dict,
                 seq_offsets=None, n_seq: int = 0, alpha: float = 0.0, workspace=None, stream=None):
    """moe_backward_fp8: the gradients of ``backward`` for an FP8 layer, its expert GEMMs
    (Fprop again, Dgrad, Wgrad) in E4M3.  ``weights8``: ``quantize_weights`` output;
    ``dgrad_weights``: ``fp8_dgrad_weights`` output."""
    wt = _weights(weights8)
    ws = workspace if workspace is not None else _workspace(backward_fp8_workspace_bytes(sh, n_seq), u.device)
    g = lambda k: _ptr(grads.get(k))
    balance = n_seq > 0 and alpha != 0.0
    _call("moe_backward_fp8", _ptr(u), _ptr(u_q), _ptr(u_scale), _ptr(e), _ptr(s), _ptr(topk_idx),
          _ptr(topk_gate), _ptr(expert_offset), _ptr(inv_row), _ptr(x_perm_q), _ptr(x_perm_scale),
          _ptr(y), ctypes.byref(wt), ctypes.byref(dgrad_weights["_struct"]), sh, _ptr(seq_offsets),
          n_seq, alpha, _ptr(dh), g("u"), g("e"), g("w_gate"), g("w_up"), g("w_down"), g("ws_gate"),
          g("ws_up"), g("ws_down"), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream),
          extra_kernels=1 if balance else 0)


def device_error(clear: bool = True) -> int:
    code = ctypes.c_int32(0)
    _call("moe_device_error", ctypes.byref(code), int(clear))
    return code.value


def quantize_weights(weights: dict, stream=None) -> dict:
    """E4M3 codes and per-128x128-block fp32 scales of bf16/fp32 expert weights
    (``w_gate``/``w_up`` [E, I, d], ``w_down`` [E, d, I] and the shared ``ws_*``), via
    moe_quantize_e4m3; returns the dict the FFN calls take for E4M3 weights."""
    out = {}
    for k, w in weights.items():
        if w is None:
            continue
        E, R, C = w.shape
        q = torch.empty(E, R, C, dtype=torch.uint8, device=w.device)
        sc = torch.empty(E, R // 128, C // 128, dtype=torch.float32, device=w.device)
        if w.numel():
            quantize_e4m3(w.reshape(E * R, C), 128, q, sc, stream=stream)
        out[k] = q
        out[k + "_scale"] = sc
    return out


# --------------------------------------------------------------- whole layer -----

@dataclasses.dataclass
class MoELayer:
    """One layer's parameters and preallocated buffers; ``step()`` runs the whole
    forward pass plus the end-of-step bias update and sequence statistic through the
    C ABI on the current stream (no host synchronisation, no allocation)."""

    T: int
    d: int
    N_r: int
    K_r: int
    N_s: int
    I: int
    G: int
    M: int
    e: torch.Tensor
    b: torch.Tensor
    weights: dict
    n_seq: int = 1
    gamma: float = 0.001
    alpha: float = 0.0001
    want_s: bool = False
    out_dtype: Optional[torch.dtype] = torch.float32   # h' (fp32 keeps the layer output
    # within 2e-2 max-abs: a bf16 store alone errs by up to 0.0156 once |h'| >= 4)
    fp8: bool = False   # expert GEMMs in E4M3: weights quantised here once (128x128
    # blocks), tokens every step (1x128 tiles); routing stays on the bf16 tokens
    gather_rows: bool = False   # bf16: gate/up reads the routed rows' tokens straight
    # from u and the dispatch writes no x_perm (saves the x_perm buffer, T*K_r*d values;
    # backward() then gathers x_perm itself).  Off by default: the gate/up GEMM runs
    # about 2.5 times longer that way

    def __post_init__(self):
        dev, dt = self.e.device, self.e.dtype
        T, K_r, N_r = self.T, self.K_r, self.N_r
        self.shape = make_shape(self.T, self.d, N_r, K_r, self.N_s, self.I, self.G, self.M)
        z = lambda *s, dtype=torch.int32: torch.empty(*s, dtype=dtype, device=dev)
        self.topk_idx = z(T, K_r)
        self.topk_gate = z(T, K_r, dtype=torch.float32)
        self.s_out = z(T, N_r, dtype=torch.float32) if self.want_s else None
        self.seq_p_sum = z(self.n_seq, N_r, dtype=torch.float32)
        self.load = z(N_r)
        self.expert_offset = z(N_r + 1)
        self.perm_token = z(T * K_r)
        self.inv_row = z(T, K_r)
        R = T * K_r + self.N_s * T
        if self.fp8:
            if dt != torch.bfloat16:
                raise ValueError("the FP8 layer takes bf16 tokens and weights")
            u8 = torch.uint8
            self.u_q = z(T, self.d, dtype=u8)
            self.u_scale = z(T, self.d // 128, dtype=torch.float32)
            self.x_perm = z(T * K_r, self.d, dtype=u8)
            self.x_perm_scale = z(T * K_r, self.d // 128, dtype=torch.float32)
            self.h_mid = z(R, self.I, dtype=u8)
            self.h_scale = z(R, self.I // 128, dtype=torch.float32)
            self.ffn_weights = quantize_weights(self.weights)
        else:
            self.x_perm = z(T * K_r, self.d, dtype=dt)
            self.h_mid = z(R, self.I, dtype=dt)
            self.ffn_weights = self.weights
        self.y = z(R, self.d, dtype=dt)
        self.out = z(T, self.d, dtype=self.out_dtype or dt)
        self.stat = z(self.n_seq, dtype=torch.float32)
        self.stat_mean = z(1, dtype=torch.float32)
        self.ws_route = _workspace(route_workspace_bytes(self.shape, self.n_seq), dev)
        # the bias update and the statistic run on a second stream beside the expert FFNs
        self._side = torch.cuda.Stream(device=dev) if dev.type == "cuda" else None
        self.ws_dispatch = _workspace(dispatch_workspace_bytes(self.shape), dev)
        self._gather = self.gather_rows and not self.fp8 and dt == torch.bfloat16
        self._x_perm_current = False

    def step(self, u: torch.Tensor, seq_offsets: torch.Tensor, update_bias: bool = True,
             events: Optional[list] = None, stream=None,
             out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Forward pass h' for the tokens u; then b <- b + gamma*sign(mean - load) and the
        per-sequence statistic.  ``events`` (optional list of 6 CUDA events) are recorded
        between the stages for per-stage timing (6 events).  h' goes to ``out`` (same
        shape and dtype as ``self.out``) when given, else to ``self.out``."""
        sh = self.shape
        out = self.out if out is None else out
        main = stream if stream is not None else torch.cuda.current_stream(self.e.device)
        ev = (lambda i: events[i].record(main)) if events else (lambda i: None)
        ev(0)
        route(u, self.e, self.b, sh, self.topk_idx, self.topk_gate, self.s_out, seq_offsets,
              self.n_seq, self.seq_p_sum, self.ws_route, stream)
        ev(1)
        if self.fp8:
            quantize_e4m3(u, 1, self.u_q, self.u_scale, stream=stream)
            dispatch(self.topk_idx, sh, self.load, self.expert_offset, self.perm_token,
                     self.inv_row, self.u_q, self.x_perm, self.u_scale, self.x_perm_scale,
                     workspace=self.ws_dispatch, stream=stream)
            joined = self._end_of_step(main, seq_offsets, update_bias)
            ev(2)
            expert_gate_up(self.x_perm, self.u_q, self.expert_offset, sh, self.ffn_weights,
                           self.h_mid, self.x_perm_scale, self.u_scale, self.h_scale,
                           stream=stream)
            ev(3)
            expert_down(self.h_mid, self.expert_offset, sh, self.ffn_weights, self.y,
                        self.h_scale, stream=stream)
        else:
            g = self._gather
            dispatch(self.topk_idx, sh, self.load, self.expert_offset, self.perm_token,
                     self.inv_row, None if g else u, None if g else self.x_perm,
                     workspace=self.ws_dispatch, stream=stream)
            self._x_perm_current = not g
            joined = self._end_of_step(main, seq_offsets, update_bias)
            ev(2)
            if g:
                expert_gate_up_gather(u, self.perm_token, self.expert_offset, sh, self.ffn_weights,
                                      self.h_mid, stream=stream)
            else:
                expert_gate_up(self.x_perm, u, self.expert_offset, sh, self.ffn_weights, self.h_mid,
                               stream=stream)
            ev(3)
            expert_down(self.h_mid, self.expert_offset, sh, self.ffn_weights, self.y,
                        stream=stream)
        ev(4)
        combine(u, self.y, self.topk_gate, self.inv_row, sh, out, stream=stream)
        main.wait_event(joined)
        ev(5)
        return out

    def _end_of_step(self, main, seq_offsets, update_bias: bool):
        """b <- b + gamma*sign(mean - load) and the sequence statistic on the side
        stream, once the dispatch has written the loads; returns the event the main
        stream waits on before the step ends (the next step's routing reads b)."""
        forked = torch.cuda.Event()
        forked.record(main)
        self._side.wait_event(forked)
        if update_bias:
            bias_update(self.b, self.load, self.shape, self.gamma, stream=self._side)
        seq_balance_stat(self.seq_p_sum, self.topk_idx, seq_offsets, self.n_seq, self.shape,
                         self.alpha, self.stat, self.stat_mean, stream=self._side)
        joined = torch.cuda.Event()
        joined.record(self._side)
        return joined

    def pipeline(self, u_host: list, out_host: list, seq_offsets: torch.Tensor,
                 load_host: Optional[list] = None, stat_host: Optional[list] = None) -> None:
        """Run one step per host batch: u_host[k] (pinned, [T, d]) in, h' to out_host[k]
        (pinned, like ``self.out``), optionally the loads and per-sequence statistics to
        load_host[k] / stat_host[k].  Three streams overlap the copy-in of batch k+1 and
        the copy-out of batch k-1 with the compute of batch k; the device holds two
        input and two output buffers.  Enqueues everything on the current stream and
        two side streams and returns; the current stream waits for the last copy-out,
        so synchronising it (or the device) completes the run."""
        comp = torch.cuda.current_stream()
        dev = self.e.device
        if not hasattr(self, "_pipe"):
            self._pipe = dict(
                s_in=torch.cuda.Stream(device=dev), s_out=torch.cuda.Stream(device=dev),
                u=[torch.empty(u_host[0].shape, dtype=u_host[0].dtype, device=dev)
                   for _ in range(2)],
                out=[self.out, torch.empty_like(self.out)])
        P = self._pipe
        s_in, s_out = P["s_in"], P["s_out"]
        ev = lambda: torch.cuda.Event()
        in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        for k in range(len(u_host)):
            slot = k & 1
            with torch.cuda.stream(s_in):
                if k >= 2:   # the compute of batch k-2 has finished reading this buffer
                    s_in.wait_event(comp_done[slot])
                P["u"][slot].copy_(u_host[k], non_blocking=True)
                in_ready[slot].record(s_in)
            comp.wait_event(in_ready[slot])
            if k >= 2:       # the copy-out of batch k-2 has finished reading this buffer
                comp.wait_event(out_done[slot])
            self.step(P["u"][slot], seq_offsets, out=P["out"][slot], stream=comp)
            if load_host is not None:
                load_host[k].copy_(self.load, non_blocking=True)
            if stat_host is not None:
                stat_host[k].copy_(self.stat, non_blocking=True)
            comp_done[slot].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[slot])
                out_host[k].copy_(P["out"][slot], non_blocking=True)
                out_done[slot].record(s_out)
        comp.wait_stream(s_out)
        comp.wait_stream(s_in)

    def backward(self, u: torch.Tensor, dh: torch.Tensor, seq_offsets: Optional[torch.Tensor] = None,
                 stream=None) -> dict:
        """Gradients at the selection of the last ``step()`` on the same ``u`` (the layer
        must have been built with ``want_s=True``): of sum(dh * h') plus, with
        ``seq_offsets``, the mean over sequences of the balance loss.  An FP8 layer runs
        its expert GEMMs' backward in E4M3 (moe_backward_fp8).  Returns fp32 tensors "u",
        "e", "w_gate", "w_up", "w_down" (and "ws_*" with shared experts); they and the
        workspace are allocated on the first call and reused."""
        if self.s_out is None:
            raise ValueError("backward() needs the affinities: build the layer with want_s=True")
        dev = self.e.device
        if not hasattr(self, "_grads"):
            keys = ["w_gate", "w_up", "w_down"] + (["ws_gate", "ws_up", "ws_down"] if self.N_s else [])
            g = {k: torch.empty(self.weights[k].shape, dtype=torch.float32, device=dev) for k in keys}
            g["u"] = torch.empty(self.T, self.d, dtype=torch.float32, device=dev)
            g["e"] = torch.empty(self.N_r, self.d, dtype=torch.float32, device=dev)
            self._grads = g
            ws_bytes = (backward_fp8_workspace_bytes if self.fp8 else backward_workspace_bytes)(self.shape, self.n_seq)
            self._bwd_ws = _workspace(ws_bytes, dev)
            if self.fp8:
                self._dgrad_w = fp8_dgrad_weights(self.ffn_weights, self.shape, stream=stream)
        n_seq = self.n_seq if seq_offsets is not None else 0
        if self.fp8:
            backward_fp8(u, self.u_q, self.u_scale, self.e, self.s_out, self.topk_idx, self.topk_gate,
                         self.expert_offset, self.inv_row, self.x_perm, self.x_perm_scale, self.y,
                         self.shape, self.ffn_weights, self._dgrad_w, dh, self._grads, seq_offsets, n_seq,
                         self.alpha if seq_offsets is not None else 0.0, workspace=self._bwd_ws, stream=stream)
            return self._grads
        if not self._x_perm_current:
            # the forward read its rows straight from u: gather x_perm (the same
            # permutation, recomputed from the step's selection)
            dispatch(self.topk_idx, self.shape, self.load, self.expert_offset, self.perm_token,
                     self.inv_row, u, self.x_perm, workspace=self.ws_dispatch, stream=stream)
            self._x_perm_current = True
        backward(u, self.e, self.s_out, self.topk_idx, self.topk_gate, self.expert_offset,
                 self.inv_row, self.x_perm, self.y, self.shape, self.weights, dh, self._grads,
                 seq_offsets, n_seq, self.alpha if seq_offsets is not None else 0.0,
                 workspace=self._bwd_ws, stream=stream)
        return self._grads

    def capture(self, u: torch.Tensor, seq_offsets: torch.Tensor, steps: int = 1,
                events: Optional[list] = None, pre=None, post=None) -> "torch.cuda.CUDAGraph":
        """Capture `steps` consecutive steps (with optional per-step ``pre(k)`` /
        ``post(k)`` callables, e.g. host<->device copies) into one CUDA graph; replaying it
        runs them with no host work per kernel.  Per-step ``events`` must be created with
        ``external=True``.  Call ``step()`` once before capturing (first-use setup)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for k in range(steps):
                if pre is not None:
                    pre(k)
                self.step(u, seq_offsets, events=events[k] if events else None)
                if post is not None:
                    post(k)
        return g
