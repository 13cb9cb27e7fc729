"""E4M3 rounding and the 1x128 / 128x1 / 128x128 fp32-scaled quantisation (CPU oracle).

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``; never by the
library or its Python binding.

The granularity follows the DeepSeek-V3 Technical Report reading guide
(xyznot.com, "Key ideas", FP8 mixed-precision bullet): E4M3 on all tensors,
activations scaled per 1x128 tile, weights per 128x128 block.  The 128x1 tiles (one
column, 128 rows) serve the backward's weight-gradient GEMMs, whose contraction runs
over the rows (tokens): a tile lies along the contraction axis there, as the 1x128
tile does in the forward (see ``moe_backward.layer_backward_fp8``).  The pages fix only
the granularity; the scale rule used here is the plainest one that maps each tile's
largest magnitude onto the format's largest finite value: scale = amax / 448 in
fp32, code = E4M3(x / scale) rounded to nearest-even with saturation, and
scale = 1 for an all-zero tile.

E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
infinities; the largest finite magnitude is 1.75 * 2^8 = 448, the smallest normal
2^-6 and the smallest subnormal 2^-9.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
TILE = 128


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at +-448.

    Works in float64, where every step below is exact: a value a in [2^E, 2^(E+1))
    has 3 fraction bits, so its grid spacing is 2^(E-3); below the smallest normal
    2^-6 the spacing stays 2^-9 (subnormals).
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                      # a = m * 2**ex with m in [0.5, 1)
    E = np.maximum(ex - 1, -6)               # binade exponent, floored at the normal minimum
    quantum = np.ldexp(1.0, E - 3)
    q = np.rint(a / quantum) * quantum       # np.rint rounds half to even
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, x)


def e4m3_encode(v) -> np.ndarray:
    """Bit pattern (uint8) of values that are already on the E4M3 grid."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    _, ex = np.frexp(a)
    E = ex - 1
    normal = a >= 2.0 ** -6
    # normal: a = (1 + m/8) * 2^E, biased exponent E+7 in 1..15
    m_norm = np.where(normal, np.rint(a / np.ldexp(1.0, E) * 8.0 - 8.0), 0)
    e_norm = np.where(normal, E + 7, 0)
    # subnormal: a = m * 2^-9
    m_sub = np.rint(a / 2.0 ** -9)
    m = np.where(normal, m_norm, m_sub).astype(np.int64)
    e = np.where(normal, e_norm, 0).astype(np.int64)
    return (sign | ((e << 3) | m).astype(np.uint8)).astype(np.uint8)


def e4m3_decode(code) -> np.ndarray:
    """Value (float64) of E4M3 bit patterns (NaN patterns are not expected)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    return s * val


def _scales(amax32: np.ndarray) -> np.ndarray:
    amax32 = amax32.astype(np.float32)
    sc = (amax32 / np.float32(E4M3_MAX)).astype(np.float32)   # one fp32 rounding
    return np.where(amax32 > 0, sc, np.float32(1.0)).astype(np.float32)


def quantize_1x128(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-row, per-128-column tile quantisation of an fp32 matrix [R, C].

    Returns (q, scale): q [R, C] float64 values on the E4M3 grid, scale [R, C/128]
    fp32.  x / scale is formed in fp32 (one rounding) before the E4M3 rounding, so
    the code depends on nothing but fp32 arithmetic.
    """
    x = np.asarray(x, dtype=np.float32)
    R, C = x.shape
    if C % TILE:
        raise ValueError("column count must be a multiple of 128")
    tiles = x.reshape(R, C // TILE, TILE)
    scale = _scales(np.abs(tiles).max(axis=-1))
    q = e4m3_round((tiles / scale[..., None]).astype(np.float32))
    return q.reshape(R, C), scale


def quantize_128x128(w) -> tuple[np.ndarray, np.ndarray]:
    """Per-128x128-block quantisation of fp32 weights [..., R, C].

    Returns (q, scale): q with w's shape (E4M3 grid values, float64) and scale
    [..., R/128, C/128] fp32.
    """
    w = np.asarray(w, dtype=np.float32)
    *lead, R, C = w.shape
    if R % TILE or C % TILE:
        raise ValueError("both matrix dimensions must be multiples of 128")
    blocks = w.reshape(*lead, R // TILE, TILE, C // TILE, TILE)
    amax = np.abs(blocks).max(axis=(-3, -1))                   # [..., R/128, C/128]
    scale = _scales(amax)
    q = e4m3_round((blocks / scale[..., :, None, :, None]).astype(np.float32))
    return q.reshape(w.shape), scale


def dequantize_1x128(q, scale) -> np.ndarray:
    q = np.asarray(q, dtype=np.float64)
    R, C = q.shape
    return (q.reshape(R, C // TILE, TILE) * scale.astype(np.float64)[..., None]).reshape(R, C)


def dequantize_128x128(q, scale) -> np.ndarray:
    q = np.asarray(q, dtype=np.float64)
    *lead, R, C = q.shape
    blocks = q.reshape(*lead, R // TILE, TILE, C // TILE, TILE)
    return (blocks * scale.astype(np.float64)[..., :, None, :, None]).reshape(q.shape)


def quantize_128x1(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-column, per-128-row tile quantisation of an fp32 matrix [n, C] whose rows
    are the tokens of one expert segment.

    The rows are cut into ceil(n/128) tiles from the first row; the last tile may be
    short (its amax is over its own rows).  Returns (q, scale): q [n, C] float64
    values on the E4M3 grid, scale [ceil(n/128), C] fp32.
    """
    x = np.asarray(x, dtype=np.float32)
    n, C = x.shape
    nb = -(-n // TILE)
    padded = np.zeros((nb * TILE, C), dtype=np.float32)
    padded[:n] = x
    tiles = padded.reshape(nb, TILE, C)
    scale = _scales(np.abs(tiles).max(axis=1))                   # [nb, C]
    q = e4m3_round((tiles / scale[:, None, :]).astype(np.float32))
    return q.reshape(nb * TILE, C)[:n], scale


def dequantize_128x1(q, scale) -> np.ndarray:
    q = np.asarray(q, dtype=np.float64)
    n = q.shape[0]
    rows = np.repeat(scale.astype(np.float64), TILE, axis=0)[:n]
    return q * rows


def bf16_round(x) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even), returned as fp32."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return b.astype(np.uint32).view(np.float32)
