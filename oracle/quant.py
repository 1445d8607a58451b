"""FP8 E4M3 quantisation of a bf16 weight matrix W[n][k] (row-major, one output feature a row).

Oracle (test infrastructure only; see ``oracle/__init__.py``).
"""
import numpy as np

from .numerics import e4m3_decode, e4m3_encode

E4M3_MAX = np.float32(448.0)


def quant_fp8_row(w):
    """Per-row FP8: ``s_n = fl32(amax_n / 448)``, ``code = e4m3(fl32(w / s_n))``.

    Follows the TFE draft head page (#42), update "main3x heads, pass kernels, FP8 linears": the
    head's linears in e4m3 with an fp32 scale a row, "scale = row absmax / 448, round to nearest
    even, from the bf16 weight".

    Readings: the quotient is an IEEE fp32 division by s (as written), rounded to fp32 and then
    to E4M3 (two roundings, as an fp32 torch division followed by a cast would do). A row of zeros
    has s = 0 and keeps its zeros (signs kept), so dequantisation gives 0 and never NaN.
    Weights are taken to be finite.

    Args: w: [n][k] array of bf16-representable values.
    Returns: (codes uint8 [n][k], s float32 [n]).
    """
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w32), axis=1)
    s = (amax / E4M3_MAX).astype(np.float32)                     # fp32 IEEE division
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.where((s > 0)[:, None], w32 / safe[:, None], w32)       # fp32 IEEE division
    return e4m3_encode(q.astype(np.float32)), s


def block32_exponent(amax):
    """Smallest integer e with ``amax <= 448 * 2^e`` (exact comparisons), for amax > 0.

    Reading (the DSpark FP8 head page (#3296), "FP8 draft head", names E8M0 scales per 32x32 block
    but not the exponent rule): the block scale is the smallest power of two that keeps every
    code of the block within the E4M3 range, in the spirit of the per-row rule ``amax / 448``
    (no code saturates).
    """
    amax = np.asarray(amax, dtype=np.float64)
    e = np.floor(np.log2(amax)) - 10.0        # a start below the answer
    while True:
        low = amax > 448.0 * np.exp2(e)       # 448 * 2^e is exact in float64
        if not low.any():
            return e.astype(np.int64)
        e = e + low


def quant_fp8_block32(w):
    """FP8 with E8M0 (power-of-two) scales per 32x32 block.

    Follows the DSpark FP8 head page (#3296), "FP8 draft head": "E4M3 codes with E8M0 scales in
    32x32 blocks", made from the bf16 head at load.

    The stored scale byte of block (i, j) is ``clamp(e + 127, 0, 254)`` with e from
    ``block32_exponent`` of the block's max |w|; an all-zero block stores byte 0. Codes are
    ``e4m3(w * 2^-(byte - 127))``; the scaling is exact, so each code is a single rounding.

    Args: w: [n][k] bf16-representable values, n and k multiples of 32.
    Returns: (codes uint8 [n][k], scale bytes uint8 [n/32][k/32]).
    """
    w64 = np.asarray(w, dtype=np.float64)
    n, k = w64.shape
    assert n % 32 == 0 and k % 32 == 0
    blocks = w64.reshape(n // 32, 32, k // 32, 32)
    amax = np.abs(blocks).max(axis=(1, 3))
    byte = np.zeros(amax.shape, dtype=np.int64)
    nz = amax > 0
    if nz.any():
        byte[nz] = np.clip(block32_exponent(amax[nz]) + 127, 0, 254)
    scale_inv = np.exp2(-(byte - 127).astype(np.float64))
    q = blocks * scale_inv[:, None, :, None]
    codes = e4m3_encode(q).reshape(n, k)
    return codes, byte.astype(np.uint8)


def dequant_fp8_row(codes, s):
    """Exact dequantised weights (float64) of the per-row form."""
    return e4m3_decode(codes) * np.asarray(s, dtype=np.float64)[:, None]


def dequant_fp8_block32(codes, scale_bytes):
    """Exact dequantised weights (float64) of the 32x32-block form."""
    codes = np.asarray(codes)
    n, k = codes.shape
    sc = np.exp2(np.asarray(scale_bytes, dtype=np.float64) - 127.0)
    full = np.repeat(np.repeat(sc, 32, axis=0), 32, axis=1)
    return e4m3_decode(codes) * full


def block32_interleave(codes):
    """Plain row-major block-32 codes [n][k] (k % 64 == 0) -> this library's interleaved layout:
    in each 64-column step c, byte 64c + 16t + 8b + e holds column 64c + 32b + 8t + e
    (t = 0..3, b = 0..1, e = 0..7). A layout of this library (the pages fix none); the values are
    those of quant_fp8_block32."""
    c = np.asarray(codes)
    n, k = c.shape
    if k % 64:
        raise ValueError("k must be a multiple of 64")
    # [n][step][b][t][e] -> [n][step][t][b][e]
    return c.reshape(n, k // 64, 2, 4, 8).transpose(0, 1, 3, 2, 4).reshape(n, k)


def block32_deinterleave(codes):
    """The inverse of block32_interleave."""
    c = np.asarray(codes)
    n, k = c.shape
    return c.reshape(n, k // 64, 4, 2, 8).transpose(0, 1, 3, 2, 4).reshape(n, k)
