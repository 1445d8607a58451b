"""Rounding to the formats the draft-head step stores: fp32, bf16 and FP8 E4M3.

Oracle (test infrastructure only; see ``oracle/__init__.py``).

Sources:
* bf16 rounding of residual adds and of SiLU(g) ("rounds each residual add once"):
  TFE draft head page (#42), commit "eagle.zig is split ... eagle_ref.py (rnd=True)".
* FP8 "e4m3 with an fp32 scale a row ... round to nearest even": TFE draft head page (#42),
  update "main3x heads, pass kernels, FP8 linears".
* "E4M3 codes with E8M0 scales in 32x32 blocks": DSpark FP8 head page (#3296), "FP8 draft head".

Reading (the pages say "e4m3" without naming the variant): E4M3 is the "fn" variant of the OCP
FP8 formats: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities, code 0x7F/0xFF
is NaN, the largest finite magnitude is 448 (the divisor the pages' per-row scale uses). Encoding
rounds to the nearest finite value with ties to the even code and saturates to +-448 (values past
448 are nearer to 448 than to any other finite code, so "nearest finite" already saturates).
"""
import numpy as np

# Largest finite bf16: (2 - 2^-7) * 2^127.
BF16_MAX = float.fromhex("0x1.fep127")


def fl32(x):
    """Round float64 values to fp32 (IEEE round to nearest even), returned as float32."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def round_bf16(x):
    """Round to the nearest bf16 value, ties to even; returned as float64.

    bf16 keeps 8 significant bits and fp32's exponent range; below 2^-126 its spacing is the
    fixed subnormal step 2^-133. Values at or past the midpoint above BF16_MAX become inf.
    NaN and +-inf pass through. This is a single rounding from the float64 input.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x)
    xf = x[fin]
    _, e = np.frexp(xf)                      # xf = m * 2^e with 0.5 <= |m| < 1
    q = np.maximum(e - 8, -133)              # weight of the last kept bit
    r = np.rint(np.ldexp(xf, -q))            # exact power-of-two scaling; rint = ties to even
    y = np.ldexp(r, q)
    big = np.abs(y) > BF16_MAX
    y[big] = np.copysign(np.inf, y[big])
    out[fin] = y
    return out


def _e4m3_value(code):
    """Value of one E4M3 byte from the format's definition (NaN for 0x7F/0xFF)."""
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6        # subnormal: m * 2^-9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_DECODE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
# Codes 0x00..0x7E are the non-negative finite values, in increasing order of value.
_E4M3_POS = E4M3_DECODE[:0x7F].copy()


def e4m3_decode(codes):
    """Decode E4M3 bytes to float64 (exact)."""
    return E4M3_DECODE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x):
    """Encode to E4M3: nearest finite value, ties to the even code, sign kept (-0 -> 0x80).

    NaN encodes to 0x7F. Magnitudes past 448 (and inf) saturate to 448.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    hi = np.minimum(np.searchsorted(_E4M3_POS, a, side="left"), 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(take_hi, hi, lo).astype(np.uint8)
    code = mag | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)
