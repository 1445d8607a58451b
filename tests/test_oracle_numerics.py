"""Pins of the oracle's rounding helpers (bf16, E4M3) to the formats' definitions, to hand-derived
values and to library casts on the cases where those casts are defined the same way."""
import json
import os

import numpy as np
import pytest
import torch

from oracle.numerics import E4M3_DECODE, e4m3_decode, e4m3_encode, fl32, round_bf16

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def all_bf16_values():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    return bits.view(np.float32)


# ---- bf16 ---------------------------------------------------------------------------------------

def test_bf16_hand_values():
    one = 1.0
    assert round_bf16(one + 2 ** -8) == 1.0                       # tie -> even (down)
    assert round_bf16(one + 3 * 2 ** -8) == 1.0 + 2 ** -6          # tie -> even (up)
    assert round_bf16(one + 2 ** -8 + 2 ** -40) == 1.0 + 2 ** -7   # above the tie: up
    assert round_bf16(-(one + 2 ** -8 + 2 ** -40)) == -(1.0 + 2 ** -7)
    assert np.signbit(round_bf16(-0.0))
    assert round_bf16(2.0 ** -133) == 2.0 ** -133                  # smallest subnormal
    assert round_bf16(2.0 ** -134) == 0.0                          # half of it: tie to even zero
    assert round_bf16(3 * 2.0 ** -134) == 2 * 2.0 ** -133
    assert round_bf16(float.fromhex("0x1.fep127")) == float.fromhex("0x1.fep127")
    assert np.isinf(round_bf16(2.0 ** 128 - 2.0 ** 119))           # midpoint above max -> inf
    assert round_bf16(2.0 ** 128 - 2.0 ** 119 - 2.0 ** 100) == float.fromhex("0x1.fep127")
    assert np.isnan(round_bf16(np.nan)) and np.isinf(round_bf16(np.inf))


def test_bf16_single_rounding_differs_from_double():
    # 1 + 2^-8 + 2^-40: the fp32 value is the tie 1 + 2^-8, which a second rounding sends to 1.
    x = 1.0 + 2 ** -8 + 2 ** -40
    assert float(fl32(x)) == 1.0 + 2 ** -8
    assert round_bf16(float(fl32(x))) == 1.0
    assert round_bf16(x) == 1.0 + 2 ** -7


def test_bf16_matches_torch_cast_on_fp32_inputs():
    rng = np.random.default_rng([0, 81, 0])
    bits = rng.integers(0, 1 << 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ours = round_bf16(x)
    lib = torch.from_numpy(x.copy()).to(torch.bfloat16).double().numpy()
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all()
    assert (np.signbit(ours) == np.signbit(lib)).all()


def test_bf16_identity_on_bf16_values():
    v = all_bf16_values()
    v = v[np.isfinite(v)]
    out = round_bf16(v)
    assert np.array_equal(out, v.astype(np.float64))


# ---- E4M3 ---------------------------------------------------------------------------------------

def test_e4m3_hand_codes():
    for code, val in GOLD["e4m3_codes"].items():
        if not code.startswith("0x"):
            continue
        c = int(code, 16)
        assert E4M3_DECODE[c] == val
        if c == 0x80:
            assert np.signbit(E4M3_DECODE[c])
    assert np.isnan(E4M3_DECODE[0x7F]) and np.isnan(E4M3_DECODE[0xFF])
    assert np.isfinite(E4M3_DECODE).sum() == 254


def test_e4m3_decode_matches_torch_float8():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    same = (lib == E4M3_DECODE) | (np.isnan(lib) & np.isnan(E4M3_DECODE))
    assert same.all()
    assert (np.signbit(lib) == np.signbit(E4M3_DECODE))[np.isfinite(lib)].all()


def test_e4m3_decode_encode_roundtrip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(e4m3_encode(e4m3_decode(codes)), codes)


def _brute_encode(x):
    """Linear scan over the 254 finite codes: nearest value, ties to the even code, sign kept."""
    if np.isnan(x):
        return 0x7F
    a = abs(x)
    best, best_d = None, None
    for c in range(0x7F):
        d = abs(a - E4M3_DECODE[c])
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best | (0x80 if np.signbit(x) else 0)


def test_e4m3_encode_brute_force_midpoints_and_samples():
    pos = E4M3_DECODE[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    probes = list(mids) + list(np.nextafter(mids, 0)) + list(np.nextafter(mids, 1e9))
    probes += list(pos) + [448.0, 449.0, 463.9, 464.0, 480.0, 1e6, np.inf, 2 ** -10, 2 ** -11,
                           3 * 2 ** -10, 1e-30, 0.0]
    rng = np.random.default_rng([0, 82, 0])
    probes += list(np.exp2(rng.uniform(-12, 10, 3000)))
    probes = np.array(probes, dtype=np.float64)
    probes = np.concatenate([probes, -probes, [np.nan, -0.0]])
    ours = e4m3_encode(probes)
    brute = np.array([_brute_encode(float(x)) for x in probes], dtype=np.uint8)
    assert np.array_equal(ours, brute)


def test_e4m3_encode_matches_torch_cast_inside_range():
    # torch's float8_e4m3fn cast rounds to nearest even; inside +-448 it is the same function.
    v = all_bf16_values().astype(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 448)]
    lib = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(v), lib)


def test_e4m3_saturates_and_keeps_sign():
    assert e4m3_encode(1e30) == 0x7E and e4m3_encode(-1e30) == 0xFE
    assert e4m3_encode(np.inf) == 0x7E and e4m3_encode(-np.inf) == 0xFE
    assert e4m3_encode(-0.0) == 0x80 and e4m3_encode(-1e-9) == 0x80 and e4m3_encode(1e-9) == 0x00
    assert e4m3_encode(np.nan) == 0x7F
    x = np.exp2(np.linspace(-12, 9, 999))
    assert np.array_equal(e4m3_encode(-x), e4m3_encode(x) | 0x80)
