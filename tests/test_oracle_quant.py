"""Pins of the oracle's FP8 quantisation: hand-derived examples of the page's rules, closed forms,
error bounds and invariants."""
import json
import os

import numpy as np
import pytest
import torch

from oracle.numerics import E4M3_DECODE, e4m3_decode
from oracle.quant import (block32_exponent, dequant_fp8_block32, dequant_fp8_row,
                          quant_fp8_block32, quant_fp8_row)
from synth import inputs

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def bf16_matrix(n, k, std, tid):
    return inputs.normal_bf16((n, k), std, tid).float().numpy()


def all_positive_bf16():
    v = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    return v.astype(np.float64)


# ---- per-row ------------------------------------------------------------------------------------

def test_row_worked_examples():
    for ex in GOLD["worked_row_quant"]:
        w = np.array([ex["w"]], dtype=np.float32)
        codes, s = quant_fp8_row(w)
        assert list(codes[0]) == ex["codes"]
        if "s" in ex:
            assert s[0] == np.float32(ex["s"])
    assert GOLD["row_scale_divisor"]["value"] == 448


def test_row_amax_code_is_448():
    w = bf16_matrix(64, 256, 0.02, 83)
    codes, s = quant_fp8_row(w)
    arg = np.argmax(np.abs(w), axis=1)
    top = codes[np.arange(64), arg]
    assert np.all((top & 0x7F) == 0x7E)
    assert np.array_equal(top >> 7, (w[np.arange(64), arg] < 0).astype(np.uint8))


def test_row_dequant_error_bound():
    # |dequant - w| <= s * half the E4M3 spacing at the code's magnitude (plus one fp32 ulp of w/s).
    w = bf16_matrix(32, 512, 0.02, 84)
    codes, s = quant_fp8_row(w)
    deq = dequant_fp8_row(codes, s)
    q = np.abs(w.astype(np.float64) / s[:, None])
    e = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
    half_ulp = np.exp2(e - 4)                      # 3 mantissa bits -> spacing 2^(e-3)
    bound = s[:, None] * (half_ulp + q * 2.0 ** -23)
    assert np.all(np.abs(deq - w) <= bound)


def test_row_sign_symmetry_and_zero_row():
    w = bf16_matrix(8, 64, 0.02, 85)
    c1, s1 = quant_fp8_row(w)
    c2, s2 = quant_fp8_row(-w)
    assert np.array_equal(s1, s2) and np.array_equal(c2, c1 ^ 0x80)
    z = np.zeros((2, 32), np.float32)
    z[1, 3] = -0.0
    cz, sz = quant_fp8_row(z)
    assert np.all(sz == 0) and np.all((cz & 0x7F) == 0)
    assert np.all(dequant_fp8_row(cz, sz) == 0)


def test_row_against_torch_float8_cast():
    # The rule written as torch ops: fp32 amax/448, fp32 division, float8_e4m3fn cast (no value of
    # w/s exceeds 448 by more than rounding, where the cast and the saturating encoder agree).
    w = bf16_matrix(128, 256, 0.02, 86)
    codes, s = quant_fp8_row(w)
    t = torch.from_numpy(w)
    ts = t.abs().amax(dim=1) / 448.0
    tq = (t / ts[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(s, ts.numpy()) and np.array_equal(codes, tq)


# ---- 32x32 blocks -------------------------------------------------------------------------------

def test_block_exponent_closed_form_exhaustive():
    # amax = m * 2^E with 1 <= m < 2: e = E - 8 + (m > 1.75), since 448 = 1.75 * 2^8.
    amax = all_positive_bf16()
    e = block32_exponent(amax)
    m, E = np.frexp(amax)                 # amax = m * 2^E, 0.5 <= m < 1
    m, E = m * 2, E - 1
    closed = E - 8 + (m > 1.75)
    assert np.array_equal(e, closed)
    assert np.all(amax <= 448.0 * np.exp2(e)) and np.all(amax > 448.0 * np.exp2(e - 1))


def test_block_worked_examples():
    for ex in GOLD["worked_block_quant"]:
        w = np.zeros((32, 32), np.float32)
        w[5, 7] = ex["amax"]
        codes, sb = quant_fp8_block32(w)
        assert sb[0, 0] == ex["scale_byte"]
        assert codes[5, 7] == ex["code_of_amax"]
        assert np.all(codes[w == 0] == 0)


def test_block_max_code_and_no_saturation():
    w = bf16_matrix(128, 256, 0.02, 87)
    w[:32, :32] *= 1000.0
    w[32:64, 32:64] = 0.0
    codes, sb = quant_fp8_block32(w)
    mags = np.abs(e4m3_decode(codes)).reshape(4, 32, 8, 32).max(axis=(1, 3))
    amax = np.abs(w).reshape(4, 32, 8, 32).max(axis=(1, 3))
    nz = amax > 0
    assert np.all(mags[nz] >= 224) and np.all(mags[nz] <= 448)
    assert sb[1, 1] == 0 and mags[1, 1] == 0
    # no code saturates: every scaled value is within the finite range before rounding
    scaled = np.abs(w.astype(np.float64)).reshape(4, 32, 8, 32) / np.exp2(
        sb.astype(np.float64) - 127)[:, None, :, None]
    assert scaled.max() <= 448.0


def test_block_exact_roundtrip_of_representable_values():
    codes = np.random.default_rng([0, 88, 0]).integers(0, 256, size=(64, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E
    codes[0, 0] = 0x7E                          # every block gets a full-range element
    for bi in range(2):
        for bj in range(2):
            codes[bi * 32, bj * 32] = 0x7E
    for scale in (-20, 0, 5):
        w = e4m3_decode(codes) * 2.0 ** scale
        c2, sb = quant_fp8_block32(w.astype(np.float32))
        assert np.array_equal(dequant_fp8_block32(c2, sb), w)


def test_block_storage_size_matches_page():
    f = GOLD["fp8_head_bytes"]
    v, h, b = f["vocab"], f["hidden"], f["block"]
    assert v * h == f["codes_bytes"] and (v // b) * (h // b) == f["scale_bytes"]
    assert f["codes_bytes"] + f["scale_bytes"] == f["total_bytes"]
    assert round(f["total_bytes"] / 1e9, 2) == f["page_gb"]
    assert E4M3_DECODE[0x7E] == 448.0


def test_block32_interleaved_layout_worked_example_and_round_trip():
    """The interleaved layout on a row whose code equals its column: each 16-byte piece holds
    8 columns of the first 32-wide block, then the same 8 of the second (hand-written)."""
    from oracle.quant import block32_deinterleave, block32_interleave
    row = np.arange(128).reshape(1, 128)
    want = ([0, 1, 2, 3, 4, 5, 6, 7, 32, 33, 34, 35, 36, 37, 38, 39,
             8, 9, 10, 11, 12, 13, 14, 15, 40, 41, 42, 43, 44, 45, 46, 47,
             16, 17, 18, 19, 20, 21, 22, 23, 48, 49, 50, 51, 52, 53, 54, 55,
             24, 25, 26, 27, 28, 29, 30, 31, 56, 57, 58, 59, 60, 61, 62, 63])
    got = block32_interleave(row)[0].tolist()
    assert got[:64] == want
    assert got[64:] == [v + 64 for v in want]
    codes = np.random.default_rng([0, 990, 0]).integers(0, 256, size=(96, 320)).astype(np.uint8)
    il = block32_interleave(codes)
    assert np.array_equal(block32_deinterleave(il), codes)
    assert not np.array_equal(il, codes)
    with pytest.raises(ValueError):
        block32_interleave(codes[:, :96])
