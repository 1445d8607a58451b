"""Pins of the oracle's head GEMV: exact rational arithmetic on tiny shapes, one-hot columns,
linearity, duplicate rows, FP8 dequantisation, and the single rounding of the residual add."""
from fractions import Fraction

import numpy as np

from oracle.gemv import (OUT_ADD_BF16, OUT_BF16, OUT_F32, W_BF16, W_FP8_BLOCK32, W_FP8_ROW, gemv,
                         gemv_abs_scale, gemv_acc)
from oracle.numerics import e4m3_decode, round_bf16
from oracle.quant import quant_fp8_block32, quant_fp8_row
from synth import inputs


def small(n, k, r, tid=90):
    w = inputs.normal_bf16((n, k), 0.02, tid).float().numpy()
    x = inputs.normal_bf16((r, k), 1.0, tid + 1).float().numpy()
    return w, x


def test_exact_rational_dot_products():
    w, x = small(24, 48, 3)
    acc = gemv_acc(w, x)
    for r in range(3):
        for n in range(24):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(w[n], x[r]))
            err = abs(Fraction(acc[r, n]) - exact)
            scale = sum(abs(Fraction(float(a)) * Fraction(float(b))) for a, b in zip(w[n], x[r]))
            assert err <= scale * Fraction(1, 2 ** 50)


def test_one_hot_selects_a_column_exactly():
    w, _ = small(64, 32, 1)
    for j in (0, 7, 31):
        x = np.zeros((2, 32), np.float32)
        x[0, j] = 1.0
        x[1, j] = -2.0
        y = gemv(w, x, out_mode=OUT_F32)
        assert np.array_equal(y[0], w[:, j]) and np.array_equal(y[1], -2 * w[:, j])


def test_linearity_zero_and_duplicates():
    w, x = small(40, 64, 4)
    w[7] = w[30]
    y = gemv_acc(w, x)
    assert np.array_equal(y[:, 7], y[:, 30])
    assert np.allclose(gemv_acc(w, 2 * x), 2 * y, rtol=0, atol=1e-15)
    assert np.allclose(gemv_acc(w, x[:1] + x[1:2]), y[:1] + y[1:2], rtol=0, atol=1e-14)
    assert np.all(gemv_acc(w, np.zeros_like(x)) == 0)


def test_fp8_forms_equal_gemv_over_dequantised_weights():
    w, x = small(64, 64, 2)
    codes, s = quant_fp8_row(w)
    deq = e4m3_decode(codes) * s.astype(np.float64)[:, None]
    assert np.array_equal(gemv_acc(codes, x, W_FP8_ROW, s), x.astype(np.float64) @ deq.T)
    cb, sb = quant_fp8_block32(w)
    blocks = e4m3_decode(cb).reshape(2, 32, 2, 32) * np.exp2(
        sb.astype(np.float64) - 127)[:, None, :, None]
    deqb = blocks.reshape(64, 64)
    # the block form as the sum over 32-wide k blocks of scale * partial sum
    xb = x.astype(np.float64)
    manual = np.zeros((2, 64))
    for kb in range(2):
        sl = slice(32 * kb, 32 * kb + 32)
        part = xb[:, sl] @ e4m3_decode(cb)[:, sl].T
        manual += part * np.repeat(np.exp2(sb[:, kb].astype(np.float64) - 127), 32)[None, :]
    assert np.allclose(gemv_acc(cb, x, W_FP8_BLOCK32, sb), manual, rtol=1e-15, atol=0)
    assert np.array_equal(gemv_acc(cb, x, W_FP8_BLOCK32, sb), xb @ deqb.T)


def test_output_modes():
    w, x = small(32, 64, 2)
    acc = gemv_acc(w, x)
    assert np.array_equal(gemv(w, x, out_mode=OUT_F32), acc.astype(np.float32))
    assert np.array_equal(gemv(w, x, out_mode=OUT_BF16),
                          round_bf16(acc.astype(np.float32).astype(np.float64)))
    res = inputs.normal_bf16((2, 32), 1.0, 95).float().numpy()
    assert np.array_equal(gemv(w, x, out_mode=OUT_ADD_BF16, res=res), round_bf16(res + acc))


def test_add_bf16_rounds_once():
    # res = 1, acc = 2^-8 + 2^-40: the exact sum is above the bf16 tie, so it rounds up; an fp32
    # intermediate would sit on the tie and round down.
    w = np.zeros((1, 8), np.float32)
    w[0, 0] = 2.0 ** -8
    w[0, 1] = 2.0 ** -40
    x = np.ones((1, 8), np.float32)
    y = gemv(w, x, out_mode=OUT_ADD_BF16, res=np.ones((1, 1)))
    assert y[0, 0] == 1.0 + 2 ** -7


def test_abs_scale_bounds_acc():
    w, x = small(32, 64, 3)
    assert np.all(np.abs(gemv_acc(w, x)) <= gemv_abs_scale(w, x))


def test_w8a8_activation_rule_matches_torch_float8_and_closed_forms():
    """W8A8: each activation row quantised by the weights' row rule; checked against torch's own
    float8_e4m3fn cast of x / (amax / 448), a one-hot closed form and a zero row."""
    import torch

    from oracle.gemv import act_e4m3, gemv_acc
    x = inputs.normal_bf16((6, 4096), 1.5, 980).float().numpy()
    t = torch.from_numpy(x)
    s = t.abs().amax(dim=1, keepdim=True) / 448.0
    ref = (t / s).to(torch.float8_e4m3fn).double() * s.double()
    assert np.array_equal(act_e4m3(x), ref.numpy())
    w = inputs.normal_bf16((64, 4096), 0.02, 981).float().numpy()
    onehot = np.zeros((1, 4096), np.float32)
    onehot[0, 77] = 3.0
    got = gemv_acc(w, onehot, W_BF16, None, act_fp8=True)[0]
    sx = np.float64(np.float32(np.float32(3.0) / np.float32(448.0)))
    assert np.array_equal(got, w[:, 77].astype(np.float64) * 448.0 * sx)
    assert np.all(gemv_acc(w, np.zeros((1, 4096), np.float32), W_BF16, None, act_fp8=True) == 0)
