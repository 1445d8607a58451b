"""Few-row head GEMV: ``acc[r][n] = sum_k W[n][k] * x[r][k]`` and its output modes.

Oracle (test infrastructure only; see ``oracle/__init__.py``).

Follows the TFE draft head page (#42), commit "pass kernels and FP8 linears" (GEMV over bf16 and
e4m3 weights "for up to 16 rows (out bf16, fp32, or added to bf16)"), and the commit "eagle.zig is
split ..." (each residual add "rounded once"). The dot products are taken in float64, in which
every bf16 x bf16, e4m3 x bf16 and bf16 x fp32 product is exact, so ``acc`` is the real result up
to float64 rounding; the oracle then rounds only where the method rounds.

Reading (the pages do not say whether the FP8 path quantises activations): activations stay bf16
(or fp32) and only weights are FP8 (W8A16), with fp32 accumulation. The W8A8 form (DSpark FP8 head
page: the Metal pass keeps "act_quant rows") quantises each activation row by the weights' row rule
(s = fl32(amax / 448), code = e4m3(fl32(x / s))) and multiplies the decoded values exactly.
"""
import numpy as np

from .numerics import fl32, round_bf16
from .quant import dequant_fp8_block32, dequant_fp8_row, quant_fp8_row

W_BF16, W_FP8_ROW, W_FP8_BLOCK32 = 0, 1, 2
OUT_NONE, OUT_F32, OUT_BF16, OUT_ADD_BF16 = 0, 1, 2, 3


def weights_f64(w, wfmt, scales=None):
    """The weight matrix as exact float64 values (dequantised for the FP8 forms)."""
    if wfmt == W_BF16:
        return np.asarray(w, dtype=np.float64)
    if wfmt == W_FP8_ROW:
        return dequant_fp8_row(w, scales)
    if wfmt == W_FP8_BLOCK32:
        return dequant_fp8_block32(w, scales)
    raise ValueError(wfmt)


def act_e4m3(x):
    """Activation rows after the W8A8 quantisation: the exact values s_r * dec(code) (float64)."""
    codes, s = quant_fp8_row(np.atleast_2d(np.asarray(x, dtype=np.float32)))
    return dequant_fp8_row(codes, s)


def gemv_acc(w, x, wfmt=W_BF16, scales=None, act_fp8=False):
    """float64 ``acc[r][n]`` for x [R][K] against W [N][K] (codes for the FP8 forms); act_fp8
    quantises the activation rows first (W8A8)."""
    wd = weights_f64(w, wfmt, scales)
    xv = act_e4m3(x) if act_fp8 else np.asarray(x, dtype=np.float64)
    return xv @ wd.T


def gemv_abs_scale(w, x, wfmt=W_BF16, scales=None, act_fp8=False):
    """``S[r][n] = sum_k |W[n][k] * x[r][k]|``: the magnitude that bounds the rounding error of an
    fp32 dot product; the fp32-accumulation tolerance is stated relative to it."""
    wd = np.abs(weights_f64(w, wfmt, scales))
    xv = act_e4m3(x) if act_fp8 else np.asarray(x, dtype=np.float64)
    return np.abs(xv) @ wd.T


def gemv(w, x, wfmt=W_BF16, scales=None, out_mode=OUT_F32, res=None, act_fp8=False):
    """The GEMV's output in the requested mode.

    F32: ``fl32(acc)``. BF16: ``bf16(fl32(acc))`` (fp32 sums, then the output cast).
    ADD_BF16: ``bf16(res + acc)``, one rounding of the exact sum (the residual add "rounded once").
    NONE: returns None.
    """
    acc = gemv_acc(w, x, wfmt, scales, act_fp8)
    if out_mode == OUT_NONE:
        return None
    if out_mode == OUT_F32:
        return fl32(acc)
    if out_mode == OUT_BF16:
        return round_bf16(fl32(acc).astype(np.float64))
    if out_mode == OUT_ADD_BF16:
        return round_bf16(np.asarray(res, dtype=np.float64) + acc)
    raise ValueError(out_mode)
