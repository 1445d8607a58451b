"""Planted controls: a plausible mistake is planted in a copy of an oracle function (on the CPU),
and the check that guards that function must catch it. CPU controls exercise the oracle's pins;
GPU controls show the parity comparisons against the CUDA path would fail on the mistaken oracle."""
import numpy as np
import pytest
import torch

from helpers import (NORM_REL, assert_bf16_rounding, check_window_attn, gemv_bf16_err, need_gpu,
                     np32)
from oracle import attn as oattn
from oracle import gemv as og
from oracle import numerics
from oracle.accept import accept
from oracle.layer import rmsnorm_rows
from oracle.quant import quant_fp8_block32, quant_fp8_row
from oracle.topk import order, topk
from synth import inputs


# ---- mutants ------------------------------------------------------------------------------------

def encode_ties_away(x):
    """E4M3 with ties rounded away from zero instead of to even."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    pos = numerics.E4M3_DECODE[:0x7F]
    hi = np.minimum(np.searchsorted(pos, a, side="left"), 0x7E)
    lo = np.maximum(hi - 1, 0)
    take_hi = (pos[hi] - a) <= (a - pos[lo])
    code = np.where(take_hi, hi, lo).astype(np.uint8) | np.where(np.signbit(x), 0x80, 0).astype(
        np.uint8)
    return code


def quant_row_multiply(w):
    """Row FP8 with w * (448 / amax) instead of w / (amax / 448)."""
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w32), axis=1)
    s = (amax / np.float32(448)).astype(np.float32)
    inv = (np.float32(448) / np.where(amax > 0, amax, 1)).astype(np.float32)
    return numerics.e4m3_encode((w32 * inv[:, None]).astype(np.float32)), s


def block_exponent_ocp(w):
    """Block FP8 with the OCP-MX exponent floor(log2 amax) - 8 (saturating)."""
    w64 = np.asarray(w, dtype=np.float64)
    n, k = w64.shape
    b = w64.reshape(n // 32, 32, k // 32, 32)
    amax = np.abs(b).max(axis=(1, 3))
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1))) - 8, -127)
    byte = np.clip(e + 127, 0, 254).astype(np.int64)
    q = b * np.exp2(-(byte - 127).astype(np.float64))[:, None, :, None]
    return numerics.e4m3_encode(q).reshape(n, k), byte.astype(np.uint8)


def topk_higher_id(logits, k):
    """Top-k whose ties go to the higher id."""
    lg = np.atleast_2d(np.asarray(logits, dtype=np.float32))
    ids = np.arange(lg.shape[1])
    out = []
    for r in range(lg.shape[0]):
        o = np.lexsort((-ids, -lg[r].astype(np.float64)))[:k]
        out.append(ids[o])
    return np.array(out, dtype=np.int32)


def rope_interleaved(v, p, base):
    """RoPE pairing (2i, 2i+1) instead of (i, i + dim/2)."""
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    i = np.arange(d // 2, dtype=np.float64)
    th = p * np.power(float(base), -2.0 * i / d)
    a, b = v[0::2], v[1::2]
    out = np.empty_like(v)
    out[0::2] = a * np.cos(th) - b * np.sin(th)
    out[1::2] = a * np.sin(th) + b * np.cos(th)
    return out


def trunc_bf16(x):
    """bf16 by truncation toward zero instead of round-to-nearest-even."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x)
    _, e = np.frexp(x[fin])
    q = np.maximum(e - 8, -133)
    out[fin] = np.ldexp(np.trunc(np.ldexp(x[fin], -q)), q)
    return out


def round_half_away_bf16(x):
    """bf16 rounding to nearest with ties away from zero instead of to even."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x)
    _, e = np.frexp(x[fin])
    q = np.maximum(e - 8, -133)
    m = np.ldexp(x[fin], -q)
    out[fin] = np.ldexp(np.sign(m) * np.floor(np.abs(m) + 0.5), q)
    return out


def accept_count_all_equal(drafts, n_asked, draws):
    """Counts every equal position instead of the equal prefix."""
    d, w = np.asarray(drafts), np.asarray(draws)
    return np.array([(d[s, :n_asked[s]] == w[s, :n_asked[s]]).sum() for s in range(len(d))])


# ---- CPU controls: the oracle's pins catch each mutant -------------------------------------------

def test_control_e4m3_tie_rule_is_caught_by_the_torch_cast_pin():
    v = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 448)]
    lib = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(numerics.e4m3_encode(v), lib)
    assert not np.array_equal(encode_ties_away(v), lib)


def test_control_row_scale_rule_is_caught():
    w = inputs.normal_bf16((256, 512), 0.02, 800).float().numpy()
    t = torch.from_numpy(w)
    ts = t.abs().amax(dim=1) / 448.0
    ref = (t / ts[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(quant_fp8_row(w)[0], ref)
    assert not np.array_equal(quant_row_multiply(w)[0], ref)


def test_control_block_exponent_rule_is_caught_by_the_no_saturation_pin():
    w = inputs.normal_bf16((256, 256), 0.02, 801).float().numpy()
    for fn, ok in ((quant_fp8_block32, True), (block_exponent_ocp, False)):
        codes, sb = fn(w)
        scaled = np.abs(w.astype(np.float64)).reshape(8, 32, 8, 32) / np.exp2(
            sb.astype(np.float64) - 127)[:, None, :, None]
        assert (scaled.max() <= 448.0) == ok


def test_control_tie_rule_is_caught_by_brute_force():
    lg = np.array([[1.0, 3.0, 2.0, 3.0, 3.0, 0.5]], np.float32)
    assert list(topk(lg, 2)[1][0]) == [1, 3]
    assert list(topk_higher_id(lg, 2)[0]) != [1, 3]


def test_control_rope_pairing_is_caught_by_the_complex_rotation_pin():
    x = inputs.normal_bf16((128,), 1.0, 802).float().numpy().astype(np.float64)
    z = (x[:64] + 1j * x[64:]) * np.exp(1j * 17 * 10000.0 ** (-np.arange(64) * 2 / 128))
    good = oattn.rope(x, 17, 10000.0)
    bad = rope_interleaved(x, 17, 10000.0)
    assert np.allclose(good[:64], z.real) and not np.allclose(bad[:64], z.real)


def test_control_accept_prefix_rule_is_caught():
    drafts = np.array([[5, 6, 7, 8, 9]])
    draws = np.array([[5, 6, 1, 8, 9]])
    assert accept(drafts, [5], draws)[0][0] == 2
    assert accept_count_all_equal(drafts, [5], draws)[0] != 2


def test_control_bf16_rounding_check_catches_truncation_and_ties_away():
    """The bf16 check holds values to round-to-nearest-even: fp32 results (the exact value plus an
    fp32-sized error) rounded by the method pass; the same results truncated, or with ties rounded
    away from zero, fail."""
    rng = np.random.default_rng([0, 803, 0])
    exact = rng.normal(0.0, 1.0, 20000) * np.exp2(rng.integers(-20, 20, 20000))
    err = 1e-6 * np.abs(exact)
    gpu_like = numerics.round_bf16(numerics.fl32(exact).astype(np.float64))
    assert_bf16_rounding(gpu_like, exact, err)
    with pytest.raises(AssertionError):
        assert_bf16_rounding(trunc_bf16(exact), exact, err)
    # exact ties: bf16 midpoints, which the even rule and the away rule round differently
    mids = (np.arange(1, 4000, 2) + 256.0) * 2.0 ** -9
    assert_bf16_rounding(numerics.round_bf16(mids), mids, 0.0)
    with pytest.raises(AssertionError):
        assert_bf16_rounding(round_half_away_bf16(mids), mids, 0.0)


# ---- GPU controls: the same mutants disagree with the CUDA path ----------------------------------

@pytest.mark.gpu
def test_gpu_control_quant_rules():
    need_gpu()
    from speculative_decoding_draft_row_gb300 import tfd
    w = inputs.normal_bf16((256, 512), 0.02, 810)
    wn = w.float().numpy()
    codes, _ = tfd.tfd_quant_fp8(w.cuda(), tfd.W_FP8_ROW)
    cb, sb = tfd.tfd_quant_fp8(w.cuda(), tfd.W_FP8_BLOCK32)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), quant_fp8_row(wn)[0])
    assert not np.array_equal(codes.cpu().numpy(), quant_row_multiply(wn)[0])
    assert np.array_equal(sb.cpu().numpy(), quant_fp8_block32(wn)[1])
    assert not np.array_equal(sb.cpu().numpy(), block_exponent_ocp(wn)[1])


@pytest.mark.gpu
def test_gpu_control_tie_rule():
    need_gpu()
    from speculative_decoding_draft_row_gb300 import tfd
    lg = np.tile(np.array([0.5, 2.0, 1.0, 2.0, 2.0], np.float32), (3, 200))
    v, i = tfd.tfd_topk(torch.from_numpy(lg).cuda(), 3)
    torch.cuda.synchronize()
    assert np.array_equal(i.cpu().numpy(), topk(lg, 3)[1])
    assert not np.array_equal(i.cpu().numpy(), topk_higher_id(lg, 3))


@pytest.mark.gpu
def test_gpu_control_rope_pairing(monkeypatch):
    need_gpu()
    from speculative_decoding_draft_row_gb300 import tfd
    S, H, D, ring = 1, 4, 128, 16
    q, k, v = (inputs.normal_bf16((S, H, D), 1.0, 820 + i) for i in range(3))
    kr = inputs.normal_bf16((S * ring, H, D), 1.0, 823).reshape(S, ring, H, D)
    vr = inputs.normal_bf16((S * ring, H, D), 1.0, 824).reshape(S, ring, H, D)
    kd, vd = kr.clone().cuda(), vr.clone().cuda()
    out = tfd.tfd_window_attn(q.cuda(), k.cuda(), v.cuda(), torch.tensor([9], dtype=torch.int32,
                              device="cuda"), kd, vd, 9)
    torch.cuda.synchronize()
    f = lambda t: t.float().numpy()
    args = (f(q), f(k), f(v), [9], f(kr), f(vr), 9)
    check_window_attn(np32(out), np32(kd), np32(vd), *args)
    monkeypatch.setattr(oattn, "rope", rope_interleaved)
    with pytest.raises(AssertionError):
        check_window_attn(np32(out), np32(kd), np32(vd), *args)


@pytest.mark.gpu
def test_gpu_control_bf16_truncation_is_caught():
    """An oracle that truncated to bf16 (instead of rounding to nearest even) fails against the
    GPU's bf16 outputs: GEMV out BF16 and ADD_BF16, RMSNorm, and the attention's output and ring
    keys."""
    need_gpu()
    from speculative_decoding_draft_row_gb300 import tfd
    w = inputs.normal_bf16((4096, 4096), 0.02, 830)
    x = inputs.normal_bf16((4, 4096), 1.0, 831)
    res = inputs.normal_bf16((4, 4096), 1.0, 832)
    y, _, _ = tfd.tfd_head_gemv(w.cuda(), tfd.W_BF16, None, x.cuda(), tfd.OUT_BF16)
    ya = res.clone().cuda()
    tfd.tfd_head_gemv(w.cuda(), tfd.W_BF16, None, x.cuda(), tfd.OUT_ADD_BF16, y=ya)
    hid = inputs.normal_bf16((4, 4096), 3.0, 833)
    hn = tfd.tfd_rmsnorm(hid.cuda(), None, 1e-6)
    torch.cuda.synchronize()
    acc = og.gemv_acc(w.float().numpy(), x.float().numpy())
    S = og.gemv_abs_scale(w.float().numpy(), x.float().numpy())
    ex_add = res.float().numpy().astype(np.float64) + acc
    ex_norm = rmsnorm_rows(hid.float().numpy(), None, 1e-6, exact=True)
    checks = [(np32(y), acc, gemv_bf16_err(S)), (np32(ya), ex_add, gemv_bf16_err(S, ex_add)),
              (np32(hn), ex_norm, NORM_REL * np.abs(ex_norm))]
    for got, ex, err in checks:
        assert_bf16_rounding(got, ex, err)
        with pytest.raises(AssertionError):
            assert_bf16_rounding(got, ex, err, rnd=trunc_bf16)
    S_, H, D, ring = 4, 32, 128, 528
    q, k, v = (inputs.normal_bf16((S_, H, D), 1.0, 840 + i) for i in range(3))
    kr = inputs.normal_bf16((S_ * ring, H, D), 1.0, 843).reshape(S_, ring, H, D)
    vr = inputs.normal_bf16((S_ * ring, H, D), 1.0, 844).reshape(S_, ring, H, D)
    pos = [511, 512, 513, 515]
    kd, vd = kr.clone().cuda(), vr.clone().cuda()
    out = tfd.tfd_window_attn(q.cuda(), k.cuda(), v.cuda(), torch.tensor(pos, dtype=torch.int32,
                              device="cuda"), kd, vd, 511)
    torch.cuda.synchronize()
    f = lambda t: t.float().numpy()
    args = (np32(out), np32(kd), np32(vd), f(q), f(k), f(v), pos, f(kr), f(vr), 511)
    check_window_attn(*args)
    with pytest.raises(AssertionError):
        check_window_attn(*args, rnd=trunc_bf16)
