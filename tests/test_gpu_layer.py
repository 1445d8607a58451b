"""GPU parity of the rest of the head layer: tfd_rmsnorm, tfd_swiglu and tfd_absorb against the
oracle (bf16 outputs held to their rounding), with the refusals and the device-data error of the
absorb."""
import numpy as np
import pytest
import torch

from helpers import (KEY_REL, NORM_REL, assert_bf16_rounding, check_window_attn, need_gpu, np32,
                     swiglu_bounds)
from oracle.attn import window_attn as oracle_attn
from oracle.layer import absorb as oracle_absorb
from oracle.layer import rmsnorm_rows, silu, swiglu
from oracle.numerics import round_bf16
from speculative_decoding_draft_row_gb300 import tfd
from synth import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,hidden,gamma,eps", [(4, 4096, True, 1e-6), (1, 8, False, 0.0),
                                                   (16, 11008, True, 1e-5), (3, 4104, False, 1e-6)])
def test_rmsnorm(rows, hidden, gamma, eps):
    need_gpu()
    x = inputs.normal_bf16((rows, hidden), 3.0, 920)
    g = inputs.normal_bf16((hidden,), 0.5, 921) if gamma else None
    out = tfd.tfd_rmsnorm(x.cuda(), None if g is None else g.cuda(), eps)
    torch.cuda.synchronize()
    ex = rmsnorm_rows(x.float().numpy(), None if g is None else g.float().numpy(), eps, exact=True)
    assert_bf16_rounding(np32(out), ex, NORM_REL * np.abs(ex), "rmsnorm")


def test_rmsnorm_in_place_and_strided():
    need_gpu()
    full = inputs.normal_bf16((5, 4096 + 64), 1.0, 922)
    xd = full.cuda()
    x = xd[:, :4096]
    ex = rmsnorm_rows(full[:, :4096].float().numpy(), None, 1e-6, exact=True)
    tfd.tfd_rmsnorm(x, None, 1e-6, out=x)
    torch.cuda.synchronize()
    assert_bf16_rounding(np32(x), ex, NORM_REL * np.abs(ex), "in place")
    assert torch.equal(xd[:, 4096:].cpu(), full[:, 4096:])  # the padding is untouched


def check_swiglu(g, u, out):
    """Exact, except where the fp32 SiLU (within 2^-20 of the exact one) can round to either bf16
    neighbour: every output bf16(s u) those roundings give is accepted."""
    gn, un, on = g.float().numpy(), u.float().numpy(), np32(out)
    lo, hi = swiglu_bounds(gn, un)
    ok = (on >= lo) & (on <= hi)
    bad = ~ok
    assert not bad.any(), f"{bad.sum()} swiglu outputs differ; first at {np.argwhere(bad)[0]}"
    # away from those midpoints the output is the oracle's, bit for bit
    assert ((on == swiglu(gn, un)) | (lo != hi)).all()


@pytest.mark.parametrize("rows,cols", [(4, 11008), (16, 8), (1, 4096)])
def test_swiglu(rows, cols):
    need_gpu()
    g = inputs.normal_bf16((rows, cols), 3.0, 923)
    u = inputs.normal_bf16((rows, cols), 2.0, 924)
    out = tfd.tfd_swiglu(g.cuda(), u.cuda())
    torch.cuda.synchronize()
    check_swiglu(g, u, out)


def test_swiglu_extremes_and_in_place():
    need_gpu()
    vals = torch.tensor([0.0, -0.0, 1.0, -1.0, 80.0, -80.0, 100.0, -100.0], dtype=torch.float32)
    g = vals.repeat(2, 64).to(torch.bfloat16)
    u = inputs.normal_bf16((2, 512), 1.0, 925)
    gd = g.cuda()
    tfd.tfd_swiglu(gd, u.cuda(), out=gd)
    torch.cuda.synchronize()
    check_swiglu(g, u, gd)


def absorb_case(S, n, H, ring, p0, tid, gamma=False):
    D = 128
    k = inputs.normal_bf16((S * n, H, D), 1.0, tid).reshape(S, n, H, D)
    v = inputs.normal_bf16((S * n, H, D), 1.0, tid + 1).reshape(S, n, H, D)
    kr = inputs.normal_bf16((S * ring, H, D), 1.0, tid + 2).reshape(S, ring, H, D)
    vr = inputs.normal_bf16((S * ring, H, D), 1.0, tid + 3).reshape(S, ring, H, D)
    kg = inputs.normal_bf16((D,), 0.5, tid + 4) if gamma else None
    return k, v, kr, vr, kg


@pytest.mark.parametrize("S,n,H,ring,p0,gamma", [(4, 128, 32, 528, [0, 100, 512, 1000], False),
                                                 (1, 144, 6, 144, [7], True),
                                                 (2, 1, 32, 16, [3, 70000], True)])
def test_absorb(S, n, H, ring, p0, gamma):
    need_gpu()
    k, v, kr, vr, kg = absorb_case(S, n, H, ring, p0, 930, gamma)
    krd, vrd = kr.clone().cuda(), vr.clone().cuda()
    tfd.tfd_absorb(k.cuda(), v.cuda(), torch.tensor(p0, dtype=torch.int32).cuda(), krd, vrd,
                   k_gamma=None if kg is None else kg.cuda())
    torch.cuda.synchronize()
    f = lambda t: None if t is None else t.float().numpy()
    terms = {}
    okr, ovr = oracle_absorb(f(k), f(v), p0, f(kr), f(vr), k_gamma=f(kg), terms=terms)
    written = ~np.isnan(terms["k_exact"])
    assert_bf16_rounding(np32(krd)[written], terms["k_exact"][written],
                         KEY_REL * terms["k_pair"][written], "absorbed keys")
    assert np.array_equal(np32(krd)[~written], okr[~written])
    assert np.array_equal(np32(vrd), ovr)


def test_absorb_then_attention_matches_the_oracle():
    """A prompt chunk absorbed into the ring, then one decode position attending over it."""
    need_gpu()
    S, n, H, ring, D = 2, 511, 8, 528, 128
    k, v, kr, vr, _ = absorb_case(S, n, H, ring, [0, 0], 940)
    krd, vrd = kr.clone().cuda(), vr.clone().cuda()
    tfd.tfd_absorb(k.cuda(), v.cuda(), torch.zeros(S, dtype=torch.int32).cuda(), krd, vrd)
    kab, vab = krd.clone(), vrd.clone()
    q, kn, vn = (inputs.normal_bf16((S, H, D), 1.0, 950 + i) for i in range(3))
    pos = [511, 511]
    out = tfd.tfd_window_attn(q.cuda(), kn.cuda(), vn.cuda(), torch.tensor(pos, dtype=torch.int32).cuda(),
                              krd, vrd, 511)
    torch.cuda.synchronize()
    f = lambda t: t.float().numpy()
    terms = {}
    oracle_absorb(f(k), f(v), [0, 0], f(kr), f(vr), terms=terms)
    # the absorbed keys (slots 0..510), as they stood before the attention wrote slot 511
    written = ~np.isnan(terms["k_exact"])
    assert_bf16_rounding(np32(kab)[written], terms["k_exact"][written],
                         KEY_REL * terms["k_pair"][written], "absorbed keys")
    # then the attention against the oracle attending over the ring the absorb wrote (each key
    # just accepted as a correct rounding)
    check_window_attn(np32(out), np32(krd), np32(vrd), f(q), f(kn), f(vn), pos, np32(kab),
                      np32(vab), 511, what="attention after absorb")


def test_absorbed_row_equals_the_attention_ring_write():
    need_gpu()
    S, H, ring, D = 3, 4, 32, 128
    k, v, kr, vr, kg = absorb_case(S, 1, H, ring, [5, 40, 77], 960, gamma=True)
    p = torch.tensor([5, 40, 77], dtype=torch.int32).cuda()
    ka, va = kr.clone().cuda(), vr.clone().cuda()
    tfd.tfd_absorb(k.cuda(), v.cuda(), p, ka, va, k_gamma=kg.cuda())
    kb, vb = kr.clone().cuda(), vr.clone().cuda()
    q = inputs.normal_bf16((S, H, D), 1.0, 965).cuda()
    tfd.tfd_window_attn(q, k[:, 0].contiguous().cuda(), v[:, 0].contiguous().cuda(), p, kb, vb, 0,
                        k_gamma=kg.cuda())
    torch.cuda.synchronize()
    assert torch.equal(ka, kb) and torch.equal(va, vb)


def test_absorb_refuses_a_span_longer_than_the_ring_and_flags_bad_positions():
    need_gpu()
    k, v, kr, vr, _ = absorb_case(1, 17, 2, 16, [0], 970)
    krd, vrd = kr.clone().cuda(), vr.clone().cuda()
    with pytest.raises(tfd.TfdError) as e:
        tfd.tfd_absorb(k.cuda(), v.cuda(), torch.zeros(1, dtype=torch.int32).cuda(), krd, vrd)
    assert e.value.status == tfd.ERR_INVALID
    k, v, kr, vr, _ = absorb_case(2, 4, 2, 16, [0, 0], 975)
    krd, vrd = kr.clone().cuda(), vr.clone().cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tfd.tfd_absorb(k.cuda(), v.cuda(), torch.tensor([-1, 2147483646], dtype=torch.int32).cuda(),
                   krd, vrd, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == tfd.ERR_DEVICE_DATA
    assert torch.equal(krd.cpu(), kr) and torch.equal(vrd.cpu(), vr)  # both streams left unwritten
