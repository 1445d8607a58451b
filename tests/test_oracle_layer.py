"""Pins of the oracle's RMSNorm of hidden rows, SwiGLU and multi-row ring absorb: library routines
(torch's rms_norm and silu in float64), closed forms, the pages' rounding order checked against a
planted mutant, and ring invariants."""
import numpy as np
import pytest
import torch

from oracle.layer import absorb, rmsnorm_rows, silu, swiglu
from oracle.numerics import round_bf16
from synth import inputs


def bf(shape, std, tid):
    return inputs.normal_bf16(shape, std, tid).float().numpy().astype(np.float64)


def test_rmsnorm_matches_torch_rms_norm():
    x = bf((5, 4096), 1.0, 900)
    g = bf((4096,), 0.5, 901) + 1.0
    for eps in (1e-6, 1e-2):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (4096,), torch.from_numpy(g), eps)
        assert np.array_equal(rmsnorm_rows(x, g, eps), round_bf16(ref.numpy()))


def test_rmsnorm_closed_forms():
    # a constant row normalises to +-gamma (eps = 0); scaling a row changes nothing
    row = np.full((1, 256), -3.0)
    g = bf((256,), 1.0, 902)
    assert np.array_equal(rmsnorm_rows(row, g, 0.0)[0], round_bf16(-g))
    x = bf((3, 512), 1.0, 903)
    assert np.array_equal(rmsnorm_rows(x, None, 0.0), rmsnorm_rows(8.0 * x, None, 0.0))
    y = rmsnorm_rows(x, None, 1e-6)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-2)


def test_silu_matches_torch_and_limits():
    g = np.concatenate([bf((20000,), 4.0, 904), [0.0, -0.0, 80.0, -80.0, 1e-30, -1e-30]])
    ref = torch.nn.functional.silu(torch.from_numpy(g)).numpy()
    assert np.allclose(silu(g), ref, rtol=1e-14, atol=1e-300)
    assert silu(np.array([0.0]))[0] == 0.0
    assert silu(np.array([80.0]))[0] == 80.0
    assert -1e-30 < silu(np.array([-80.0]))[0] < 0.0


def test_swiglu_rounds_silu_before_the_multiply():
    """The pages round SiLU(g) to bf16 before multiplying by u: a mutant that multiplies the
    unrounded SiLU disagrees on a real fraction of inputs, and the oracle agrees with torch's bf16
    silu (fp32 math, one rounding) wherever fp32 cannot flip the rounding."""
    g = bf((40000,), 2.0, 905)
    u = bf((40000,), 2.0, 906)
    out = swiglu(g, u)
    mutant = round_bf16(silu(g) * u)
    assert (out != mutant).mean() > 0.01
    s_torch = torch.nn.functional.silu(torch.from_numpy(g).to(torch.bfloat16)).double().numpy()
    s_oracle = round_bf16(silu(g))
    differ = s_torch != s_oracle
    # any disagreement must sit within fp32 error of a bf16 rounding midpoint
    ex = silu(g[differ])
    mid = (s_torch[differ] + s_oracle[differ]) / 2
    assert np.all(np.abs(ex - mid) <= 4e-7 * np.abs(ex))
    assert np.array_equal(out[~differ], round_bf16(s_torch[~differ] * u[~differ]))


def test_absorb_ring_slots_and_refusal():
    S, n, H, D, ring = 2, 7, 3, 128, 8
    k = bf((S * n, H, D), 1.0, 907).reshape(S, n, H, D)
    v = bf((S * n, H, D), 1.0, 908).reshape(S, n, H, D)
    kr = bf((S * ring, H, D), 1.0, 909).reshape(S, ring, H, D)
    vr = bf((S * ring, H, D), 1.0, 910).reshape(S, ring, H, D)
    p0 = [0, 13]
    k2, v2 = absorb(k, v, p0, kr, vr)
    for s in range(S):
        written = {(p0[s] + i) % ring for i in range(n)}
        for slot in range(ring):
            if slot in written:
                i = [i for i in range(n) if (p0[s] + i) % ring == slot][0]
                assert np.array_equal(v2[s, slot], v[s, i])
            else:
                assert np.array_equal(k2[s, slot], kr[s, slot]) and np.array_equal(v2[s, slot], vr[s, slot])
    # position 0: RoPE is the identity, so the key is bf16(rmsnorm(k))
    ref = torch.nn.functional.rms_norm(torch.from_numpy(k[0, 0]), (D,), None, 1e-6).numpy()
    assert np.array_equal(k2[0, 0], round_bf16(ref))
    # the rotation keeps each (i, i + 64) pair's length
    kn = torch.nn.functional.rms_norm(torch.from_numpy(k[1, 3]), (D,), None, 1e-6).numpy()
    got = k2[1, (13 + 3) % ring]
    assert np.allclose(np.hypot(got[:, :64], got[:, 64:]), np.hypot(kn[:, :64], kn[:, 64:]), rtol=2e-2)
    with pytest.raises(ValueError):
        absorb(bf((1, ring + 1, H, D), 1.0, 911).reshape(1, ring + 1, H, D), np.zeros((1, ring + 1, H, D)),
               [0], kr[:1], vr[:1])


def test_absorb_of_a_span_equals_absorbs_of_its_pieces():
    S, n, H, D, ring = 1, 6, 2, 128, 16
    k = bf((S * n, H, D), 1.0, 912).reshape(S, n, H, D)
    v = bf((S * n, H, D), 1.0, 913).reshape(S, n, H, D)
    kr = np.zeros((S, ring, H, D))
    vr = np.zeros((S, ring, H, D))
    whole = absorb(k, v, [30], kr, vr)
    a = absorb(k[:, :2], v[:, :2], [30], kr, vr)
    b = absorb(k[:, 2:], v[:, 2:], [32], *a)
    assert np.array_equal(whole[0], b[0]) and np.array_equal(whole[1], b[1])


def test_unrounded_rmsnorm_and_absorb_terms():
    """rmsnorm_rows(exact=True) rounds to rmsnorm_rows; the absorb's exact keys round to the keys
    it writes and keep each rotation pair's magnitude; unwritten slots are NaN in the terms."""
    from oracle.attn import rmsnorm, rope
    x = bf((3, 256), 3.0, 180)
    ex = rmsnorm_rows(x, None, 1e-6, exact=True)
    assert np.array_equal(round_bf16(ex), rmsnorm_rows(x, None, 1e-6))
    S, n, H, D, ring = 1, 3, 2, 128, 8
    k, v = bf((S, n, H, D), 1.0, 181), bf((S, n, H, D), 1.0, 182)
    kr, vr = bf((S, ring, H, D), 1.0, 183), bf((S, ring, H, D), 1.0, 184)
    terms = {}
    okr, _ = absorb(k, v, [6], kr, vr, terms=terms)
    written = ~np.isnan(terms["k_exact"][..., 0])
    assert written.sum() == n * H and written[0, [6, 7, 0]].all()
    w = ~np.isnan(terms["k_exact"])
    assert np.array_equal(round_bf16(terms["k_exact"][w]), okr[w])
    ke, kp = terms["k_exact"][0, 6, 0], terms["k_pair"][0, 6, 0]
    assert np.allclose(np.hypot(ke[:64], ke[64:]), kp[:64], rtol=1e-12)
    assert np.allclose(ke, rope(rmsnorm(k[0, 0, 0], np.ones(D), 1e-6), 6, 10000.0), rtol=0, atol=0)
