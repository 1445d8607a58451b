"""Pins of the oracle's window attention: closed forms (window 0, equal keys, two keys), RoPE as a
complex rotation, relative-position invariance, norms, and the ring write."""
import numpy as np

from oracle.attn import rmsnorm, rope, window_attn
from oracle.numerics import round_bf16
from synth import inputs


def rand(shape, tid, std=1.0):
    return inputs.normal_bf16(shape, std, tid).float().numpy().astype(np.float64)


def test_window_zero_returns_current_value():
    S, H, D, ring = 2, 3, 128, 8
    q, k, v = rand((S, H, D), 140), rand((S, H, D), 141), rand((S, H, D), 142)
    kr, vr = rand((S, ring, H, D), 143), rand((S, ring, H, D), 144)
    out, kr2, vr2 = window_attn(q, k, v, [5, 0], kr, vr, window=0)
    assert np.array_equal(out.reshape(S, H, D), round_bf16(v))
    assert np.array_equal(vr2[0, 5], v[0]) and np.array_equal(vr2[1, 0], v[1])


def test_equal_keys_average_the_values():
    S, H, D, ring = 1, 2, 128, 16
    q, k, v = rand((S, H, D), 145), rand((S, H, D), 146), rand((S, H, D), 147)
    p = 9
    kcur = np.stack([round_bf16(rope(rmsnorm(k[0, h], np.ones(D), 1e-6), p, 10000.0))
                     for h in range(H)])
    kr = np.broadcast_to(kcur, (S, ring, H, D)).copy()
    vr = rand((S, ring, H, D), 148)
    out, _, vr2 = window_attn(q, k, v, [p], kr, vr, window=5)
    for h in range(H):
        mean = vr2[0, [j % ring for j in range(p - 5, p + 1)], h].mean(axis=0)
        # the output is the bf16 rounding of the mean: within half a bf16 step of it
        assert np.all(np.abs(out[0, h * D:(h + 1) * D] - mean) <= 2.0 ** -8 * np.abs(mean) * (1 + 1e-9) + 1e-12)


def test_two_keys_logistic_weight():
    # p = 1, window 1: keys at positions 0 (ring) and 1 (current). Put the ring key equal to the
    # current key plus a multiple of the current key so the score gap is known in closed form.
    D = 128
    q = rand((1, 1, D), 150)
    k = rand((1, 1, D), 151)
    v = rand((1, 1, D), 152)
    kcur = round_bf16(rope(rmsnorm(k[0, 0], np.ones(D), 1e-6), 1, 10000.0))
    qn = rope(rmsnorm(q[0, 0], np.ones(D), 1e-6), 1, 10000.0)
    kr = np.zeros((1, 2, 1, D))
    kr[0, 0, 0] = 2 * kcur                           # score0 = 2 * score1
    vr = rand((1, 2, 1, D), 153)
    out, _, _ = window_attn(q, k, v, [1], kr, vr, window=1)
    s1 = kcur @ qn / np.sqrt(D)
    w0 = 1.0 / (1.0 + np.exp(-s1))                   # softmax of (2 s1, s1)
    ref = w0 * vr[0, 0, 0] + (1 - w0) * v[0, 0]
    assert np.allclose(out[0], round_bf16(ref), rtol=0, atol=2 ** -7 * np.abs(ref).max())


def test_rope_is_complex_rotation():
    D = 128
    x = rand((D,), 154)
    for p in (0, 1, 17, 511, 100000):
        z = (x[:64] + 1j * x[64:]) * np.exp(1j * p * 10000.0 ** (-np.arange(64) * 2 / D))
        y = rope(x, p, 10000.0)
        assert np.allclose(y[:64], z.real, atol=1e-12) and np.allclose(y[64:], z.imag, atol=1e-12)
    assert np.array_equal(rope(x, 0, 10000.0), x)
    assert np.isclose(np.linalg.norm(rope(x, 123, 10000.0)), np.linalg.norm(x))


def test_scores_depend_on_relative_position_only():
    D = 128
    a, b = rand((D,), 155), rand((D,), 156)
    for p, j in ((40, 3), (511, 0), (7, 7)):
        s0 = rope(a, p, 10000.0) @ rope(b, j, 10000.0)
        s1 = rope(a, p + 1000, 10000.0) @ rope(b, j + 1000, 10000.0)
        assert np.isclose(s0, s1, rtol=1e-9, atol=1e-9)


def test_rmsnorm_unit_rms_and_gamma():
    x = rand((128,), 157)
    y = rmsnorm(x, np.ones(128), 0.0)
    assert np.isclose(np.sqrt(np.mean(y * y)), 1.0)
    g = rand((128,), 158)
    assert np.allclose(rmsnorm(x, g, 1e-6), rmsnorm(x, np.ones(128), 1e-6) * g)


def test_ring_write_and_window_positions():
    S, H, D, ring = 1, 1, 128, 6
    q, k, v = rand((S, H, D), 160), rand((S, H, D), 161), rand((S, H, D), 162)
    kr, vr = rand((S, ring, H, D), 163), rand((S, ring, H, D), 164)
    p = 13                                              # slot 1
    _, kr2, vr2 = window_attn(q, k, v, [p], kr, vr, window=4)
    changed = [i for i in range(ring) if not np.array_equal(kr2[0, i], kr[0, i])]
    assert changed == [1]
    # slot 0 (position 12, inside the window) and slot 2 (position 8, inside) keep their rows;
    # slot 3 (position 9) too; a window of 4 reads positions 9..13 only: changing slot 2 (pos 8 or
    # 14) must not change the output.
    out_a, _, _ = window_attn(q, k, v, [p], kr, vr, window=4)
    kr_b = kr.copy()
    kr_b[0, 2] += 5.0
    out_b, _, _ = window_attn(q, k, v, [p], kr_b, vr, window=4)
    assert np.array_equal(out_a, out_b)


def test_unrounded_terms_round_to_the_outputs_and_hold_their_invariants():
    """The oracle's values before rounding (used to hold the GPU's bf16 outputs to their
    rounding): they round to the oracle's own outputs; RoPE keeps every pair's magnitude, so the
    exact key's pairs have the magnitudes reported for the normalised key; the softmax-weighted
    magnitudes bound the output; with a given current key the output is attention over it."""
    from oracle.numerics import round_bf16
    S, H, D, ring = 2, 3, 128, 8
    q, k, v = rand((S, H, D), 170), rand((S, H, D), 171), rand((S, H, D), 172)
    kr, vr = rand((S, ring, H, D), 173), rand((S, ring, H, D), 174)
    pos = [9, 40000]
    terms = {}
    out, kr2, _ = window_attn(q, k, v, pos, kr, vr, 5, terms=terms)
    assert np.array_equal(round_bf16(terms["out_exact"]), out)
    for s in range(S):
        assert np.array_equal(round_bf16(terms["k_exact"][s]), kr2[s, pos[s] % ring])
    ke = terms["k_exact"]
    assert np.allclose(np.hypot(ke[..., :64], ke[..., 64:]), terms["k_pair"][..., :64], rtol=1e-12)
    assert (terms["abs_out"] >= np.abs(terms["out_exact"]) * (1 - 1e-12)).all()
    assert (terms["abs_dev"] <= 2 * terms["abs_out"] + 1e-12).all()
    # the current key given: its values are the ones attended
    kc = round_bf16(ke) + 0.25
    out_c, kr3, _ = window_attn(q, k, v, pos, kr, vr, 5, k_cur=kc)
    for s in range(S):
        assert np.array_equal(kr3[s, pos[s] % ring], kc[s])
    assert not np.array_equal(out_c, out)
