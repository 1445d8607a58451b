"""Pins of the oracle's chained draft pass on cases with closed-form answers."""
import numpy as np

from oracle.draft_pass import draft_pass, pass_accept
from oracle.gemv import W_BF16
from oracle.quant import quant_fp8_row
from synth import inputs


def small_pass(steps=3, S=2, H=2, D=128, hidden=256, inner=96, vocab=300, ring=12, zero_lin=False):
    qs = [inputs.normal_bf16((S, H, D), 1.0, 170 + 3 * t).float().numpy() for t in range(steps)]
    ks = [inputs.normal_bf16((S, H, D), 1.0, 171 + 3 * t).float().numpy() for t in range(steps)]
    vs = [inputs.normal_bf16((S, H, D), 1.0, 172 + 3 * t).float().numpy() for t in range(steps)]
    kr = inputs.normal_bf16((S, ring, H, D), 1.0, 190).float().numpy()
    vr = inputs.normal_bf16((S, ring, H, D), 1.0, 191).float().numpy()
    wo = inputs.normal_bf16((hidden, H * D), 0.02, 192).float().numpy()
    w2 = inputs.normal_bf16((hidden, inner), 0.02, 193).float().numpy()
    if zero_lin:
        wo[:] = 0
        w2[:] = 0
    wo_c, wo_s = quant_fp8_row(wo)
    w2_c, w2_s = quant_fp8_row(w2)
    us = [inputs.normal_bf16((S, inner), 1.0, 194 + t).float().numpy() for t in range(steps)]
    resid = inputs.normal_bf16((S, hidden), 1.0, 198).float().numpy()
    head = inputs.normal_bf16((vocab, hidden), 0.02, 199).float().numpy()
    return dict(steps=steps, qs=qs, ks=ks, vs=vs, pos0=[7, 3], k_ring=kr, v_ring=vr, window=4,
                wo_codes=wo_c, wo_s=wo_s, w2_codes=w2_c, w2_s=w2_s, us=us, resid0=resid,
                head_w=head, head_fmt=W_BF16, head_scales=None)


def test_zero_linears_draft_the_head_argmax_of_the_residual():
    args = small_pass(zero_lin=True)
    res = draft_pass(**args)
    expect = np.argmax(args["resid0"].astype(np.float64) @ args["head_w"].astype(np.float64).T,
                       axis=1)
    for t in range(args["steps"]):
        assert np.array_equal(res["drafts"][:, t], expect)
    assert np.array_equal(res["resid"], args["resid0"])


def test_residual_chains_and_ring_advances():
    args = small_pass()
    res = draft_pass(**args)
    assert not np.array_equal(res["resid"], args["resid0"])
    ring = args["k_ring"].shape[1]
    for s, p0 in enumerate(args["pos0"]):
        touched = [i for i in range(ring) if not np.array_equal(res["k_ring"][s, i],
                                                                args["k_ring"][s, i])]
        assert touched == sorted((p0 + t) % ring for t in range(args["steps"]))
    n_kept, _, _, bad = pass_accept(res["drafts"], [3, 3], res["drafts"])
    assert list(n_kept) == [3, 3] and not bad
