"""GPU parity of the chained draft pass: every step checked against the oracle applied to the
GPU's own inputs of that step (the residual chains through bf16 roundings, so each step is held to
the per-call tolerances), then the accept count, then the graph-captured replay against eager."""
import numpy as np
import pytest
import torch

from helpers import assert_bf16_close, need_gpu, np32
from oracle import gemv as og
from oracle.accept import accept as oracle_accept
from oracle.attn import window_attn as oracle_attn
from oracle.quant import quant_fp8_row
from speculative_decoding_draft_row_gb300 import tfd
from speculative_decoding_draft_row_gb300.draft_pass import DraftPass
from synth import inputs

pytestmark = pytest.mark.gpu


def build(steps=5, S=4, H=2, D=128, hidden=256, inner=96, vocab=3000, ring=40, window=31):
    wo = quant_fp8_row(inputs.normal_bf16((hidden, H * D), 0.02, 600).float().numpy())
    w2 = quant_fp8_row(inputs.normal_bf16((hidden, inner), 0.02, 601).float().numpy())
    head = inputs.normal_bf16((vocab, hidden), 0.02, 602)
    kr = inputs.normal_bf16((S * ring, H, D), 1.0, 603).reshape(S, ring, H, D)
    vr = inputs.normal_bf16((S * ring, H, D), 1.0, 604).reshape(S, ring, H, D)
    dp = DraftPass(torch.from_numpy(wo[0]).cuda(), torch.from_numpy(wo[1]).cuda(),
                   torch.from_numpy(w2[0]).cuda(), torch.from_numpy(w2[1]).cuda(), head.cuda(),
                   tfd.W_BF16, None, kr.clone().cuda(), vr.clone().cuda(), window, steps)
    qs = [inputs.normal_bf16((S, H, D), 1.0, 610 + 3 * t) for t in range(steps)]
    ks = [inputs.normal_bf16((S, H, D), 1.0, 611 + 3 * t) for t in range(steps)]
    vs = [inputs.normal_bf16((S, H, D), 1.0, 612 + 3 * t) for t in range(steps)]
    us = [inputs.normal_bf16((S, inner), 1.0, 630 + t) for t in range(steps)]
    resid = inputs.normal_bf16((S, hidden), 1.0, 640)
    pos0 = [33, 34, 35, 100]
    dp.load(qs, ks, vs, us, pos0, resid.cuda())
    return dp, dict(wo=wo, w2=w2, head=head.float().numpy(), kr=kr, vr=vr, qs=qs, ks=ks, vs=vs,
                    us=us, resid=resid, pos0=pos0, window=window)


def test_each_step_against_the_oracle_then_accept():
    need_gpu()
    dp, o = build()
    kr, vr = o["kr"].float().numpy(), o["vr"].float().numpy()
    for t in range(dp.steps):
        res_before = np32(dp.resid)
        dp.step_attn(t)
        torch.cuda.synchronize()
        pos = [p + t for p in o["pos0"]]
        att, kr, vr = oracle_attn(o["qs"][t].float().numpy(), o["ks"][t].float().numpy(),
                                  o["vs"][t].float().numpy(), pos, kr, vr, o["window"])
        assert_bf16_close(np32(dp.attn), att, f"step {t} attention")
        kr = np32(dp.k_ring)                          # continue from the GPU's own ring
        dp.step_wo()
        torch.cuda.synchronize()
        mid = og.gemv(o["wo"][0], np32(dp.attn), og.W_FP8_ROW, o["wo"][1], og.OUT_ADD_BF16,
                      res=res_before)
        assert_bf16_close(np32(dp.resid), mid, f"step {t} residual after wo")
        mid = np32(dp.resid)
        dp.step_w2(t)
        torch.cuda.synchronize()
        end = og.gemv(o["w2"][0], o["us"][t].float().numpy(), og.W_FP8_ROW, o["w2"][1],
                      og.OUT_ADD_BF16, res=mid)
        assert_bf16_close(np32(dp.resid), end, f"step {t} residual after w2")
        dp.step_head(t)
        torch.cuda.synchronize()
        acc = og.gemv_acc(o["head"], np32(dp.resid))
        S_ = og.gemv_abs_scale(o["head"], np32(dp.resid))
        for s in range(dp.S):
            d = dp.drafts[s, t].item()
            assert acc[s, d] >= acc[s].max() - 2e-5 * S_[s].max(), f"step {t} stream {s} draft"
    drafts = dp.drafts.cpu().numpy()
    draws, _ = inputs.draws_with_prefix(drafts)
    n_asked = np.array([5, 4, 5, 2], np.int32)
    dp.load(o["qs"], o["ks"], o["vs"], o["us"], o["pos0"], dp.resid, n_asked, draws)
    dp.enqueue_accept()
    torch.cuda.synchronize()
    ok, ah, kh, bad = oracle_accept(drafts, n_asked, draws)
    assert np.array_equal(dp.n_kept.cpu().numpy(), ok) and not bad
    assert np.array_equal(dp.asked_hist.cpu().numpy(), ah)
    assert np.array_equal(dp.kept_hist.cpu().numpy(), kh)
    assert dp.status.item() == 0


def test_graph_replay_equals_eager():
    need_gpu()
    dp1, _ = build()
    dp2, _ = build()
    # three passes each: dp1 eagerly; dp2 one eager pass inside capture(), then two replays
    dp1.enqueue()
    dp2.capture()
    dp1.enqueue()
    dp2.run()
    dp1.enqueue()
    dp2.run()
    torch.cuda.synchronize()
    assert torch.equal(dp1.drafts, dp2.drafts)
    assert torch.equal(dp1.resid, dp2.resid)
    assert torch.equal(dp1.k_ring, dp2.k_ring) and torch.equal(dp1.v_ring, dp2.v_ring)
