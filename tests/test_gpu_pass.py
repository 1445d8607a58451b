"""GPU parity of the chained draft pass: every step checked against the oracle applied to the
GPU's own inputs of that step (the residual chains through bf16 roundings, so each step is held to
the per-call tolerances: attention and residual adds to their bf16 rounding, the draft to the
argmax rule), then the accept count, then the graph-captured replay against eager. Run at a small
shape and at the measured shape (4 streams x 32 heads x 128, hidden 4096, w2 inner 11008, ring
528, window 511, the 163840-row head in bf16 and in interleaved block-32 FP8)."""
import numpy as np
import pytest
import torch

from helpers import (assert_bf16_rounding, check_window_attn, full_head_oracle, gemv_bf16_err,
                     need_gpu, np32, oracle_fp8_codes)
from oracle import gemv as og
from oracle.accept import accept as oracle_accept
from oracle.quant import block32_interleave, quant_fp8_row
from speculative_decoding_draft_row_gb300 import tfd
from speculative_decoding_draft_row_gb300.draft_pass import DraftPass
from synth import inputs

pytestmark = pytest.mark.gpu


def build(steps=5, S=4, H=2, D=128, hidden=256, inner=96, vocab=3000, ring=40, window=31,
          head_fmt=tfd.W_BF16, pos0=(33, 34, 35, 100), full_head=None):
    """A pass with its inputs. The FP8 linears (and an FP8 head) are quantised by the oracle and
    passed to both sides; full_head = (bf16 weight, oracle codes, scales) of the measured head."""
    wo = quant_fp8_row(inputs.linear(hidden, H * D, 600).float().numpy())
    w2 = quant_fp8_row(inputs.linear(hidden, inner, 601).float().numpy())
    if full_head is None:
        head = inputs.normal_bf16((vocab, hidden), 0.02, 602)
        hcodes, hscales = None, None
    else:
        head, hcodes, hscales = full_head
    kr = inputs.normal_bf16((S * ring, H, D), 1.0, 603).reshape(S, ring, H, D)
    vr = inputs.normal_bf16((S * ring, H, D), 1.0, 604).reshape(S, ring, H, D)
    if head_fmt == tfd.W_BF16:
        hd, hs = head.cuda(), None
    else:
        hd = torch.from_numpy(block32_interleave(hcodes)).cuda()
        hs = torch.from_numpy(hscales).cuda()
    dp = DraftPass(torch.from_numpy(wo[0]).cuda(), torch.from_numpy(wo[1]).cuda(),
                   torch.from_numpy(w2[0]).cuda(), torch.from_numpy(w2[1]).cuda(), hd,
                   head_fmt, hs, kr.clone().cuda(), vr.clone().cuda(), window, steps)
    qs = [inputs.normal_bf16((S, H, D), 1.0, 610 + 3 * t) for t in range(steps)]
    ks = [inputs.normal_bf16((S, H, D), 1.0, 611 + 3 * t) for t in range(steps)]
    vs = [inputs.normal_bf16((S, H, D), 1.0, 612 + 3 * t) for t in range(steps)]
    us = [inputs.normal_bf16((S, inner), 1.0, 630 + t) for t in range(steps)]
    resid = inputs.normal_bf16((S, hidden), 1.0, 640)
    dp.load(qs, ks, vs, us, list(pos0), resid.cuda())
    if head_fmt == tfd.W_BF16:
        ho = (head.float().numpy(), og.W_BF16, None)
    else:
        ho = (hcodes, og.W_FP8_BLOCK32, hscales)
    return dp, dict(wo=wo, w2=w2, head=ho, qs=qs, ks=ks, vs=vs, us=us, resid=resid,
                    pos0=list(pos0), window=window)


def run_and_check(dp, o, head_oracle):
    for t in range(dp.steps):
        res_before = np32(dp.resid)
        kr_before, vr_before = np32(dp.k_ring), np32(dp.v_ring)
        dp.step_attn(t)
        torch.cuda.synchronize()
        pos = [p + t for p in o["pos0"]]
        check_window_attn(np32(dp.attn), np32(dp.k_ring), np32(dp.v_ring),
                          o["qs"][t].float().numpy(), o["ks"][t].float().numpy(),
                          o["vs"][t].float().numpy(), pos, kr_before, vr_before, o["window"],
                          what=f"step {t} attention")
        dp.step_wo()
        torch.cuda.synchronize()
        a = np32(dp.attn)
        ex = res_before + og.gemv_acc(o["wo"][0], a, og.W_FP8_ROW, o["wo"][1])
        S = og.gemv_abs_scale(o["wo"][0], a, og.W_FP8_ROW, o["wo"][1])
        assert_bf16_rounding(np32(dp.resid), ex, gemv_bf16_err(S, ex), f"step {t} resid after wo")
        mid = np32(dp.resid)
        dp.step_w2(t)
        torch.cuda.synchronize()
        u = o["us"][t].float().numpy()
        ex = mid + og.gemv_acc(o["w2"][0], u, og.W_FP8_ROW, o["w2"][1])
        S = og.gemv_abs_scale(o["w2"][0], u, og.W_FP8_ROW, o["w2"][1])
        assert_bf16_rounding(np32(dp.resid), ex, gemv_bf16_err(S, ex), f"step {t} resid after w2")
        dp.step_head(t)
        torch.cuda.synchronize()
        acc, S_ = head_oracle(np32(dp.resid))
        for s in range(dp.S):
            d = dp.drafts[s, t].item()
            assert acc[s, d] >= acc[s].max() - 2e-5 * S_[s].max(), f"step {t} stream {s} draft"
            assert abs(dp.draft_vals[s, t].item() - acc[s, d]) <= 1e-5 * S_[s, d] + 1e-30
    drafts = dp.drafts.cpu().numpy()
    draws, _ = inputs.draws_with_prefix(drafts)
    n_asked = np.array([5, 4, 5, 2], np.int32)[:dp.S]
    dp.load(o["qs"], o["ks"], o["vs"], o["us"], o["pos0"], dp.resid, n_asked, draws)
    dp.enqueue_accept()
    torch.cuda.synchronize()
    ok, ah, kh, bad = oracle_accept(drafts, n_asked, draws)
    assert np.array_equal(dp.n_kept.cpu().numpy(), ok) and not bad
    assert np.array_equal(dp.asked_hist.cpu().numpy(), ah)
    assert np.array_equal(dp.kept_hist.cpu().numpy(), kh)
    assert dp.status.item() == 0


def test_each_step_against_the_oracle_then_accept():
    need_gpu()
    dp, o = build()
    w, fmt, sc = o["head"]
    run_and_check(dp, o, lambda x: (og.gemv_acc(w, x, fmt, sc), og.gemv_abs_scale(w, x, fmt, sc)))


@pytest.fixture(scope="module")
def measured_head():
    need_gpu()
    w, _ = inputs.head(tie_frac=0.01)
    codes, scales = oracle_fp8_codes(w.float().numpy(), og.W_FP8_BLOCK32)
    return w, codes, scales


@pytest.mark.parametrize("head_fmt", [tfd.W_BF16, tfd.W_FP8_BLOCK32_IL])
def test_measured_shape_each_step_against_the_oracle(measured_head, head_fmt):
    """The pass at the shape bench.py measures, every step against the oracle."""
    need_gpu()
    dp, o = build(S=4, H=32, D=128, hidden=4096, inner=11008, ring=528, window=511,
                  head_fmt=head_fmt, pos0=(511, 511, 600, 1000), full_head=measured_head)
    w, fmt, sc = o["head"]
    run_and_check(dp, o, lambda x: full_head_oracle(w, x, fmt, sc))


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
