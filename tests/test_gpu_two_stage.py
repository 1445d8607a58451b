"""GPU parity of the two-stage head (low-rank GEMVs, top-cand_k, exact rescore, argmax) and of
tfd_rescore alone, against the oracle."""
import numpy as np
import pytest
import torch

from helpers import assert_fp32_close, assert_topk_valid, need_gpu, np32, same_bits
from oracle import gemv as og
from oracle.numerics import fl32
from oracle.two_stage import rescore as oracle_rescore
from oracle.topk import topk as oracle_topk
from speculative_decoding_draft_row_gb300 import tfd
from synth import inputs

pytestmark = pytest.mark.gpu


def two_stage_gpu(a, b, w, x, cand_k):
    h, _, _ = tfd.tfd_head_gemv(b, tfd.W_BF16, None, x, tfd.OUT_F32)
    z, _, _ = tfd.tfd_head_gemv(a, tfd.W_BF16, None, h, tfd.OUT_F32)
    cv, ci = tfd.tfd_topk(z, cand_k)
    # the same candidates from the GEMV with its fused top-k (sub-group maxima from its epilogue)
    _, fv, fi = tfd.tfd_head_gemv(a, tfd.W_BF16, None, h, tfd.OUT_NONE, topk=cand_k)
    e, ids, vals = tfd.tfd_rescore(w, x, ci)
    torch.cuda.synchronize()
    assert torch.equal(fi, ci) and same_bits(np32(fv), np32(cv)), "fused top-k != top-k of z"
    return h, z, cv, ci, e, ids, vals


def check(a, b, w, x, cand_k):
    h, z, cv, ci, e, ids, vals = two_stage_gpu(a.cuda(), b.cuda(), w.cuda(), x.cuda(), cand_k)
    an, bn, wn, xn = (t.float().numpy() for t in (a, b, w, x))
    # h = B x: fp32 accumulation
    assert_fp32_close(np32(h), og.gemv_acc(bn, xn).astype(np.float32), og.gemv_abs_scale(bn, xn), "h")
    # z = A h, on the GPU's own h (the oracle's h may differ in the last bits)
    hg = np32(h)
    assert_fp32_close(np32(z), og.gemv_acc(an, hg).astype(np.float32), og.gemv_abs_scale(an, hg), "z")
    # candidates: bit-exact top-k of the GPU's z
    ov, oi = oracle_topk(np32(z), cand_k)
    assert np.array_equal(ci.cpu().numpy(), oi) and same_bits(np32(cv), ov)
    # ... and a valid top-k of the oracle's own chain: z_o = A fl32(B x). The GPU's z differs
    # from z_o by its own fp32 sums (1e-5 |A| |h|) and by A times the error of its h (1e-5 S_h
    # each, plus the oracle's fl32 of h): S = |A| (1.01 |h_o| + S_h) bounds both
    h_o = fl32(og.gemv_acc(bn, xn)).astype(np.float64)
    z_o = og.gemv_acc(an, h_o)
    S_z = np.abs(h_o) * 1.01 + og.gemv_abs_scale(bn, xn)
    S_z = S_z @ np.abs(an.astype(np.float64)).T
    assert_topk_valid(np32(cv), ci.cpu().numpy(), z_o, S_z, cand_k, what="candidates vs oracle z")
    # rescore of the GPU's candidates
    cand = ci.cpu().numpy()
    oe, _, _ = oracle_rescore(wn, xn, cand)
    S = np.stack([np.abs(wn[cand[r]]).astype(np.float64) @ np.abs(xn[r]).astype(np.float64)
                  for r in range(cand.shape[0])])
    assert_fp32_close(np32(e), oe, S, "exact logits")
    ge = np32(e)
    for r in range(cand.shape[0]):
        o = np.lexsort((cand[r], -ge[r]))[0]          # argmax of the GPU's own exact logits
        assert ids[r].item() == cand[r][o] and same_bits(np32(vals)[r:r + 1], ge[r, o:o + 1])
    # the draft's exact oracle logit is the best among the candidates, up to the fp32 tolerance
    gid = ids.cpu().numpy()
    for r in range(cand.shape[0]):
        j = int(np.flatnonzero(cand[r] == gid[r])[0])
        assert oe[r][j] >= np.nanmax(oe[r]) - 2e-5 * S[r].max()
    return ids.cpu().numpy()


@pytest.mark.parametrize("cand_k", [1, 64, 512])
def test_reduced_vocab(cand_k):
    need_gpu()
    vocab = 20480
    a = inputs.normal_bf16((vocab, 256), 0.05, 440)
    b = inputs.normal_bf16((256, 4096), 0.05, 441)
    w = inputs.normal_bf16((vocab, 4096), 0.02, 442)
    x = inputs.normal_bf16((16, 4096), 1.0, 443)
    check(a, b, w, x, cand_k)


def test_candidates_cover_the_vocabulary_gives_the_exact_argmax():
    need_gpu()
    vocab = 512
    a = inputs.normal_bf16((vocab, 256), 0.05, 450)
    b = inputs.normal_bf16((256, 1024), 0.05, 451)
    w = inputs.normal_bf16((vocab, 1024), 0.02, 452)
    x = inputs.normal_bf16((16, 1024), 1.0, 453)
    ids = check(a, b, w, x, 512)
    exact = og.gemv_acc(w.float().numpy(), x.float().numpy())
    S = og.gemv_abs_scale(w.float().numpy(), x.float().numpy())
    for r in range(16):
        srt = np.sort(exact[r])
        if srt[-1] - srt[-2] > 2e-5 * S[r].max():
            assert ids[r] == np.argmax(exact[r])


@pytest.mark.parametrize("cand_k", [1, 64, 512])
def test_full_two_stage(cand_k):
    need_gpu()
    a, b = inputs.low_rank()
    w, _ = inputs.head(tie_frac=0.01)
    x = inputs.rows(16)
    check(a, b, w, x, cand_k)


def test_rescore_bad_ids_and_ties():
    need_gpu()
    w = torch.zeros((6, 16), dtype=torch.bfloat16)
    w[2, 0] = 1.0
    w[4, 0] = 1.0
    x = torch.ones((1, 16), dtype=torch.bfloat16)
    cand = torch.tensor([[4, 2, 9, -1]], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    e, ids, vals = tfd.tfd_rescore(w.cuda(), x.cuda(), cand.cuda(), dev_status=st)
    torch.cuda.synchronize()
    oe, oi, ov = oracle_rescore(w.float().numpy(), x.float().numpy(), cand.numpy())
    assert ids.item() == oi[0] == 2 and vals.item() == ov[0]
    ge = np32(e)
    assert np.isnan(ge[0, 2]) and np.isnan(ge[0, 3]) and ge[0, 0] == 1.0
    assert st.item() == tfd.ERR_DEVICE_DATA
