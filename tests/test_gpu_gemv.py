"""GPU parity of tfd_head_gemv (bf16 / FP8 row / FP8 block weights, every output mode, fused
top-1 and top-k) against the oracle, on small ragged shapes and on the full 163840 x 4096 head."""
import numpy as np
import pytest
import torch

from helpers import (assert_bf16_rounding, assert_fp32_close, assert_sorted_keys, assert_topk_valid,
                     full_head_oracle, gemv_bf16_err,
                     need_gpu, np32, same_bits)
from oracle import gemv as og
from oracle.quant import quant_fp8_block32, quant_fp8_row
from oracle.topk import top1_confidence
from oracle.topk import topk as oracle_topk
from speculative_decoding_draft_row_gb300 import tfd
from synth import inputs

pytestmark = pytest.mark.gpu


def make_case(n, k, rows, wfmt, xf32=False, tid=300, tie_frac=0.0):
    w = inputs.normal_bf16((n, k), 0.02, tid)
    if tie_frac:
        inputs.copy_rows(w, *inputs.tie_rows(n, tie_frac, tensor_id=tid + 5))
    wn = w.float().numpy()
    if xf32:
        x = torch.from_numpy(inputs.normal_f32((rows, k), 1.0, tid + 1))
    else:
        x = inputs.normal_bf16((rows, k), 1.0, tid + 1)
    xn = x.float().numpy()
    if wfmt == tfd.W_BF16:
        return dict(w=w.cuda(), scales=None, wo=wn, so=None, x=x.cuda(), xo=xn)
    if wfmt == tfd.W_FP8_ROW:
        c, s = quant_fp8_row(wn)
        return dict(w=torch.from_numpy(c).cuda(), scales=torch.from_numpy(s).cuda(), wo=c, so=s,
                    x=x.cuda(), xo=xn)
    c, s = quant_fp8_block32(wn)
    return dict(w=torch.from_numpy(c).cuda(), scales=torch.from_numpy(s).cuda(), wo=c, so=s,
                x=x.cuda(), xo=xn)


def oracle_acc_S(case, wfmt):
    acc = og.gemv_acc(case["wo"], case["xo"], wfmt, case["so"])
    S = og.gemv_abs_scale(case["wo"], case["xo"], wfmt, case["so"])
    return acc, S


SHAPES = [  # (n, k, rows, wfmt, xf32)
    (4096, 256, 1, tfd.W_BF16, False),        # the tiny draft step
    (1000, 272, 3, tfd.W_BF16, False),        # ragged n and k
    (63, 16, 9, tfd.W_BF16, False),
    (4177, 4096, 16, tfd.W_BF16, False),
    (2048, 256, 16, tfd.W_BF16, True),        # fp32 activations (low-rank second GEMV)
    (65553, 256, 16, tfd.W_BF16, True),       # short k, many rows: one k-slice, 256-row groups
    (4096, 4096, 17, tfd.W_BF16, False),      # 17-32 rows: four n-tiles, k split over a cluster
    (32768, 4096, 32, tfd.W_BF16, False),
    (4177, 1040, 24, tfd.W_BF16, False),
    (4096, 4096, 32, tfd.W_FP8_ROW, False),
    (2048, 4096, 20, tfd.W_FP8_BLOCK32, False),
    (65536, 272, 3, tfd.W_BF16, False),
    (40000, 64, 9, tfd.W_BF16, False),
    (1000, 272, 5, tfd.W_FP8_ROW, False),
    (4096, 4096, 4, tfd.W_FP8_ROW, False),    # wo
    (4096, 11008, 4, tfd.W_FP8_ROW, False),   # w2
    (4160, 1024, 16, tfd.W_FP8_ROW, False),
    (2048, 4096, 10, tfd.W_FP8_BLOCK32, False),
    (96, 96, 1, tfd.W_FP8_BLOCK32, False),
    (4096, 512, 16, tfd.W_FP8_BLOCK32, True),
]


@pytest.mark.parametrize("n,k,rows,wfmt,xf32", SHAPES)
def test_f32_logits_and_top1(n, k, rows, wfmt, xf32):
    need_gpu()
    case = make_case(n, k, rows, wfmt, xf32)
    y, tv, ti = tfd.tfd_head_gemv(case["w"], wfmt, case["scales"], case["x"], tfd.OUT_F32, topk=1)
    torch.cuda.synchronize()
    acc, S = oracle_acc_S(case, wfmt)
    yg = np32(y)
    assert_fp32_close(yg, acc.astype(np.float32), S, "logits")
    ov, oi = oracle_topk(yg, 1)                    # the fused top-1 is the top-1 of its own logits
    assert np.array_equal(np32(ti).astype(np.int32), oi) and same_bits(np32(tv), ov)
    assert_topk_valid(np32(tv), ti.cpu().numpy(), acc, S, 1, what="top-1")


@pytest.mark.parametrize("out_mode", [tfd.OUT_BF16, tfd.OUT_ADD_BF16, tfd.OUT_NONE])
@pytest.mark.parametrize("wfmt", [tfd.W_BF16, tfd.W_FP8_ROW, tfd.W_FP8_BLOCK32])
def test_output_modes(out_mode, wfmt):
    need_gpu()
    n, k, rows = 4096, 4096, 4
    case = make_case(n, k, rows, wfmt, tid=310)
    res = inputs.normal_bf16((rows, n), 1.0, 315)
    y = res.clone().cuda() if out_mode == tfd.OUT_ADD_BF16 else None
    y, tv, ti = tfd.tfd_head_gemv(case["w"], wfmt, case["scales"], case["x"], out_mode, y=y,
                                  topk=1)
    torch.cuda.synchronize()
    acc, S = oracle_acc_S(case, wfmt)
    if out_mode == tfd.OUT_BF16:
        assert_bf16_rounding(np32(y), acc, gemv_bf16_err(S), "out bf16")
    elif out_mode == tfd.OUT_ADD_BF16:
        ex = res.float().numpy().astype(np.float64) + acc
        assert_bf16_rounding(np32(y), ex, gemv_bf16_err(S, ex), "out added to bf16")
    else:
        assert y is None
    assert_topk_valid(np32(tv), ti.cpu().numpy(), acc, S, 1, what="top-1")


@pytest.mark.parametrize("wfmt", [tfd.W_BF16, tfd.W_FP8_ROW, tfd.W_FP8_BLOCK32])
def test_fused_topk_matches_own_logits_and_oracle(wfmt):
    need_gpu()
    case = make_case(8192, 4096, 16, wfmt, tid=320, tie_frac=0.01)
    acc, S = oracle_acc_S(case, wfmt)
    for k in (8, 64, 512):
        y, tv, ti = tfd.tfd_head_gemv(case["w"], wfmt, case["scales"], case["x"], tfd.OUT_F32,
                                      topk=k)
        _, tv2, ti2 = tfd.tfd_head_gemv(case["w"], wfmt, case["scales"], case["x"], tfd.OUT_NONE,
                                        topk=k)
        torch.cuda.synchronize()
        yg = np32(y)
        ov, oi = oracle_topk(yg, k)
        assert np.array_equal(ti.cpu().numpy(), oi) and same_bits(np32(tv), ov)
        assert np.array_equal(ti2.cpu().numpy(), oi) and same_bits(np32(tv2), ov)
        assert_sorted_keys(np32(tv), ti.cpu().numpy())
        assert_topk_valid(np32(tv), ti.cpu().numpy(), acc, S, k, what=f"top-{k}")


@pytest.mark.parametrize("n,k,rows,xf32", [(4096, 4096, 1, False), (4096, 4096, 10, False),
                                           (2080, 1088, 16, False), (2048, 512, 7, True)])
def test_block32_interleaved_equals_plain_bit_for_bit(n, k, rows, xf32):
    """The interleaved block-32 layout changes only how the codes are loaded: logits and top-k
    are bit-identical to the plain layout's."""
    need_gpu()
    case = make_case(n, k, rows, tfd.W_FP8_BLOCK32, xf32, tid=350)
    il = tfd.tfd_fp8_block32_relayout(case["w"], True)
    y0, v0, i0 = tfd.tfd_head_gemv(case["w"], tfd.W_FP8_BLOCK32, case["scales"], case["x"],
                                   tfd.OUT_F32, topk=16)
    y1, v1, i1 = tfd.tfd_head_gemv(il, tfd.W_FP8_BLOCK32_IL, case["scales"], case["x"],
                                   tfd.OUT_F32, topk=16)
    torch.cuda.synchronize()
    assert same_bits(np32(y0), np32(y1)) and torch.equal(i0, i1) and same_bits(np32(v0), np32(v1))
    acc, S = oracle_acc_S(case, tfd.W_FP8_BLOCK32)
    assert_fp32_close(np32(y1), acc, S, "interleaved block-32 logits")


def scaled_block_case(n, k, rows, tid):
    """FP8 block-32 codes of weights whose 32 x 32 blocks differ in magnitude (factors from 2^-6
    to 2^5, some blocks all zero), so that neighbouring blocks of a row block get different E8M0
    scales (and zero scale bytes)."""
    rng = np.random.default_rng(tid)
    w = inputs.normal_bf16((n, k), 0.05, tid).float().numpy()
    f = rng.choice(np.array([0.0, 2.0 ** -6, 0.3, 1.0, 1.0, 1.0, 5.5, 32.0], np.float32),
                   size=(n // 32, k // 32))
    w = w * np.repeat(np.repeat(f, 32, 0), 32, 1)
    w = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    c, sc = quant_fp8_block32(w)
    x = inputs.normal_bf16((rows, k), 1.0, tid + 1)
    return c, sc, x


@pytest.mark.parametrize("n,k,rows", [(2048, 4096, 16), (2080, 1088, 5), (4096, 4096, 1),
                                      (2048, 4096, 32)])
def test_block32_scales_that_differ_between_blocks(n, k, rows):
    """Block scales that change from one 32-wide block to the next (and all-zero blocks): the
    plain and interleaved layouts, W16 and W8A8, against the oracle; the two layouts bit-equal."""
    need_gpu()
    c, sc, x = scaled_block_case(n, k, rows, 380 + rows)
    xn = x.float().numpy()
    cd, sd, xd = torch.from_numpy(c).cuda(), torch.from_numpy(sc).cuda(), x.cuda()
    il = tfd.tfd_fp8_block32_relayout(cd, True)
    y0, v0, i0 = tfd.tfd_head_gemv(cd, tfd.W_FP8_BLOCK32, sd, xd, tfd.OUT_F32, topk=16)
    y1, v1, i1 = tfd.tfd_head_gemv(il, tfd.W_FP8_BLOCK32_IL, sd, xd, tfd.OUT_F32, topk=16)
    torch.cuda.synchronize()
    assert same_bits(np32(y0), np32(y1)) and torch.equal(i0, i1) and same_bits(np32(v0), np32(v1))
    acc = og.gemv_acc(c, xn, og.W_FP8_BLOCK32, sc)
    S = og.gemv_abs_scale(c, xn, og.W_FP8_BLOCK32, sc)
    assert_fp32_close(np32(y1), acc, S, "block-32 logits, mixed scales")
    assert_topk_valid(np32(v1), i1.cpu().numpy(), acc, S, 16, what="top-16, mixed scales")
    if rows <= 16:
        y2, _, _ = tfd.tfd_head_gemv(il, tfd.W_FP8_BLOCK32_IL, sd, xd, tfd.OUT_F32, act_e4m3=True)
        torch.cuda.synchronize()
        acc = og.gemv_acc(c, xn, og.W_FP8_BLOCK32, sc, act_fp8=True)
        S = og.gemv_abs_scale(c, xn, og.W_FP8_BLOCK32, sc, act_fp8=True)
        assert_fp32_close(np32(y2), acc, S, "W8A8 block-32 logits, mixed scales")


W8A8_SHAPES = [(4096, 4096, 1, tfd.W_FP8_ROW), (4096, 4096, 10, tfd.W_FP8_ROW),
               (4096, 4096, 32, tfd.W_FP8_ROW), (2080, 4096, 25, tfd.W_FP8_BLOCK32_IL),
               (1000, 272, 3, tfd.W_FP8_ROW), (4096, 11008, 4, tfd.W_FP8_ROW),
               (4096, 4096, 5, tfd.W_FP8_BLOCK32), (2080, 1088, 16, tfd.W_FP8_BLOCK32),
               (4096, 4096, 9, tfd.W_FP8_BLOCK32_IL), (2080, 1088, 1, tfd.W_FP8_BLOCK32_IL)]


@pytest.mark.parametrize("n,k,rows,wfmt", W8A8_SHAPES)
def test_w8a8(n, k, rows, wfmt):
    """Activations quantised per row to E4M3 in the call (W8A8): fp32-accumulation tolerance
    against the oracle's exact product of the decoded codes; fused top-8 of its own logits."""
    need_gpu()
    base = tfd.W_FP8_BLOCK32 if wfmt == tfd.W_FP8_BLOCK32_IL else wfmt
    case = make_case(n, k, rows, base, tid=370)
    w = case["w"] if wfmt != tfd.W_FP8_BLOCK32_IL else tfd.tfd_fp8_block32_relayout(case["w"], True)
    y, tv, ti = tfd.tfd_head_gemv(w, wfmt, case["scales"], case["x"], tfd.OUT_F32, topk=8,
                                  act_e4m3=True)
    torch.cuda.synchronize()
    acc = og.gemv_acc(case["wo"], case["xo"], base, case["so"], act_fp8=True)
    S = og.gemv_abs_scale(case["wo"], case["xo"], base, case["so"], act_fp8=True)
    assert_fp32_close(np32(y), acc, S, "W8A8 logits")
    ov, oi = oracle_topk(np32(y), 8)
    assert np.array_equal(ti.cpu().numpy(), oi) and same_bits(np32(tv), ov)


def test_w8a8_zero_row_and_refusals():
    need_gpu()
    case = make_case(4096, 4096, 3, tfd.W_FP8_ROW, tid=375)
    x = case["x"].clone()
    x[1] = 0
    y, _, _ = tfd.tfd_head_gemv(case["w"], tfd.W_FP8_ROW, case["scales"], x, tfd.OUT_F32,
                                act_e4m3=True)
    torch.cuda.synchronize()
    assert torch.all(y[1] == 0)
    assert not torch.isnan(y).any()
    wb = inputs.normal_bf16((64, 256), 0.02, 376).cuda()
    with pytest.raises(tfd.TfdError):
        tfd.tfd_head_gemv(wb, tfd.W_BF16, None, inputs.rows(2, 256).cuda(), tfd.OUT_F32,
                          act_e4m3=True)


@pytest.mark.parametrize("wfmt,rows", [(tfd.W_BF16, 32), (tfd.W_FP8_BLOCK32_IL, 19)])
def test_32_row_window_fused_topk_and_confidence(wfmt, rows):
    """A 32-row decode window: fused top-64 and top-1 with its confidence, against the oracle."""
    need_gpu()
    base = tfd.W_FP8_BLOCK32 if wfmt == tfd.W_FP8_BLOCK32_IL else wfmt
    case = make_case(8192, 4096, rows, base, tid=380, tie_frac=0.01)
    w = case["w"] if wfmt != tfd.W_FP8_BLOCK32_IL else tfd.tfd_fp8_block32_relayout(case["w"], True)
    y, tv, ti = tfd.tfd_head_gemv(w, wfmt, case["scales"], case["x"], tfd.OUT_F32, topk=64)
    conf = torch.empty(rows, dtype=torch.float32, device="cuda")
    _, v1, i1 = tfd.tfd_head_gemv(w, wfmt, case["scales"], case["x"], tfd.OUT_NONE, topk=1,
                                  top1_conf=conf)
    torch.cuda.synchronize()
    acc, S = oracle_acc_S(case, base)
    assert_fp32_close(np32(y), acc, S, "logits")
    ov, oi = oracle_topk(np32(y), 64)
    assert np.array_equal(ti.cpu().numpy(), oi) and same_bits(np32(tv), ov)
    assert np.array_equal(i1.cpu().numpy()[:, 0], oi[:, 0])
    assert np.allclose(np32(conf), top1_confidence(np32(y)), rtol=1e-4)


def test_fused_topk_over_a_long_ragged_vocabulary():
    """270016 logits a row (not a multiple of 8 x 16): the fused top-k from the GEMV's sub-group
    maxima, ragged parts at the end of the row."""
    need_gpu()
    case = make_case(270016, 64, 3, tfd.W_BF16, tid=360, tie_frac=0.01)
    y, tv, ti = tfd.tfd_head_gemv(case["w"], tfd.W_BF16, None, case["x"], tfd.OUT_F32, topk=100)
    torch.cuda.synchronize()
    ov, oi = oracle_topk(np32(y), 100)
    assert np.array_equal(ti.cpu().numpy(), oi) and same_bits(np32(tv), ov)


def test_fused_topk_with_one_k_slice():
    """The short-k, many-row form (one k-slice per block, 256-row groups) with a fused top-64."""
    need_gpu()
    case = make_case(65553, 256, 16, tfd.W_BF16, xf32=True, tid=340, tie_frac=0.01)
    acc, S = oracle_acc_S(case, tfd.W_BF16)
    y, tv, ti = tfd.tfd_head_gemv(case["w"], tfd.W_BF16, None, case["x"], tfd.OUT_F32, topk=64)
    _, tv1, ti1 = tfd.tfd_head_gemv(case["w"], tfd.W_BF16, None, case["x"], tfd.OUT_F32, topk=1)
    torch.cuda.synchronize()
    assert_fp32_close(np32(y), acc, S, "logits")
    ov, oi = oracle_topk(np32(y), 64)
    assert np.array_equal(ti.cpu().numpy(), oi) and same_bits(np32(tv), ov)
    assert np.array_equal(ti1.cpu().numpy()[:, 0], oi[:, 0])
    assert same_bits(np32(tv1)[:, 0], ov[:, 0])


@pytest.mark.parametrize("out_mode,rows,n", [(tfd.OUT_BF16, 16, 8192), (tfd.OUT_ADD_BF16, 5, 8000),
                                             (tfd.OUT_NONE, 9, 8016)])
def test_fused_topk_ranks_the_fp32_logits_in_every_output_mode(out_mode, rows, n):
    """The fused top-k ranks the fp32 logits, whatever the stored output; a vocabulary that ends
    inside a 64-row group and a 16-row sub-group included."""
    need_gpu()
    case = make_case(n, 1024, rows, tfd.W_BF16, tid=330, tie_frac=0.01)
    y32, tv, ti = tfd.tfd_head_gemv(case["w"], tfd.W_BF16, None, case["x"], tfd.OUT_F32, topk=100)
    y = None
    if out_mode == tfd.OUT_ADD_BF16:
        y = torch.zeros((rows, n), dtype=torch.bfloat16, device="cuda")
    _, tv2, ti2 = tfd.tfd_head_gemv(case["w"], tfd.W_BF16, None, case["x"], out_mode, y=y, topk=100)
    torch.cuda.synchronize()
    ov, oi = oracle_topk(np32(y32), 100)
    assert np.array_equal(ti.cpu().numpy(), oi) and same_bits(np32(tv), ov)
    assert torch.equal(ti2, ti) and same_bits(np32(tv2), np32(tv))


@pytest.mark.parametrize("wfmt,rows", [(tfd.W_BF16, 1), (tfd.W_BF16, 16), (tfd.W_FP8_ROW, 5),
                                       (tfd.W_BF16, 24)])
def test_top1_confidence(wfmt, rows):
    need_gpu()
    case = make_case(20480, 4096, rows, wfmt, tid=380, tie_frac=0.01)
    conf = torch.empty(rows, dtype=torch.float32, device="cuda")
    y, tv, ti = tfd.tfd_head_gemv(case["w"], wfmt, case["scales"], case["x"], tfd.OUT_F32, topk=1,
                                  top1_conf=conf)
    torch.cuda.synchronize()
    acc, S = oracle_acc_S(case, wfmt)
    c = conf.cpu().numpy().astype(np.float64)
    # against the confidence of the GPU's own fp32 logits: fp32 summation error only
    assert np.allclose(c, top1_confidence(np32(y)), rtol=1e-4, atol=0)
    # against the exact logits: each logit is within 1e-5 S, so the ratio within 2e-5 max S
    tol = 2e-5 * S.max(axis=1) + 1e-4
    assert np.all(np.abs(c - top1_confidence(acc)) <= tol * top1_confidence(acc))
    # the confidence does not change the top-1
    _, tv2, ti2 = tfd.tfd_head_gemv(case["w"], wfmt, case["scales"], case["x"], tfd.OUT_F32, topk=1)
    torch.cuda.synchronize()
    assert torch.equal(ti, ti2) and torch.equal(tv, tv2)


def test_part_count_does_not_change_results():
    need_gpu()
    case = make_case(20480, 4096, 5, tfd.W_BF16, tid=330, tie_frac=0.01)
    ref = None
    for parts in (0, 1, 2, 7, 64, 320, 1024):
        y, tv, ti = tfd.tfd_head_gemv(case["w"], tfd.W_BF16, None, case["x"], tfd.OUT_F32, topk=1,
                                      parts=parts)
        torch.cuda.synchronize()
        got = (np32(y), np32(tv), ti.cpu().numpy())
        if ref is None:
            ref = got
        else:
            assert same_bits(got[0], ref[0]) and same_bits(got[1], ref[1])
            assert np.array_equal(got[2], ref[2])


@pytest.mark.parametrize("wfmt", [tfd.W_BF16, tfd.W_FP8_ROW, tfd.W_FP8_BLOCK32])
def test_planted_ties_go_to_the_lower_id(wfmt):
    """Each activation row's best weight row is copied (with its whole 32-row block, so that every
    weight form stays identical) into another part of the vocabulary, below or above it: the
    duplicates must get bit-identical logits and the lower id must win."""
    need_gpu()
    n, k, rows = 20480, 4096, 8
    w = inputs.normal_bf16((n, k), 0.02, 340)
    x = inputs.normal_bf16((rows, k), 1.0, 341)
    acc0 = og.gemv_acc(w.float().numpy(), x.float().numpy())
    for r, src in enumerate(np.argmax(acc0, axis=1)):
        b = int(src) // 32
        b2 = (b + n // 64 + 7 * r) % (n // 32)
        w[b2 * 32:(b2 + 1) * 32] = w[b * 32:(b + 1) * 32].clone()
    wn = w.float().numpy()
    if wfmt == tfd.W_BF16:
        wd, sd, wo, so = w.cuda(), None, wn, None
    else:
        c, s = (quant_fp8_row if wfmt == tfd.W_FP8_ROW else quant_fp8_block32)(wn)
        wd, sd, wo, so = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), c, s
    y, tv, ti = tfd.tfd_head_gemv(wd, wfmt, sd, x.cuda(), tfd.OUT_F32, topk=1)
    torch.cuda.synchronize()
    yg = np32(y)
    acc = og.gemv_acc(wo, x.float().numpy(), wfmt, so)
    S = og.gemv_abs_scale(wo, x.float().numpy(), wfmt, so)
    tied = 0
    for r in range(rows):
        top = acc[r].max()
        best = np.flatnonzero(acc[r] == top)
        rest = acc[r][acc[r] < top]
        clear = top - rest.max() > 2e-5 * S[r].max()
        if len(best) > 1:
            assert len(set(yg[r, best].view(np.uint32).tolist())) == 1
            if clear:
                tied += 1
                assert ti[r, 0].item() == best.min()
    assert tied >= rows // 2


def test_id_map_reports_mapped_ids_and_breaks_ties_by_them():
    need_gpu()
    n, k, rows = 4096, 256, 6
    case = make_case(n, k, rows, tfd.W_BF16, tid=350)
    perm = np.random.default_rng([0, 351, 0]).permutation(n).astype(np.int32)
    wp = case["w"][torch.from_numpy(perm.astype(np.int64)).cuda()]
    idm = torch.from_numpy(perm).cuda()
    y1, tv1, ti1 = tfd.tfd_head_gemv(case["w"], tfd.W_BF16, None, case["x"], tfd.OUT_F32, topk=1)
    y2, tv2, ti2 = tfd.tfd_head_gemv(wp, tfd.W_BF16, None, case["x"], tfd.OUT_F32, topk=1,
                                     id_map=idm)
    _, tv3, ti3 = tfd.tfd_head_gemv(wp, tfd.W_BF16, None, case["x"], tfd.OUT_F32, topk=16,
                                    id_map=idm)
    torch.cuda.synchronize()
    assert np.array_equal(ti1.cpu().numpy(), ti2.cpu().numpy()) and same_bits(np32(tv1), np32(tv2))
    ov, oi = oracle_topk(np32(y2), 16, id_map=perm)
    assert np.array_equal(ti3.cpu().numpy(), oi) and same_bits(np32(tv3), ov)


def test_fp8_decode_is_exact_for_every_code():
    """One-hot activations pick single columns: y = scale * dec(code), exactly, for all codes
    (subnormal codes included) and for every byte position within a 16-byte weight chunk."""
    need_gpu()
    codes = np.arange(256, dtype=np.uint8)
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    n, k, rows = 256, 64, 16
    cm = np.zeros((n, k), np.uint8)
    for c in range(rows):
        cm[:, c] = np.roll(codes, 17 * c)
    s = np.exp2(np.random.default_rng([0, 360, 0]).integers(-20, 5, n)).astype(np.float32)
    x = np.zeros((rows, k), np.float32)
    for r in range(rows):
        x[r, r] = (-1.0) ** r * 2.0 ** (r - 6)
    xd = torch.from_numpy(x).to(torch.bfloat16).cuda()
    y, _, _ = tfd.tfd_head_gemv(torch.from_numpy(cm).cuda(), tfd.W_FP8_ROW,
                                torch.from_numpy(s).cuda(), xd, tfd.OUT_F32)
    torch.cuda.synchronize()
    assert same_bits(np32(y), og.gemv(cm, x, og.W_FP8_ROW, s, og.OUT_F32))
    sb = np.full((n // 32, k // 32), 120, np.uint8)
    sb[3, 0] = 0
    sb[5, 1] = 200
    yb, _, _ = tfd.tfd_head_gemv(torch.from_numpy(cm).cuda(), tfd.W_FP8_BLOCK32,
                                 torch.from_numpy(sb).cuda(), xd, tfd.OUT_F32)
    torch.cuda.synchronize()
    assert same_bits(np32(yb), og.gemv(cm, x, og.W_FP8_BLOCK32, sb, og.OUT_F32))


def test_add_bf16_in_place_on_a_strided_output():
    need_gpu()
    n, k, rows = 4096, 4096, 4
    case = make_case(n, k, rows, tfd.W_FP8_ROW, tid=370)
    big = inputs.normal_bf16((rows, n + 64), 1.0, 371).cuda()
    y = big[:, 32:32 + n]
    before = big.clone()
    tfd.tfd_head_gemv(case["w"], tfd.W_FP8_ROW, case["scales"], case["x"], tfd.OUT_ADD_BF16, y=y)
    torch.cuda.synchronize()
    acc, S = oracle_acc_S(case, tfd.W_FP8_ROW)
    ex = np32(before[:, 32:32 + n]).astype(np.float64) + acc
    assert_bf16_rounding(np32(y), ex, gemv_bf16_err(S, ex), "in place, strided")
    assert torch.equal(big[:, :32], before[:, :32]) and torch.equal(big[:, 32 + n:],
                                                                    before[:, 32 + n:])


@pytest.fixture(scope="module")
def full_head():
    need_gpu()
    w, ties = inputs.head(tie_frac=0.01)
    return w, w.cuda(), ties


@pytest.mark.parametrize("rows", [1, 5, 10, 15, 16])
def test_full_bf16_head(full_head, rows):
    need_gpu()
    w, wd, ties = full_head
    x = inputs.rows(16)[:rows]
    y, tv, ti = tfd.tfd_head_gemv(wd, tfd.W_BF16, None, x.cuda(), tfd.OUT_F32, topk=1, parts=64)
    _, tv2, ti2 = tfd.tfd_head_gemv(wd, tfd.W_BF16, None, x.cuda(), tfd.OUT_F32, topk=1)
    torch.cuda.synchronize()
    yg = np32(y)
    acc, S = full_head_oracle(w.float().numpy(), x.float().numpy())
    assert_fp32_close(yg, acc.astype(np.float32), S, "full-head logits")
    ov, oi = oracle_topk(yg, 1)
    assert np.array_equal(ti.cpu().numpy(), oi) and same_bits(np32(tv), ov)
    assert np.array_equal(ti2.cpu().numpy(), oi)
    assert_topk_valid(np32(tv), ti.cpu().numpy(), acc, S, 1, what="full top-1")
    dst, src = ties
    assert same_bits(yg[:, dst], yg[:, src])          # planted duplicates: identical logits


@pytest.mark.parametrize("mode", [tfd.W_FP8_BLOCK32, tfd.W_FP8_ROW])
@pytest.mark.parametrize("rows", [1, 15])
def test_full_fp8_head_top64(full_head, mode, rows):
    need_gpu()
    w, wd, _ = full_head
    codes, scales = tfd.tfd_quant_fp8(wd, mode)
    x = inputs.rows(16)[:rows]
    y, tv, ti = tfd.tfd_head_gemv(codes, mode, scales, x.cuda(), tfd.OUT_F32, topk=64)
    _, tv2, ti2 = tfd.tfd_head_gemv(codes, mode, scales, x.cuda(), tfd.OUT_NONE, topk=64)
    torch.cuda.synchronize()
    c = codes.cpu().numpy()
    s = scales.cpu().numpy()
    acc, S = full_head_oracle(c, x.float().numpy(), mode, s)
    yg = np32(y)
    assert_fp32_close(yg, acc.astype(np.float32), S, "fp8 logits")
    ov, oi = oracle_topk(yg, 64)
    assert np.array_equal(ti.cpu().numpy(), oi) and same_bits(np32(tv), ov)
    assert np.array_equal(ti2.cpu().numpy(), oi) and same_bits(np32(tv2), ov)
    assert_topk_valid(np32(tv), ti.cpu().numpy(), acc, S, 64, what="fp8 top-64")


@pytest.mark.parametrize("parts,k", [(64, 64), (65, 64), (300, 100), (1000, 512), (64, 100)])
def test_fused_topk_threshold_from_part_maxima(parts, k):
    """With k <= parts the fused top-k takes its threshold from the k-th largest part maximum (one
    block per row); otherwise from the sub-group maxima (a cluster per row). Either way the result
    is the exact top-k of the call's own logits."""
    need_gpu()
    case = make_case(40960, 1024, 9, tfd.W_BF16, tid=390, tie_frac=0.01)
    y, tv, ti = tfd.tfd_head_gemv(case["w"], tfd.W_BF16, None, case["x"], tfd.OUT_F32, topk=k,
                                  parts=parts)
    torch.cuda.synchronize()
    ov, oi = oracle_topk(np32(y), k)
    assert np.array_equal(ti.cpu().numpy(), oi) and same_bits(np32(tv), ov)


def test_fused_topk_of_all_equal_logits_falls_back_to_the_exact_select():
    """Zero weights give a row of equal logits: every logit reaches the threshold, the candidate
    list overflows, and the exact select over the row must still give the k lowest ids."""
    need_gpu()
    w = torch.zeros((65536, 256), dtype=torch.bfloat16, device="cuda")
    x = inputs.normal_bf16((3, 256), 1.0, 395).cuda()
    _, tv, ti = tfd.tfd_head_gemv(w, tfd.W_BF16, None, x, tfd.OUT_NONE, topk=64)
    torch.cuda.synchronize()
    assert np.array_equal(ti.cpu().numpy(), np.tile(np.arange(64, dtype=np.int32), (3, 1)))
    assert np.all(np32(tv) == 0.0)


@pytest.mark.parametrize("wfmt,rows,topk", [(tfd.W_BF16, 1, 1), (tfd.W_FP8_ROW, 16, 64),
                                            (tfd.W_FP8_BLOCK32, 9, 8), (tfd.W_BF16, 12, 0)])
def test_group_queue_repeats_bit_for_bit_and_leaves_the_counters_zero(wfmt, rows, topk):
    """Calls with a workspace take 64-row groups from a queue shared by the blocks, so which block
    computes a group changes from call to call: logits and top-k must still repeat bit for bit,
    and each call must leave the workspace's counters at zero for the next."""
    need_gpu()
    case = make_case(65536, 4096, rows, wfmt, tid=397, tie_frac=0.01)
    ws = tfd.zeroed_workspace(max(256, tfd.tfd_head_gemv_workspace(rows, 65536, topk)))
    outs = []
    for _ in range(3):
        y, tv, ti = tfd.tfd_head_gemv(case["w"], wfmt, case["scales"], case["x"], tfd.OUT_F32,
                                      topk=topk, ws=ws)
        torch.cuda.synchronize()
        assert torch.all(ws[:256] == 0), "counters left non-zero"
        outs.append((np32(y), None if ti is None else (np32(tv), ti.cpu().numpy())))
    for y, t in outs[1:]:
        assert same_bits(y, outs[0][0])
        if t is not None:
            assert same_bits(t[0], outs[0][1][0]) and np.array_equal(t[1], outs[0][1][1])
    if topk:
        ov, oi = oracle_topk(outs[0][0], topk)
        assert np.array_equal(outs[0][1][1], oi) and same_bits(outs[0][1][0], ov)
