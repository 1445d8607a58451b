"""tfd_head_gemv_noalloc: the head GEMV for callers that cannot allocate device memory (serving
loops that keep cudaMalloc, which can block or synchronise the device, off the hot path; plugins
whose host framework owns all device memory), running on the library's fixed scratch array. Checked through the C ABI against tfd_head_gemv with a caller
workspace, on two calls in a row (the second must not see the first's leftovers). This file is
collected last, and it also passes when run alone in a fresh process."""
import numpy as np
import pytest
import torch

from helpers import assert_fp32_close, need_gpu, np32
from oracle import gemv as og
from speculative_decoding_draft_row_gb300 import tfd
from synth import inputs

pytestmark = pytest.mark.gpu


def case(n, k, rows, tid):
    w = inputs.normal_bf16((n, k), 0.02, tid)
    x = inputs.normal_bf16((rows, k), 1.0, tid + 1)
    return w, x


@pytest.mark.parametrize("n,k,rows,topk", [(163840, 4096, 5, 1), (4096, 4096, 4, 8),
                                           (8192, 256, 16, 1)])
def test_matches_the_workspace_entry_point_on_two_calls(n, k, rows, topk):
    need_gpu()
    w, x1 = case(n, k, rows, 700)
    x2 = inputs.normal_bf16((rows, k), 1.0, 702)
    wd = w.cuda()
    for x in (x1, x2):
        xd = x.cuda()
        y_ref, v_ref, i_ref = tfd.tfd_head_gemv(wd, tfd.W_BF16, None, xd, tfd.OUT_F32, topk=topk)
        y_na = torch.empty_like(y_ref)
        v_na = torch.empty_like(v_ref)
        i_na = torch.empty_like(i_ref)
        tfd.tfd_head_gemv_noalloc(wd, tfd.W_BF16, None, xd, tfd.OUT_F32, y=y_na, topk=topk,
                                  top_vals=v_na, top_ids=i_na)
        torch.cuda.synchronize()
        S = og.gemv_abs_scale(w.float().numpy(), x.float().numpy())
        assert_fp32_close(np32(y_na), np32(y_ref), S, "no-alloc logits")
        assert_fp32_close(np32(v_na), np32(v_ref),
                          np.take_along_axis(S, i_ref.cpu().numpy().astype(np.int64), 1),
                          "no-alloc top values")
        assert torch.equal(i_na, i_ref)


def test_refuses_requests_larger_than_the_scratch():
    need_gpu()
    w, x = case(163840, 4096, 16, 710)
    wd, xd = w.cuda(), x.cuda()
    assert tfd.tfd_head_gemv_workspace(16, 163840, 64) > tfd.NOALLOC_SCRATCH_BYTES
    with pytest.raises(tfd.TfdError) as e:
        tfd.tfd_head_gemv_noalloc(wd, tfd.W_BF16, None, xd, tfd.OUT_NONE, topk=64)
    assert e.value.status == tfd.ERR_WORKSPACE
