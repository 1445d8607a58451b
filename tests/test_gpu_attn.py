"""GPU parity of tfd_window_attn (qk_norm, RoPE, ring write, window attention) against the oracle."""
import numpy as np
import pytest
import torch

from helpers import check_window_attn, need_gpu, np32
from speculative_decoding_draft_row_gb300 import tfd
from synth import inputs

pytestmark = pytest.mark.gpu


def run_case(S, H, ring, window, pos, tid, gamma=False, eps=1e-6):
    """Runs tfd_window_attn and checks it against the oracle: ring keys and output held to their
    bf16 rounding, values and untouched ring rows exact."""
    D = 128
    q, k, v = (inputs.normal_bf16((S, H, D), 1.0, tid + i) for i in range(3))
    kr = inputs.normal_bf16((S * ring, H, D), 1.0, tid + 3).reshape(S, ring, H, D)
    vr = inputs.normal_bf16((S * ring, H, D), 1.0, tid + 4).reshape(S, ring, H, D)
    qg = inputs.normal_bf16((D,), 0.5, tid + 5) if gamma else None
    kg = inputs.normal_bf16((D,), 0.5, tid + 6) if gamma else None
    posd = torch.tensor(pos, dtype=torch.int32).cuda()
    krd, vrd = kr.clone().cuda(), vr.clone().cuda()
    out = tfd.tfd_window_attn(q.cuda(), k.cuda(), v.cuda(), posd, krd, vrd, window,
                              q_gamma=None if qg is None else qg.cuda(),
                              k_gamma=None if kg is None else kg.cuda(), eps=eps)
    torch.cuda.synchronize()
    f = lambda t: None if t is None else t.float().numpy()
    check_window_attn(np32(out), np32(krd), np32(vrd), f(q), f(k), f(v), pos, f(kr), f(vr), window,
                      q_gamma=f(qg), k_gamma=f(kg), eps=eps, what="attention")
    return out, v


@pytest.mark.parametrize("window", [511, 128, 1, 0])
def test_pass_shapes(window):
    need_gpu()
    out, v = run_case(4, 32, 528, window, [511, 512, 513, 515], 500)
    if window == 0:
        assert np.array_equal(np32(out).reshape(4, 32, 128), v.float().numpy())


def test_short_history_gamma_and_ring_wrap():
    need_gpu()
    run_case(3, 5, 20, 19, [0, 3, 1000], 520, gamma=True)


def test_large_position():
    need_gpu()
    run_case(2, 4, 64, 63, [100000, 262143], 530)


def test_negative_position_reports_and_skips():
    need_gpu()
    D = 128
    q = torch.zeros((2, 1, D), dtype=torch.bfloat16, device="cuda")
    kr = torch.zeros((2, 8, 1, D), dtype=torch.bfloat16, device="cuda")
    vr = torch.zeros_like(kr)
    out = torch.full((2, D), 7.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.tensor([-1, 2], dtype=torch.int32, device="cuda")
    tfd.tfd_window_attn(q, q, q, pos, kr, vr, 4, out=out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == tfd.ERR_DEVICE_DATA
    assert torch.all(out[0] == 7.0)
