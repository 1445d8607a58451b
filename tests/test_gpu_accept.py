"""GPU parity of tfd_accept against the oracle: counts and histograms bit-exact."""
import itertools

import numpy as np
import pytest
import torch

from helpers import need_gpu
from oracle.accept import accept as oracle_accept
from speculative_decoding_draft_row_gb300 import tfd

pytestmark = pytest.mark.gpu


def test_every_pattern_of_a_five_draft_window():
    need_gpu()
    win = 5
    drafts, draws, asked = [], [], []
    for pattern in itertools.product([0, 1], repeat=win):
        for na in range(win + 1):
            d = np.arange(win) + 10
            drafts.append(d)
            draws.append(np.where(np.array(pattern) == 1, d, d + 100))
            asked.append(na)
    drafts = np.array(drafts, np.int32)
    draws = np.array(draws, np.int32)
    asked = np.array(asked, np.int32)
    ah = torch.full((win,), 3, dtype=torch.int64, device="cuda")
    kh = torch.full((win,), 1, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_kept = tfd.tfd_accept(torch.from_numpy(drafts).cuda(), torch.from_numpy(asked).cuda(),
                            torch.from_numpy(draws).cuda(), asked_hist=ah, kept_hist=kh,
                            dev_status=st)
    torch.cuda.synchronize()
    ok, oah, okh, bad = oracle_accept(drafts, asked, draws, [3] * win, [1] * win)
    assert np.array_equal(n_kept.cpu().numpy(), ok)
    assert np.array_equal(ah.cpu().numpy(), oah) and np.array_equal(kh.cpu().numpy(), okh)
    assert st.item() == 0 and not bad


def test_bad_asked_counts():
    need_gpu()
    drafts = torch.tensor([[1, 2], [1, 2], [1, 2]], dtype=torch.int32, device="cuda")
    asked = torch.tensor([2, 3, -1], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ah = torch.zeros(2, dtype=torch.int64, device="cuda")
    kh = torch.zeros(2, dtype=torch.int64, device="cuda")
    n_kept = tfd.tfd_accept(drafts, asked, drafts, asked_hist=ah, kept_hist=kh, dev_status=st)
    torch.cuda.synchronize()
    ok, oah, okh, bad = oracle_accept(drafts.cpu().numpy(), asked.cpu().numpy(),
                                      drafts.cpu().numpy())
    assert bad and st.item() == tfd.ERR_DEVICE_DATA
    assert np.array_equal(n_kept.cpu().numpy(), ok)
    assert np.array_equal(ah.cpu().numpy(), oah) and np.array_equal(kh.cpu().numpy(), okh)
