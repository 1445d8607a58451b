"""GPU parity of tfd_topk over given fp32 logits: ids and values bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from helpers import need_gpu, same_bits
from oracle.topk import topk as oracle_topk
from speculative_decoding_draft_row_gb300 import tfd
from synth import inputs

pytestmark = pytest.mark.gpu


def run(lg, k, id_map=None):
    d = torch.from_numpy(np.ascontiguousarray(lg)).cuda()
    idm = None if id_map is None else torch.from_numpy(np.asarray(id_map, np.int32)).cuda()
    v, i = tfd.tfd_topk(d, k, id_map=idm)
    torch.cuda.synchronize()
    return v.cpu().numpy(), i.cpu().numpy()


def tie_heavy(r, n, tid):
    rng = np.random.default_rng([0, tid, 0])
    pool = np.array([-np.inf, -1.5, -0.0, 0.0, 0.25, 1.0, 3.0, np.inf, np.nan], np.float32)
    out = pool[rng.integers(0, len(pool), size=(r, n))]
    return out


@pytest.mark.parametrize("rows,n,k", [(1, 1, 1), (1, 7, 7), (3, 1000, 1), (3, 1000, 8),
                                      (16, 4096, 64), (2, 5000, 512), (16, 163840, 1),
                                      (16, 163840, 64), (16, 163840, 512), (1, 163840, 512)])
def test_random_logits(rows, n, k):
    need_gpu()
    lg = inputs.normal_f32((rows, n), 1.0, 400 + k)
    v, i = run(lg, k)
    ov, oi = oracle_topk(lg, k)
    assert np.array_equal(i, oi) and same_bits(v, ov)


@pytest.mark.parametrize("rows,n,k", [(4, 3000, 1), (4, 3000, 16), (2, 20000, 512),
                                      (16, 163840, 64)])
def test_ties_zeros_infinities_nan(rows, n, k):
    need_gpu()
    lg = tie_heavy(rows, n, 410 + k)
    v, i = run(lg, k)
    ov, oi = oracle_topk(lg, k)
    assert np.array_equal(i, oi) and same_bits(v, ov)


def test_all_equal_values():
    need_gpu()
    lg = np.full((3, 50000), 0.5, np.float32)
    v, i = run(lg, 512)
    assert np.array_equal(i, np.tile(np.arange(512, dtype=np.int32), (3, 1)))
    assert np.all(v == 0.5)


def test_id_map_and_strided_rows():
    need_gpu()
    rows, n, ld, k = 5, 30000, 30016, 100
    full = tie_heavy(rows, ld, 420)
    idm = np.random.default_rng([0, 421, 0]).permutation(n).astype(np.int32) + 1000
    d = torch.from_numpy(full).cuda()
    vals, ids = tfd.tfd_topk(d, k, id_map=torch.from_numpy(idm).cuda(), n=n)
    torch.cuda.synchronize()
    ov, oi = oracle_topk(full[:, :n], k, id_map=idm)
    assert np.array_equal(ids.cpu().numpy(), oi) and same_bits(vals.cpu().numpy(), ov)


def test_workspace_is_left_zeroed_and_reusable():
    need_gpu()
    lg = inputs.normal_f32((16, 163840), 1.0, 430)
    d = torch.from_numpy(lg).cuda()
    ws = tfd.zeroed_workspace(tfd.tfd_topk_workspace(16, 163840, 64))
    for _ in range(3):
        v, i = tfd.tfd_topk(d, 64, ws=ws)
    torch.cuda.synchronize()
    ov, oi = oracle_topk(lg, 64)
    assert np.array_equal(i.cpu().numpy(), oi) and same_bits(v.cpu().numpy(), ov)


# ---- the threshold filter's own paths -----------------------------------------------------------

def narrow_offset(r, n, tid):
    """Logits 10 + 1e-3 N(0, 1): every sub-group maximum falls in one 12-bit bin of value keys."""
    return (10.0 + 1e-3 * inputs.normal_f32((r, n), 1.0, tid)).astype(np.float32)


def coarse_levels(r, n, tid):
    """N(0, 1) rounded to even integers: hundreds to tens of thousands of exact ties at the k-th
    value, enough at n = 163840, k = 512 to overflow a row's candidate list."""
    return (np.round(inputs.normal_f32((r, n), 1.0, tid) / 2) * 2).astype(np.float32)


def one_peak_per_subgroup(r, n, tid):
    """Each 16-logit sub-group holds one large value among small ones: the maxima are the top."""
    lg = inputs.normal_f32((r, n), 1e-3, tid)
    lg[:, ::16] += 5.0 + inputs.normal_f32((r, (n + 15) // 16), 1.0, tid + 1)
    return lg


@pytest.mark.parametrize("make,rows,n,k", [(narrow_offset, 4, 163840, 64),
                                           (narrow_offset, 2, 163840, 512),
                                           (coarse_levels, 3, 163840, 64),
                                           (coarse_levels, 2, 40000, 512),
                                           (coarse_levels, 2, 163840, 512),
                                           (one_peak_per_subgroup, 4, 100000, 300),
                                           (one_peak_per_subgroup, 2, 7777, 486)])
def test_threshold_filter_paths(make, rows, n, k):
    need_gpu()
    lg = make(rows, n, 440 + k)
    v, i = run(lg, k)
    ov, oi = oracle_topk(lg, k)
    assert np.array_equal(i, oi) and same_bits(v, ov)


@pytest.mark.parametrize("n,k", [(1000, 100), (8176, 512), (511, 33), (17, 2)])
def test_fewer_subgroups_than_k(n, k):
    """ceil(n / 16) < k: no threshold applies and every logit is a candidate."""
    need_gpu()
    lg = inputs.normal_f32((3, n), 1.0, 450 + k)
    v, i = run(lg, k)
    ov, oi = oracle_topk(lg, k)
    assert np.array_equal(i, oi) and same_bits(v, ov)


def test_mostly_nan_and_minus_inf_rows():
    need_gpu()
    rows, n, k = 3, 50000, 64
    lg = np.full((rows, n), np.nan, np.float32)
    lg[1, :] = -np.inf
    rng = np.random.default_rng([0, 460, 0])
    for r in range(rows):
        at = rng.choice(n, size=40, replace=False)
        lg[r, at] = rng.standard_normal(40).astype(np.float32)
    v, i = run(lg, k)
    ov, oi = oracle_topk(lg, k)
    assert np.array_equal(i, oi) and same_bits(v, ov)


@pytest.mark.parametrize("n,k", [(600000, 64), (524289, 7)])
def test_rows_longer_than_the_shared_memory_maxima(n, k):
    """Over 8 x 4096 x 16 logits a row's sub-group maxima live in the workspace."""
    need_gpu()
    lg = inputs.normal_f32((2, n), 1.0, 470 + k)
    v, i = run(lg, k)
    ov, oi = oracle_topk(lg, k)
    assert np.array_equal(i, oi) and same_bits(v, ov)
