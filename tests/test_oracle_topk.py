"""Pins of the oracle's top-k: brute force with Python's own sort, the page's tie rule, signed zeros,
NaN, the id map, and invariance to the number of parts."""
import json
import math
import os

import numpy as np
import pytest

from oracle.topk import CANON_NAN, canonical, topk, topk_parts

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def brute(row, k, ids):
    items = [(1 if math.isnan(v) else 0, 0.0 if math.isnan(v) else -v, int(i), v)
             for v, i in zip(row.tolist(), ids)]
    items.sort()
    return [(it[3], it[2]) for it in items[:k]]


def tie_heavy(r, n, tid):
    rng = np.random.default_rng([0, tid, 0])
    pool = np.array([-np.inf, -1.5, -0.0, 0.0, 0.25, 0.25, 1.0, 3.0, np.inf, np.nan], np.float32)
    return pool[rng.integers(0, len(pool), size=(r, n))]


@pytest.mark.parametrize("k", [1, 2, 5, 17, 64])
def test_brute_force_with_ties_zeros_nan(k):
    lg = tie_heavy(6, 97, 100 + k)
    vals, ids = topk(lg, k)
    for r in range(6):
        ref = brute(lg[r], k, range(97))
        assert list(ids[r]) == [i for _, i in ref]
        assert np.array_equal(vals[r].view(np.uint32), canonical([v for v, _ in ref]).view(np.uint32))


def test_page_tie_rule_lower_id():
    lg = np.array([[1.0, 3.0, 2.0, 3.0, 3.0, 0.5]], np.float32)
    vals, ids = topk(lg, 2)
    assert list(ids[0]) == [1, 3] and list(vals[0]) == [3.0, 3.0]
    assert GOLD["cand_k_range"]["max"] == 512


def test_zero_signs_and_nan_rank():
    lg = np.array([[-0.0, 0.0, np.nan, -np.inf, np.nan]], np.float32)
    vals, ids = topk(lg, 5)
    assert list(ids[0]) == [0, 1, 3, 2, 4]
    assert vals[0][0] == 0 and not np.signbit(vals[0][0])
    assert vals[0][3].view(np.uint32) == CANON_NAN.view(np.uint32)


def test_id_map_permutation_invariance():
    rng = np.random.default_rng([0, 110, 0])
    lg = tie_heavy(3, 200, 111)
    perm = rng.permutation(200)
    v1, i1 = topk(lg, 33)
    v2, i2 = topk(lg[:, perm], 33, id_map=perm)
    assert np.array_equal(i1, i2) and np.array_equal(v1.view(np.uint32), v2.view(np.uint32))


@pytest.mark.parametrize("parts", [1, 2, 3, 7, 64, 300])
def test_part_count_invariance(parts):
    lg = np.concatenate([tie_heavy(2, 300, 120), np.random.default_rng([0, 121, 0])
                        .standard_normal((2, 300)).astype(np.float32)], axis=0)
    for k in (1, 8, 64):
        v1, i1 = topk(lg, k)
        v2, i2 = topk_parts(lg, k, parts)
        assert np.array_equal(i1, i2) and np.array_equal(v1.view(np.uint32), v2.view(np.uint32))


def test_k_bounds():
    with pytest.raises(ValueError):
        topk(np.zeros((1, 4), np.float32), 5)
    with pytest.raises(ValueError):
        topk(np.zeros((1, 4), np.float32), 0)


def test_top1_confidence_closed_forms_and_softmax():
    from scipy.special import softmax

    from oracle.topk import top1_confidence
    n = 1000
    assert np.isclose(top1_confidence(np.zeros((1, n)))[0], 1.0 / n)
    two = np.full((1, 10), -np.inf)
    two[0, 3] = two[0, 7] = 2.5
    assert top1_confidence(two)[0] == 0.5
    lg = np.random.default_rng([0, 122, 0]).standard_normal((4, 5000)) * 3
    ref = softmax(lg, axis=1).max(axis=1)
    assert np.allclose(top1_confidence(lg), ref, rtol=1e-12)
    assert np.allclose(top1_confidence(lg + 123.0), ref, rtol=1e-9)
    withnan = lg.copy()
    withnan[:, 10] = np.nan
    withnan[:, 11] = -np.inf
    assert np.allclose(top1_confidence(withnan),
                       top1_confidence(np.delete(lg, [10, 11], axis=1)), rtol=1e-12)
    assert np.isnan(top1_confidence(np.full((1, 3), np.nan))[0])
