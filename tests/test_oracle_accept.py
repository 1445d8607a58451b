"""Pins of the oracle's accept-prefix count: the page's rule on hand examples and on every equality
pattern of a 5-draft window (checked against a cumulative-product formulation)."""
import itertools
import json
import os

import numpy as np

from oracle.accept import accept

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def test_hand_examples():
    for ex in GOLD["accept_examples"]:
        n_kept, ah, kh, bad = accept([ex["drafts"]], [ex["n_asked"]], [ex["draws"]])
        assert n_kept[0] == ex["n_kept"] and not bad
        assert list(ah) == [1] * ex["n_asked"] + [0] * (5 - ex["n_asked"])
        assert list(kh) == [1] * ex["n_kept"] + [0] * (5 - ex["n_kept"])


def test_exhaustive_patterns():
    win = 5
    drafts, draws, asked = [], [], []
    for pattern in itertools.product([0, 1], repeat=win):
        for na in range(win + 1):
            d = np.arange(win) + 10
            w = np.where(np.array(pattern) == 1, d, d + 100)
            drafts.append(d), draws.append(w), asked.append(na)
    drafts, draws, asked = np.array(drafts), np.array(draws), np.array(asked)
    n_kept, ah, kh, bad = accept(drafts, asked, draws)
    eq = (drafts == draws).astype(np.int64)
    alive = np.cumprod(eq, axis=1) * (np.arange(win)[None, :] < asked[:, None])
    assert np.array_equal(n_kept, alive.sum(axis=1)) and not bad
    assert np.array_equal(ah, (np.arange(win)[None, :] < asked[:, None]).sum(axis=0))
    assert np.array_equal(kh, alive.sum(axis=0))


def test_accumulates_and_flags_bad_asked():
    n_kept, ah, kh, bad = accept([[1, 2], [1, 2]], [2, 3], [[1, 2], [1, 2]],
                                 asked_hist=[10, 10], kept_hist=[4, 4])
    assert bad and list(n_kept) == [2, 0]
    assert list(ah) == [11, 11] and list(kh) == [5, 5]
