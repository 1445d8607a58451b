"""Pins of the oracle's two-stage head: cand_k = vocab is the exact argmax, cand_k = 1 is the
low-rank argmax, more candidates never lower the pick, and bad candidate ids rank last."""
import numpy as np

from oracle.two_stage import low_rank_logits, rescore, two_stage
from synth import inputs


def case(vocab=512, rank=16, hidden=64, rows=4):
    a = inputs.normal_bf16((vocab, rank), 0.05, 130).float().numpy()
    b = inputs.normal_bf16((rank, hidden), 0.05, 131).float().numpy()
    w = inputs.normal_bf16((vocab, hidden), 0.02, 132).float().numpy()
    x = inputs.normal_bf16((rows, hidden), 1.0, 133).float().numpy()
    return a, b, w, x


def test_full_candidate_list_is_exact_argmax():
    a, b, w, x = case()
    res = two_stage(a, b, w, x, cand_k=512)
    exact = np.float32(x.astype(np.float64) @ w.astype(np.float64).T)
    assert np.array_equal(res["ids"], np.argmax(exact, axis=1))   # argmax: first (lowest) id


def test_single_candidate_is_low_rank_argmax():
    a, b, w, x = case()
    res = two_stage(a, b, w, x, cand_k=1)
    _, z = low_rank_logits(a, b, x)
    assert np.array_equal(res["ids"], np.argmax(z, axis=1))


def test_monotone_in_cand_k_and_exact_when_covered():
    a, b, w, x = case()
    exact = np.float32(x.astype(np.float64) @ w.astype(np.float64).T)
    best = np.argmax(exact, axis=1)
    prev = np.full(4, -np.inf)
    for ck in (1, 2, 8, 64, 200, 512):
        res = two_stage(a, b, w, x, cand_k=ck)
        assert np.all(res["vals"] >= prev)
        prev = res["vals"]
        covered = np.array([best[r] in res["cand"][r] for r in range(4)])
        assert np.array_equal(res["ids"][covered], best[covered])


def test_low_rank_h_is_unrounded_fp32():
    a, b, w, x = case()
    h, z = low_rank_logits(a, b, x)
    assert h.dtype == np.float32
    # h is not restricted to bf16 values
    assert np.any(h.view(np.uint32) & 0xFFFF)


def test_rescore_ties_and_bad_ids():
    w = np.zeros((6, 8), np.float32)
    w[2, 0] = 1.0
    w[4, 0] = 1.0
    x = np.ones((1, 8), np.float32)
    e, ids, vals = rescore(w, x, np.array([[4, 2, 9, -1]]))
    assert ids[0] == 2 and vals[0] == 1.0
    assert np.isnan(e[0, 2]) and np.isnan(e[0, 3])
