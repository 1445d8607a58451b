"""Shared helpers of the GPU parity tests: tolerance checks against the oracle.

Tolerances (written here once, used by every parity test):
* fp32 accumulation (GEMV and rescore logits): |gpu - oracle| <= 1e-5 * S, with
  S = sum_k |W x| the magnitude that bounds an fp32 dot product's rounding error.
* bf16 outputs: |gpu - oracle| <= 1e-2 + 2e-3 |oracle|, or the two are one bf16 step apart (the
  output's own rounding can flip when the exact value sits within fp32 error of a bf16 midpoint).
* integer and byte results (FP8 codes and scales, top-k over given logits, accept counts, ids of
  planted exact ties): bit-exact.
* argmax / top-k ids of computed logits: equal wherever the oracle's margin at the k-th place
  exceeds the fp32 tolerance; inside the margin any near-tied id is valid.
"""
import numpy as np
import pytest
import torch

FP32_REL = 1e-5
BF16_ABS, BF16_REL = 1e-2, 2e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def np32(t):
    return t.detach().float().cpu().numpy()


def bf16_step(o):
    a = np.abs(np.asarray(o, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 2.0 ** -126)))
    return np.exp2(np.maximum(e, -126) - 7)


def assert_fp32_close(gpu, oracle, S, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    oracle = np.asarray(oracle, dtype=np.float64)
    d = np.abs(gpu - oracle)
    lim = FP32_REL * np.asarray(S, dtype=np.float64) + 1e-30
    bad = ~(d <= lim)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs off; first at {tuple(i)}: gpu "
                             f"{gpu[tuple(i)]!r} oracle {oracle[tuple(i)]!r} S {S[tuple(i)]!r}")


def assert_bf16_close(gpu, oracle, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    oracle = np.asarray(oracle, dtype=np.float64)
    d = np.abs(gpu - oracle)
    ok = (d <= BF16_ABS + BF16_REL * np.abs(oracle)) | (d <= bf16_step(oracle) * (1 + 1e-9))
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {(~ok).sum()} bf16 outputs off; first at {tuple(i)}: gpu "
                             f"{gpu[tuple(i)]!r} oracle {oracle[tuple(i)]!r}")


def assert_topk_valid(gpu_vals, gpu_ids, oracle_acc, S, k, ids_of=None, what=""):
    """Top-k of computed logits: the ids the GPU picked must be the oracle's up to near-ties at
    the k-th place, and the values must be within the fp32 tolerance of the oracle's."""
    gv = np.asarray(gpu_vals, dtype=np.float64)
    gi = np.asarray(gpu_ids, dtype=np.int64)
    acc = np.asarray(oracle_acc, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    R, n = acc.shape
    local = np.arange(n) if ids_of is None else np.asarray(ids_of, dtype=np.int64)
    pos_of = {int(v): i for i, v in enumerate(local)}
    for r in range(R):
        tol = 2 * FP32_REL * S[r].max()
        order = np.lexsort((local, -acc[r]))
        kth = acc[r][order[k - 1]]
        picked = [pos_of[int(i)] for i in gi[r]]
        assert len(set(picked)) == k, f"{what}: row {r} repeats an id"
        for j, p in enumerate(picked):
            assert acc[r][p] >= kth - tol, f"{what}: row {r} picked id {gi[r][j]} below the k-th"
            assert abs(gv[r][j] - acc[r][p]) <= FP32_REL * S[r][p] + 1e-30, \
                f"{what}: row {r} value of id {gi[r][j]}"
        missing = set(order[:k].tolist()) - set(picked)
        for p in missing:
            assert acc[r][p] <= kth + tol, f"{what}: row {r} missed id {local[p]} above the k-th"


def assert_sorted_keys(vals, ids, what=""):
    """Each row sorted by (value desc, id asc)."""
    vals = np.asarray(vals, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    for r in range(vals.shape[0]):
        v, i = vals[r], ids[r]
        ok = (v[:-1] > v[1:]) | ((v[:-1] == v[1:]) & (i[:-1] < i[1:]))
        assert ok.all(), f"{what}: row {r} not sorted"


def same_bits(a, b):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    b = np.ascontiguousarray(np.asarray(b, dtype=np.float32))
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))
