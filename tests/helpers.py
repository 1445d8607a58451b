"""Shared helpers of the GPU parity tests: tolerance checks against the oracle.

Tolerances (written here once, used by every parity test):
* fp32 accumulation (GEMV and rescore logits): |gpu - oracle| <= 1e-5 * S, with
  S = sum_k |W x| the magnitude that bounds an fp32 dot product's rounding error.
* bf16 outputs are held to their rounding: the GPU's value must be the round-to-nearest-even bf16
  of some value within ``err`` of the oracle's exact (unrounded) value, i.e. lie in
  [bf16(exact - err), bf16(exact + err)] (rounding is monotone). Away from a bf16 rounding
  midpoint that interval is one value, so the GPU must match the oracle bit for bit; only where the
  exact value sits within ``err`` of a midpoint is the neighbouring bf16 value accepted too. ``err``
  bounds the fp32 computation's error before the output rounding, per operation:
    - GEMV out BF16: 1e-5 S; out ADD_BF16 (bf16(res + acc), one rounding): 1e-5 S plus the fp32
      add, 2^-23 |res + acc|;
    - RMSNorm: 2^-16 |exact| (fp32 sum of squares, square root, two multiplies: about 2^-19 at
      hidden 11008);
    - keys after qk_norm and RoPE (ring writes of the attention, absorbed rows): 2^-18 times the
      element's rotation-pair magnitude (fp32 RMSNorm about 2^-21, the reduced RoPE angle about
      3e-7 rad, fp32 sine, cosine and rotation: about 1.2e-6 in all);
    - attention output: with each key's log-weight known to within
      eta_j = 2^-18 (A_j + max A) + 2^-20 (q' error and the dot product about 2e-6 A_j, the
      max-subtractions 2^-24 of |score| each, exponentials 2^-22), the output is within
      sum_j p_j eta_j |v_j - out| (first order, times 1.01), plus 2^-17 sum_j p_j |v_j| for the
      fp32 sums and the final division;
    - SwiGLU: SiLU(g) within 2^-20 relative (exponential, add, divide, multiply), rounded to bf16,
      times u (exact in fp32), rounded once: every bf16(s u) with s a bf16 rounding of a value in
      that range.
* integer and byte results (FP8 codes and scales, top-k over given logits, accept counts, ids of
  planted exact ties): bit-exact.
* argmax / top-k ids of computed logits: equal wherever the oracle's margin at the k-th place
  exceeds the fp32 tolerance; inside the margin any near-tied id is valid.
"""
import os

import numpy as np
import pytest
import torch

from oracle.numerics import round_bf16

FP32_REL = 1e-5
ADD_REL = 2.0 ** -23
NORM_REL = 2.0 ** -16
KEY_REL = 2.0 ** -18
ATTN_SCORE, ATTN_EXP, ATTN_SUM = 2.0 ** -18, 2.0 ** -20, 2.0 ** -17
SILU_REL = 2.0 ** -20


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def np32(t):
    return t.detach().float().cpu().numpy()


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


def assert_bf16_rounding(gpu, exact, err, what="", rnd=round_bf16):
    """bf16 outputs: gpu == rnd(y) for some y with |y - exact| <= err (see the module docstring).
    ``rnd`` is the rounding the method prescribes (bf16 round-to-nearest-even); a control passes a
    wrong rounding to show that the check tells them apart."""
    gpu = np.asarray(gpu, dtype=np.float64)
    exact = np.asarray(exact, dtype=np.float64)
    err = np.broadcast_to(np.asarray(err, dtype=np.float64), exact.shape)
    lo, hi = rnd(exact - err), rnd(exact + err)
    fin = np.isfinite(exact)
    ok = np.where(fin, (gpu >= lo) & (gpu <= hi), (gpu == exact) | (np.isnan(gpu) & np.isnan(exact)))
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError(f"{what}: {(~ok).sum()} of {ok.size} bf16 outputs off; first at {i}: "
                             f"gpu {gpu[i]!r} exact {exact[i]!r} err {err[i]!r} accepted "
                             f"[{lo[i]!r}, {hi[i]!r}]")


def gemv_bf16_err(S, exact=None):
    """err of a GEMV bf16 output: 1e-5 S, plus the fp32 add of the residual for ADD_BF16 (exact
    = res + acc)."""
    S = np.asarray(S, dtype=np.float64)
    e = FP32_REL * S
    return e if exact is None else e + ADD_REL * np.abs(np.asarray(exact, dtype=np.float64))


def attn_out_err(terms):
    """err of the attention output from the oracle's magnitudes (module docstring)."""
    return 1.01 * (ATTN_SCORE * terms["abs_dev_a"] + ATTN_EXP * terms["abs_dev"]) + \
        ATTN_SUM * terms["abs_out"]


def swiglu_bounds(g, u, rnd=round_bf16):
    """The smallest and largest SwiGLU output an fp32 SiLU within SILU_REL allows (elementwise)."""
    from oracle.layer import silu
    ex = silu(np.asarray(g, dtype=np.float64))
    u = np.asarray(u, dtype=np.float64)
    d = SILU_REL * np.abs(ex)
    a, b = rnd(rnd(ex - d) * u), rnd(rnd(ex + d) * u)
    return np.minimum(a, b), np.maximum(a, b)


def check_window_attn(out, k_ring_gpu, v_ring_gpu, q, k_new, v_new, pos, k_ring, v_ring, window,
                      q_gamma=None, k_gamma=None, eps=1e-6, what="", rnd=round_bf16):
    """Window attention against the oracle: the ring keys written at each stream's current slot
    held to their rounding; every other ring row unchanged, the value rows copied exactly; then
    the output held to its rounding, the oracle attending over the keys the GPU wrote (each one
    just accepted as a correct rounding of the oracle's exact key)."""
    from oracle.attn import window_attn as oracle_attn
    S, H, D = np.asarray(q).shape
    ring = np.asarray(k_ring).shape[1]
    kg, vg = np.asarray(k_ring_gpu, dtype=np.float64), np.asarray(v_ring_gpu, dtype=np.float64)
    terms = {}
    _, okr, ovr = oracle_attn(q, k_new, v_new, pos, k_ring, v_ring, window, q_gamma=q_gamma,
                              k_gamma=k_gamma, eps=eps, terms=terms)
    slots = [int(p) % ring for p in pos]
    cur = np.stack([kg[s, slots[s]] for s in range(S)])
    assert_bf16_rounding(cur, terms["k_exact"], KEY_REL * terms["k_pair"], f"{what} ring keys", rnd)
    other = np.ones(kg.shape[:2], dtype=bool)
    for s in range(S):
        other[s, slots[s]] = False
    assert np.array_equal(kg[other], okr[other]), f"{what}: ring rows other than the current changed"
    assert np.array_equal(vg, ovr), f"{what}: value rows"
    terms = {}
    oracle_attn(q, k_new, v_new, pos, k_ring, v_ring, window, q_gamma=q_gamma, k_gamma=k_gamma,
                eps=eps, k_cur=cur, terms=terms)
    assert_bf16_rounding(out, terms["out_exact"], attn_out_err(terms), f"{what} output", rnd)


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


def oracle_fp8_codes(w, mode, chunk=2048):
    """The oracle's FP8 codes and scales of a large bf16 weight (mode 1 row, 2 block-32), computed
    a chunk of rows at a time on host threads (each chunk is whole 32-row blocks, so the result is
    the oracle's quantisation of the whole matrix)."""
    from concurrent.futures import ThreadPoolExecutor

    from oracle.quant import quant_fp8_block32, quant_fp8_row
    w = np.asarray(w)
    fn = quant_fp8_row if mode == 1 else quant_fp8_block32
    with ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
        parts = list(ex.map(lambda a: fn(w[a:a + chunk]), range(0, w.shape[0], chunk)))
    return (np.concatenate([c for c, _ in parts]), np.concatenate([s for _, s in parts]))


def full_head_oracle(w, x, wfmt=0, scales=None, chunk=16384):
    """Oracle logits and S of a large head, computed a chunk of vocabulary rows at a time (wfmt:
    0 bf16, 1 FP8 row, 2 FP8 block-32 in the plain layout)."""
    from oracle import gemv as og
    n = w.shape[0]
    accs, Ss = [], []
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        if wfmt == og.W_FP8_BLOCK32:
            sc = scales[a // 32:b // 32]
        elif wfmt == og.W_FP8_ROW:
            sc = scales[a:b]
        else:
            sc = None
        wc = w[a:b]
        accs.append(og.gemv_acc(wc, x, wfmt, sc))
        Ss.append(og.gemv_abs_scale(wc, x, wfmt, sc))
    return np.concatenate(accs, axis=1), np.concatenate(Ss, axis=1)


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
