"""Seeded synthetic tensors with the shapes and distributions of the draft-head workloads.

Recipe: normal draws come from numpy's PCG64 as ``default_rng([config_seed, tensor_id, chunk])`` in
float32, are multiplied by the standard deviation in float32, and are stored as bf16 by torch's
round-to-nearest-even cast. Large matrices are drawn in chunks of 4096 rows (chunk = row // 4096),
in parallel threads, so a 163840 x 4096 head takes seconds. ``config_seed`` is 0 for every workload.

Tensor ids (one per role, so every tensor has its own stream):
  1 head W, 2 activation rows x, 3 planted-tie choice, 4 low-rank A, 5 low-rank B,
  10+3t / 11+3t / 12+3t q, k, v of pass step t, 30 / 31 prefilled K / V rings,
  40 wo, 41 w2, 50+t w2 input of step t, 60 residual, 70 draws, 80+ test-only tensors.
"""
import functools
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

CHUNK_ROWS = 4096


def _chunk(seed, tensor_id, chunk, shape, std):
    rng = np.random.default_rng([seed, tensor_id, chunk])
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def normal_f32(shape, std, tensor_id, seed=0):
    """float32 numpy array of N(0, std^2) draws, chunked over the leading dimension."""
    shape = tuple(int(s) for s in shape)
    rows = shape[0]
    inner = shape[1:]
    nch = max(1, -(-rows // CHUNK_ROWS))
    if nch == 1:
        return _chunk(seed, tensor_id, 0, shape, std)
    out = np.empty(shape, dtype=np.float32)

    def fill(c):
        a, b = c * CHUNK_ROWS, min(rows, (c + 1) * CHUNK_ROWS)
        out[a:b] = _chunk(seed, tensor_id, c, (b - a,) + inner, std)

    with ThreadPoolExecutor(max_workers=16) as ex:
        list(ex.map(fill, range(nch)))
    return out


def normal_bf16(shape, std, tensor_id, seed=0):
    """CPU bf16 tensor of N(0, std^2) draws (torch's RNE cast of the float32 draws)."""
    return torch.from_numpy(normal_f32(shape, std, tensor_id, seed)).to(torch.bfloat16)


def tie_rows(vocab, frac, seed=0, tensor_id=3):
    """(dst, src) row indices for planting exact ties: ``round(frac * vocab)`` destination rows, each
    to be overwritten by a copy of a distinct source row; positions are uniform over the vocabulary
    (so they fall in every part), and no source is also a destination."""
    rng = np.random.default_rng([seed, tensor_id, 0])
    m = int(round(frac * vocab))
    picks = rng.choice(vocab, size=2 * m, replace=False)
    return np.sort(picks[:m]), picks[m:]


def copy_rows(w, dst, src):
    """In-place ``w[dst] = w[src]`` (torch tensor rows)."""
    w[torch.as_tensor(np.asarray(dst), dtype=torch.long)] = w[torch.as_tensor(np.asarray(src),
                                                                              dtype=torch.long)]
    return w


# --- workload builders ------------------------------------------------------------------------

def head(vocab=163840, hidden=4096, std=0.02, tie_frac=0.0, seed=0):
    """Vocabulary head W [vocab][hidden] bf16 (tensor 1), with optional planted duplicate rows.

    The result is cached per process (the full head takes seconds to draw): callers must not modify
    it in place."""
    return _head(vocab, hidden, std, tie_frac, seed)


@functools.lru_cache(maxsize=2)
def _head(vocab, hidden, std, tie_frac, seed):
    w = normal_bf16((vocab, hidden), std, 1, seed)
    ties = None
    if tie_frac > 0:
        ties = tie_rows(vocab, tie_frac, seed)
        copy_rows(w, *ties)
    return w, ties


def rows(r, hidden=4096, seed=0, tensor_id=2):
    """Activation rows x [r][hidden] bf16 ~ N(0, 1)."""
    return normal_bf16((r, hidden), 1.0, tensor_id, seed)


def low_rank(vocab=163840, rank=256, hidden=4096, std=0.05, seed=0):
    """Low-rank factors A [vocab][rank] (tensor 4) and B [rank][hidden] (tensor 5), bf16."""
    return normal_bf16((vocab, rank), std, 4, seed), normal_bf16((rank, hidden), std, 5, seed)


def pass_step_qkv(t, streams=4, heads=32, dim=128, seed=0):
    """q, k, v [streams][heads][dim] bf16 ~ N(0,1) of pass step t."""
    return tuple(normal_bf16((streams, heads, dim), 1.0, 10 + 3 * t + i, seed) for i in range(3))


def rings(streams=4, ring=528, heads=32, dim=128, seed=0):
    """K and V rings [streams][ring][heads][dim] bf16 ~ N(0,1), every slot filled."""
    shape = (streams * ring, heads, dim)
    k = normal_bf16(shape, 1.0, 30, seed).reshape(streams, ring, heads, dim)
    v = normal_bf16(shape, 1.0, 31, seed).reshape(streams, ring, heads, dim)
    return k, v


def linear(out_features, in_features, tensor_id, std=0.02, seed=0):
    """A linear weight [out][in] bf16 ~ N(0, std^2)."""
    return normal_bf16((out_features, in_features), std, tensor_id, seed)


def draws_with_prefix(drafts, seed=0, tensor_id=70):
    """Round draws that agree with ``drafts`` [S][win] on a seeded prefix: per stream a length
    m ~ U{0..win}; draws[i] = drafts[i] for i < m and draws[m] != drafts[m] (when m < win); the rest
    are arbitrary ids. Returns (draws int32 [S][win], m int64 [S])."""
    drafts = np.asarray(drafts, dtype=np.int64)
    S, win = drafts.shape
    rng = np.random.default_rng([seed, tensor_id, 0])
    m = rng.integers(0, win + 1, size=S)
    draws = rng.integers(0, 1 << 17, size=(S, win))
    for s in range(S):
        draws[s, :m[s]] = drafts[s, :m[s]]
        if m[s] < win and draws[s, m[s]] == drafts[s, m[s]]:
            draws[s, m[s]] = drafts[s, m[s]] + 1
    return draws.astype(np.int32), m
