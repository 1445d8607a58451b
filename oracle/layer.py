"""The rest of the head layer: RMSNorm of the hidden rows, SwiGLU, and the multi-row ring absorb.

Oracle (test infrastructure only; see ``oracle/__init__.py``).

Follows the TFE draft head page (#42): the description of eagle.cu ("row kernels (RMSNorm, RoPE,
window attention, SwiGLU, top-1 with confidence)"), the commit that splits eagle.zig (the reference
"rounds SiLU(g) to bf16 before the multiply and rounds each residual add once"), commit
"... ocabulary head" (qk_norm before RoPE; a prompt chunk gives the head its last ring of rows) and
the commit on absorbs ("absorb refuses a larger span": never more rows than the ring holds).

Readings, where the pages are silent:
* RMSNorm of a hidden row: x / sqrt(mean(x^2) + eps) * gamma over the row, in exact arithmetic,
  rounded once to bf16;
* SwiGLU: s = bf16(SiLU(g)) with SiLU(g) = g / (1 + exp(-g)), then out = bf16(s * u);
* absorb: rows i = 0 .. n-1 of a span take positions p0 + i; each key row gets the same qk_norm
  and RoPE as the window attention's current key and is rounded to bf16 into ring slot
  (p0 + i) mod ring; each value row is written as given; a span longer than the ring is refused,
  so no two rows of one absorb share a slot.
"""
import numpy as np

from .attn import rmsnorm, rope
from .numerics import round_bf16


def rmsnorm_rows(x, gamma=None, eps=1e-6, exact=False):
    """RMSNorm of every row of x [R][H] (bf16 values); returns bf16 values as float64 [R][H], or
    with exact=True the values before that rounding."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    g = np.ones(x.shape[1]) if gamma is None else np.asarray(gamma, dtype=np.float64)
    ex = np.stack([rmsnorm(row, g, eps) for row in x])
    return ex if exact else round_bf16(ex)


def silu(g):
    """SiLU in float64: g * sigmoid(g), written so that large |g| neither overflows nor loses
    the sign."""
    g = np.asarray(g, dtype=np.float64)
    return np.where(g >= 0, g / (1.0 + np.exp(-np.abs(g))),
                    g * np.exp(-np.abs(g)) / (1.0 + np.exp(-np.abs(g))))


def swiglu(g, u):
    """out = bf16(bf16(SiLU(g)) * u) elementwise (g, u bf16 values)."""
    s = round_bf16(silu(g))
    return round_bf16(s * np.asarray(u, dtype=np.float64))


def absorb(k_rows, v_rows, p0, k_ring, v_ring, k_gamma=None, eps=1e-6, rope_base=10000.0,
           terms=None):
    """Write a span of rows into each stream's ring.

    Args:
      k_rows, v_rows: [S][n][heads][dim] bf16 values.
      p0: [S] position of each stream's first row (>= 0).
      k_ring, v_ring: [S][ring][heads][dim] (not modified; updated copies returned).
      terms: optional dict, filled with ``k_exact`` [S][ring][heads][dim], each written key before
        its bf16 rounding, and ``k_pair``, the magnitude of each element's rotation pair of the
        normalised key (both NaN at slots the absorb does not write).
    Returns (k_ring', v_ring'). Raises ValueError when n > ring.
    """
    k_rows = np.asarray(k_rows, dtype=np.float64)
    S, n, H, D = k_rows.shape
    k_ring = np.array(k_ring, dtype=np.float64, copy=True)
    v_ring = np.array(v_ring, dtype=np.float64, copy=True)
    ring = k_ring.shape[1]
    if n > ring:
        raise ValueError("an absorb may not write more rows than the ring holds")
    gk = np.ones(D) if k_gamma is None else np.asarray(k_gamma, dtype=np.float64)
    if terms is not None:
        terms["k_exact"] = np.full(k_ring.shape, np.nan)
        terms["k_pair"] = np.full(k_ring.shape, np.nan)
    for s in range(S):
        for i in range(n):
            p = int(p0[s]) + i
            slot = p % ring
            for h in range(H):
                kr = rmsnorm(k_rows[s, i, h], gk, eps)
                kx = rope(kr, p, rope_base)
                k_ring[s, slot, h] = round_bf16(kx)
                v_ring[s, slot, h] = np.asarray(v_rows[s][i][h], dtype=np.float64)
                if terms is not None:
                    terms["k_exact"][s, slot, h] = kx
                    terms["k_pair"][s, slot, h] = np.tile(np.hypot(kr[:D // 2], kr[D // 2:]), 2)
    return k_ring, v_ring
