"""qk_norm + RoPE + ring-window attention for one decode position per stream.

Oracle (test infrastructure only; see ``oracle/__init__.py``).

Follows the TFE draft head page (#42): commit "... ocabulary head" (qk_norm is "an RMSNorm on each
query and key head before RoPE"; "the window goes up to 511 (512 keys)"; the head's rows live in a
ring), commit "pass kernels and FP8 linears" (single-query window attention, window 511 in one
block) and the first commits (an absorb never writes more rows than the ring holds).

Readings, where the pages are silent:
* rmsnorm(v) = v / sqrt(mean(v^2) + eps) * gamma over each head's ``dim`` values; eps is an argument
  (1e-6 in the measured workload) and gamma defaults to ones;
* RoPE pairs element i with element i + dim/2 ("half-split") and turns the pair by
  ``p * base^(-2i/dim)`` radians;
* the query stays unrounded; the key is rounded to bf16 when it is written to ring slot
  ``p mod ring``; the value is written as given;
* "window W (W+1 keys)": the keys are positions max(0, p - W) .. p, the current one included;
* every head has its own key/value head (no grouping); scores are scaled by 1/sqrt(dim); the
  softmax subtracts the maximum; the output is rounded to bf16.
"""
import numpy as np

from .numerics import round_bf16


def rmsnorm(v, gamma, eps):
    v = np.asarray(v, dtype=np.float64)
    return v / np.sqrt(np.mean(v * v) + eps) * np.asarray(gamma, dtype=np.float64)


def rope(v, p, base):
    """Half-split rotary embedding of one head vector at position p."""
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    theta = p * np.power(float(base), -2.0 * i / d)
    c, s = np.cos(theta), np.sin(theta)
    a, b = v[:half], v[half:]
    return np.concatenate([a * c - b * s, a * s + b * c])


def window_attn(q, k_new, v_new, pos, k_ring, v_ring, window, q_gamma=None, k_gamma=None,
                eps=1e-6, rope_base=10000.0):
    """One decode position per stream.

    Args:
      q, k_new, v_new: [S][heads][dim] bf16 values.
      pos: [S] current positions (>= 0).
      k_ring, v_ring: [S][ring][heads][dim] bf16 values (not modified; updated copies returned).
      window: previous keys attended (0..511), ring >= window + 1.
    Returns: (out float64 [S][heads*dim] of bf16 values, k_ring', v_ring').
    """
    q = np.asarray(q, dtype=np.float64)
    S, H, D = q.shape
    k_ring = np.array(k_ring, dtype=np.float64, copy=True)
    v_ring = np.array(v_ring, dtype=np.float64, copy=True)
    ring = k_ring.shape[1]
    gq = np.ones(D) if q_gamma is None else np.asarray(q_gamma, dtype=np.float64)
    gk = np.ones(D) if k_gamma is None else np.asarray(k_gamma, dtype=np.float64)
    out = np.empty((S, H * D), dtype=np.float64)
    for s in range(S):
        p = int(pos[s])
        slot = p % ring
        for h in range(H):
            qn = rope(rmsnorm(q[s, h], gq, eps), p, rope_base)
            kn = round_bf16(rope(rmsnorm(k_new[s][h], gk, eps), p, rope_base))
            k_ring[s, slot, h] = kn
            v_ring[s, slot, h] = np.asarray(v_new[s][h], dtype=np.float64)
            first = max(0, p - window)
            slots = [j % ring for j in range(first, p + 1)]
            keys = k_ring[s, slots, h]
            vals = v_ring[s, slots, h]
            score = keys @ qn / np.sqrt(D)
            wgt = np.exp(score - score.max())
            wgt /= wgt.sum()
            out[s, h * D:(h + 1) * D] = round_bf16(wgt @ vals)
    return out, k_ring, v_ring
