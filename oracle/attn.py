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
                eps=1e-6, rope_base=10000.0, k_cur=None, terms=None):
    """One decode position per stream.

    Args:
      q, k_new, v_new: [S][heads][dim] bf16 values.
      pos: [S] current positions (>= 0).
      k_ring, v_ring: [S][ring][heads][dim] bf16 values (not modified; updated copies returned).
      window: previous keys attended (0..511), ring >= window + 1.
      k_cur: optional [S][heads][dim] bf16 values taken as the rounded current key instead of
        the oracle's own rounding of it. Where the exact key lies within fp32 error of a bf16
        rounding midpoint both neighbours are correct roundings; a check that has accepted the
        GPU's choice there passes it here, so the output is compared on the same keys.
      terms: optional dict, filled with the values before the output rounding and the magnitudes
        that bound an fp32 computation's rounding error (test tolerances are stated against them):
        ``out_exact`` [S][heads*dim] the attention output before its bf16 rounding;
        ``k_exact`` [S][heads][dim] the current key before its bf16 rounding;
        ``k_pair`` [S][heads][dim] the magnitude of each element's rotation pair of the normalised
        key, sqrt(a_i^2 + a_{i+dim/2}^2) (RoPE preserves it);
        ``abs_out`` [S][heads*dim] sum_j p_j |v_j|;
        ``abs_dev`` [S][heads*dim] sum_j p_j |v_j - out|;
        ``abs_dev_a`` [S][heads*dim] sum_j p_j (A_j + max_i A_i) |v_j - out|, where
        A_j = sum_e m_e |k_j[e]| / sqrt(dim) with m_e the pair magnitude of the normalised query
        (A_j bounds |score_j| and scales its rounding error).
    Returns: (out float64 [S][heads*dim] of bf16 values, k_ring', v_ring').
    """
    q = np.asarray(q, dtype=np.float64)
    S, H, D = q.shape
    half = D // 2
    k_ring = np.array(k_ring, dtype=np.float64, copy=True)
    v_ring = np.array(v_ring, dtype=np.float64, copy=True)
    ring = k_ring.shape[1]
    gq = np.ones(D) if q_gamma is None else np.asarray(q_gamma, dtype=np.float64)
    gk = np.ones(D) if k_gamma is None else np.asarray(k_gamma, dtype=np.float64)
    out = np.empty((S, H * D), dtype=np.float64)
    if terms is not None:
        for name, shape in (("out_exact", (S, H * D)), ("k_exact", (S, H, D)),
                            ("k_pair", (S, H, D)), ("abs_out", (S, H * D)),
                            ("abs_dev", (S, H * D)), ("abs_dev_a", (S, H * D))):
            terms[name] = np.zeros(shape, dtype=np.float64)
    for s in range(S):
        p = int(pos[s])
        slot = p % ring
        for h in range(H):
            qr = rmsnorm(q[s, h], gq, eps)
            qn = rope(qr, p, rope_base)
            kr = rmsnorm(k_new[s][h], gk, eps)
            kx = rope(kr, p, rope_base)
            kn = round_bf16(kx) if k_cur is None else np.asarray(k_cur[s][h], dtype=np.float64)
            k_ring[s, slot, h] = kn
            v_ring[s, slot, h] = np.asarray(v_new[s][h], dtype=np.float64)
            first = max(0, p - window)
            slots = [j % ring for j in range(first, p + 1)]
            keys = k_ring[s, slots, h]
            vals = v_ring[s, slots, h]
            score = keys @ qn / np.sqrt(D)
            wgt = np.exp(score - score.max())
            wgt /= wgt.sum()
            ox = wgt @ vals
            out[s, h * D:(h + 1) * D] = round_bf16(ox)
            if terms is not None:
                sl = slice(h * D, (h + 1) * D)
                terms["out_exact"][s, sl] = ox
                terms["k_exact"][s, h] = kx
                terms["k_pair"][s, h] = np.tile(np.hypot(kr[:half], kr[half:]), 2)
                mq = np.tile(np.hypot(qr[:half], qr[half:]), 2)
                a = np.abs(keys) @ mq / np.sqrt(D)
                dev = np.abs(vals - ox)
                terms["abs_out"][s, sl] = wgt @ np.abs(vals)
                terms["abs_dev"][s, sl] = wgt @ dev
                terms["abs_dev_a"][s, sl] = (wgt * (a + a.max())) @ dev
    return out, k_ring, v_ring
