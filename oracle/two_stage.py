"""Two-stage vocabulary head: low-rank logits, top cand_k, exact rescore, argmax.

Oracle (test infrastructure only; see ``oracle/__init__.py``).

Follows the TFE draft head page (#42), commit "... ocabulary head": a two_stage head "takes the top
cand_k low-rank logits (fp32, a tie at the k-th value by the lower token id) and drafts the argmax of
their exact logits from the target's own head, a dense bf16 copy", with cand_k from 1 to 512.

Readings: the low-rank head is ``z = A (B x)`` with A [V][r] and B [r][H] bf16; the intermediate
``h = B x`` is kept in fp32 (not rounded to bf16); ``z`` is fp32; the exact logits ``e_c`` are fp32;
the argmax ranks by (e desc, id asc) like every top-k here. The factors are independent of the exact
head (synthetic tensors).
"""
import numpy as np

from .numerics import fl32
from .topk import canonical, order, topk


def low_rank_logits(a, b, x):
    """(h fp32 [R][r], z fp32 [R][V]) with ``h = fl32(B x)`` and ``z = fl32(A h)``."""
    x64 = np.asarray(x, dtype=np.float64)
    h = fl32(x64 @ np.asarray(b, dtype=np.float64).T)
    z = fl32(h.astype(np.float64) @ np.asarray(a, dtype=np.float64).T)
    return h, z


def rescore(w_exact, x, cand):
    """Exact logits of the candidates and their argmax.

    ``e[r][j] = fl32(W_exact[cand[r][j]] . x[r])``; the draft of row r is the candidate with the
    largest e (ties to the lower id). A candidate id outside [0, vocab) has logit NaN (reading: it
    ranks last and the call reports bad device data).

    Returns (e float32 [R][cand_k], ids int32 [R], vals float32 [R]).
    """
    w = np.asarray(w_exact)
    x64 = np.asarray(x, dtype=np.float64)
    cand = np.asarray(cand, dtype=np.int64)
    R, ck = cand.shape
    e = np.full((R, ck), np.nan, dtype=np.float32)
    for r in range(R):
        ok = (cand[r] >= 0) & (cand[r] < w.shape[0])
        rows = np.asarray(w[cand[r][ok]], dtype=np.float64)
        e[r][ok] = fl32(rows @ x64[r])
    ids = np.empty(R, dtype=np.int32)
    vals = np.empty(R, dtype=np.float32)
    for r in range(R):
        o = order(e[r], cand[r])[0]
        ids[r] = cand[r][o]
        vals[r] = canonical(e[r][o])
    return e, ids, vals


def two_stage(a, b, w_exact, x, cand_k):
    """The whole two-stage head. Returns a dict with h, z, cand (ids), cand_vals, e, ids, vals."""
    h, z = low_rank_logits(a, b, x)
    cand_vals, cand = topk(z, cand_k)
    e, ids, vals = rescore(w_exact, x, cand)
    return dict(h=h, z=z, cand=cand, cand_vals=cand_vals, e=e, ids=ids, vals=vals)
