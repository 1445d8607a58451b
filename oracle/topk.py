"""Top-k by (value descending, id ascending), and its split-into-parts-and-join form.

Oracle (test infrastructure only; see ``oracle/__init__.py``).

Follows the TFE draft head page (#42): commit "... ocabulary head" ("the top cand_k low-rank logits
(fp32, a tie at the k-th value by the lower token id)"; "the top-1 kernel through an id map") and
commit "pass kernels and FP8 linears" ("the top-1 of a vocabulary row in 64 parts and a join").

Readings:
* ids compared on ties are the mapped ids when an id map is given;
* -0 and +0 compare equal (a tie, so the lower id goes first);
* NaN ranks below -inf, NaNs among themselves by id;
* returned values are canonical: -0 is returned as +0 and any NaN as the quiet NaN 0x7FC00000.
"""
import numpy as np

CANON_NAN = np.frombuffer(np.uint32(0x7FC00000).tobytes(), dtype=np.float32)[0]


def canonical(v):
    """-0 -> +0 and NaN -> the canonical quiet NaN (float32)."""
    v = np.asarray(v, dtype=np.float32) + np.float32(0.0)       # -0 + 0 = +0
    return np.where(np.isnan(v), CANON_NAN, v).astype(np.float32)


def order(values, ids):
    """Indices of one row sorted by (NaN last, value desc, id asc)."""
    v = np.asarray(values, dtype=np.float64)
    nan = np.isnan(v)
    neg = np.where(nan, 0.0, -v)
    return np.lexsort((np.asarray(ids, dtype=np.int64), neg, nan))


def topk(logits, k, id_map=None):
    """Top-k of each row of ``logits`` [R][n].

    Returns (vals float32 [R][k], ids int32 [R][k]), each row sorted by (value desc, id asc).
    """
    lg = np.atleast_2d(np.asarray(logits, dtype=np.float32))
    R, n = lg.shape
    if not 1 <= k <= n:
        raise ValueError("k must be in 1..n")
    ids_all = np.arange(n, dtype=np.int64) if id_map is None else np.asarray(id_map, dtype=np.int64)
    vals = np.empty((R, k), dtype=np.float32)
    ids = np.empty((R, k), dtype=np.int32)
    for r in range(R):
        o = order(lg[r], ids_all)[:k]
        vals[r] = canonical(lg[r][o])
        ids[r] = ids_all[o]
    return vals, ids


def topk_parts(logits, k, parts, id_map=None):
    """The same top-k computed the split way: each of ``parts`` contiguous ranges of the row keeps
    its own top-min(k, len) and a join takes the top-k of the union. Used to show that the part
    count cannot change the result."""
    lg = np.atleast_2d(np.asarray(logits, dtype=np.float32))
    R, n = lg.shape
    ids_all = np.arange(n, dtype=np.int64) if id_map is None else np.asarray(id_map, dtype=np.int64)
    bounds = [(p * n) // parts for p in range(parts + 1)]
    vals = np.empty((R, k), dtype=np.float32)
    ids = np.empty((R, k), dtype=np.int32)
    for r in range(R):
        cand_v, cand_i = [], []
        for p in range(parts):
            a, b = bounds[p], bounds[p + 1]
            if a == b:
                continue
            o = order(lg[r][a:b], ids_all[a:b])[:k]
            cand_v.append(lg[r][a:b][o])
            cand_i.append(ids_all[a:b][o])
        cv = np.concatenate(cand_v)
        ci = np.concatenate(cand_i)
        o = order(cv, ci)[:k]
        vals[r] = canonical(cv[o])
        ids[r] = ci[o]
    return vals, ids


def top1_confidence(logits):
    """Softmax probability of each row's top-1: ``1 / sum_i exp(l_i - max l)``.

    Follows the TFE draft head page (#42), "What this changes": the row kernels include a "top-1
    with confidence". Reading: the confidence is the softmax probability of the picked logit over
    the whole row; NaN and -inf logits add nothing; a row with no other value gives NaN.
    Computed in float64 from the given logits.
    """
    lg = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    out = np.empty(lg.shape[0], dtype=np.float64)
    for r, row in enumerate(lg):
        fin = row[~np.isnan(row) & (row > -np.inf)]
        out[r] = np.nan if fin.size == 0 else 1.0 / np.sum(np.exp(fin - fin.max()))
    return out
