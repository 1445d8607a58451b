"""The chained draft pass: per step and for every stream at once, window attention, wo, w2, the
vocabulary head and its top-1; after the last step, the accept-prefix count.

Oracle (test infrastructure only; see ``oracle/__init__.py``).

Follows the TFE draft head page (#42): commit "pass kernels and FP8 linears" (a 5-step pass's
attention, wo and w2 few-row GEMVs and top-1 per step, streams as GEMV rows) and the update
"main3x heads, pass kernels, FP8 linears" (wo and w2 through the row-scaled FP8 GEMV, residual adds
rounded once to bf16).

Readings: the measured pass carries one bf16 residual per stream across steps; each step adds
``wo . attn`` and then ``w2 . u_t`` to it (ADD_BF16, in place), where ``u_t`` is the step's given
w2 input (the pages do not put w1/w3 on this path); the head reads the residual and the step's
draft is its top-1 id; step t attends at position ``pos + t``.
"""
import numpy as np

from .accept import accept
from .attn import window_attn
from .gemv import OUT_ADD_BF16, OUT_F32, W_FP8_ROW, gemv
from .topk import topk


def draft_pass(steps, qs, ks, vs, pos0, k_ring, v_ring, window, wo_codes, wo_s, w2_codes, w2_s, us,
               resid0, head_w, head_fmt, head_scales, eps=1e-6, rope_base=10000.0):
    """Returns dict(drafts int32 [S][steps], resid float64 [S][H], k_ring, v_ring, logits list)."""
    resid = np.asarray(resid0, dtype=np.float64).copy()
    S = resid.shape[0]
    drafts = np.zeros((S, steps), dtype=np.int32)
    logits_all = []
    for t in range(steps):
        pos = np.asarray(pos0, dtype=np.int64) + t
        att, k_ring, v_ring = window_attn(qs[t], ks[t], vs[t], pos, k_ring, v_ring, window,
                                          eps=eps, rope_base=rope_base)
        resid = gemv(wo_codes, att, W_FP8_ROW, wo_s, OUT_ADD_BF16, res=resid)
        resid = gemv(w2_codes, us[t], W_FP8_ROW, w2_s, OUT_ADD_BF16, res=resid)
        logits = gemv(head_w, resid, head_fmt, head_scales, OUT_F32)
        logits_all.append(logits)
        _, ids = topk(logits, 1)
        drafts[:, t] = ids[:, 0]
    return dict(drafts=drafts, resid=resid, k_ring=k_ring, v_ring=v_ring, logits=logits_all)


def pass_accept(drafts, n_asked, draws):
    """Accept-prefix count of the pass's drafts against the round's draws."""
    return accept(drafts, n_asked, draws)
