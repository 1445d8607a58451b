"""Accept-prefix count of a verify round.

Oracle (test infrastructure only; see ``oracle/__init__.py``).

Follows the TFE draft head page (#42), commit "... rnel test TF_DS_ACCEPT_LOG=N": the log reports
"the drafts asked and kept at each window position (a draft is kept when it and every earlier draft
equal the round's draws)".

Readings: only drafts are counted (the verifier's bonus token is not); a stream whose asked count
is outside [0, win] is bad device data: it keeps 0, adds nothing to the histograms and the call
reports the error.
"""
import numpy as np


def accept(drafts, n_asked, draws, asked_hist=None, kept_hist=None):
    """Returns (n_kept int32 [S], asked_hist int64 [win], kept_hist int64 [win], bad: bool).

    The histograms are accumulated onto copies of the given ones (zeros when None).
    """
    drafts = np.asarray(drafts, dtype=np.int64)
    draws = np.asarray(draws, dtype=np.int64)
    S, win = drafts.shape
    ah = np.zeros(win, np.int64) if asked_hist is None else np.array(asked_hist, np.int64)
    kh = np.zeros(win, np.int64) if kept_hist is None else np.array(kept_hist, np.int64)
    n_kept = np.zeros(S, dtype=np.int32)
    bad = False
    for s in range(S):
        na = int(n_asked[s])
        if na < 0 or na > win:
            bad = True
            continue
        kept = 0
        while kept < na and drafts[s, kept] == draws[s, kept]:
            kept += 1
        n_kept[s] = kept
        for i in range(na):
            ah[i] += 1
        for i in range(kept):
            kh[i] += 1
    return n_kept, ah, kh, bad
