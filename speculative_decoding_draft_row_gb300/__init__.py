"""GB300-native draft-head decode step: a C-ABI CUDA library (libtfd.so, header include/tfd.h)
and its thin Python binding (``tfd``).

The hot path: few-row vocabulary-head GEMV in bf16 or FP8 (E4M3, per-row or 32x32-block scales)
fused with a split-vocabulary top-1/top-k, the two-stage head (low-rank top-cand_k then exact
rescore), qk_norm + RoPE ring-window attention, and the accept-prefix count.
"""
from . import build  # noqa: F401
