"""Plain CPU oracle of the draft-head decode step.

TEST INFRASTRUCTURE ONLY. This package is the slow, obviously-correct restatement of what the
draft-head step computes, written from the method's description. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference``
arm) may import it. The CUDA library never calls it, and it never calls the CUDA library: the two
share no code. Floating point is carried in float64; the oracle rounds only where the method
rounds (to fp32, bf16 or FP8 E4M3).

Modules (each function cites the passage it follows):

* ``numerics``  - bf16 and FP8 E4M3 rounding and decoding.
* ``quant``     - FP8 quantisation of a bf16 weight: per-row ``s = amax/448`` and E8M0 32x32 blocks.
* ``gemv``      - few-row head GEMV (bf16, FP8 row-scaled, FP8 block-scaled) and its output modes.
* ``topk``      - top-k by (value desc, id asc), split into parts and joined.
* ``two_stage`` - low-rank top-cand_k, exact rescore, argmax.
* ``attn``      - qk_norm + RoPE + ring-window attention for one decode position.
* ``accept``    - accept-prefix count with per-position asked/kept histograms.
* ``draft_pass``- the chained multi-step draft pass (composition of the above).

Every function here is pinned by ``tests/test_oracle_*.py`` against closed forms, brute force,
invariants or library special cases; none is "parity unpinned".
"""
