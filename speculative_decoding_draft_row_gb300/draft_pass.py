"""The chained draft pass: per step, for all streams at once (streams are the GEMV rows), window
attention, wo and w2 residual GEMVs (FP8 row-scaled, added to bf16), the vocabulary head with its
fused top-1; after the last step, the accept-prefix count of the drafts against the round's draws.

Follows the TFE draft head page (#42): commit "pass kernels and FP8 linears" (a 5-step pass over 4
streams: attention, wo, w2 and the top-1 per step) and the update "main3x heads, pass kernels, FP8
linears" (wo and w2 in e4m3 with a row scale; a pass's steps captured once as a CUDA graph and
replayed). The steps' inputs (q, k, v, the w2 input, positions) are staged in fixed buffers so the
whole pass can be captured. Every computation is a libtfd call; this module only marshals buffers.
"""
import torch

from . import tfd


class DraftPass:
    def __init__(self, wo_codes, wo_scales, w2_codes, w2_scales, head, head_fmt, head_scales,
                 k_ring, v_ring, window, steps, eps=1e-6, rope_base=10000.0):
        dev = head.device
        self.steps = steps
        self.S, self.ring, self.H, self.D = k_ring.shape
        self.hidden = wo_codes.shape[0]
        self.inner = w2_codes.shape[1]
        self.window, self.eps, self.rope_base = window, eps, rope_base
        self.wo, self.wo_s, self.w2, self.w2_s = wo_codes, wo_scales, w2_codes, w2_scales
        self.head, self.head_fmt, self.head_s = head, head_fmt, head_scales
        self.k_ring, self.v_ring = k_ring, v_ring
        S, H, D = self.S, self.H, self.D
        bf = torch.bfloat16
        self.q = torch.zeros((steps, S, H, D), dtype=bf, device=dev)
        self.k = torch.zeros_like(self.q)
        self.v = torch.zeros_like(self.q)
        self.u = torch.zeros((steps, S, self.inner), dtype=bf, device=dev)
        self.pos = torch.zeros((steps, S), dtype=torch.int32, device=dev)
        self.resid = torch.zeros((S, self.hidden), dtype=bf, device=dev)
        self.attn = torch.zeros((S, H * D), dtype=bf, device=dev)
        self.drafts = torch.zeros((S, steps), dtype=torch.int32, device=dev)
        self.draft_vals = torch.zeros((S, steps), dtype=torch.float32, device=dev)
        self.n_asked = torch.zeros(S, dtype=torch.int32, device=dev)
        self.draws = torch.zeros((S, steps), dtype=torch.int32, device=dev)
        self.n_kept = torch.zeros(S, dtype=torch.int32, device=dev)
        self.asked_hist = torch.zeros(steps, dtype=torch.int64, device=dev)
        self.kept_hist = torch.zeros(steps, dtype=torch.int64, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = tfd.zeroed_workspace(tfd.tfd_head_gemv_workspace(S, head.shape[0], 1), dev)
        self.graph = None

    def load(self, qs, ks, vs, us, pos0, resid, n_asked=None, draws=None):
        """Copy one pass's inputs into the fixed buffers (host or device tensors)."""
        for t in range(self.steps):
            self.q[t].copy_(qs[t], non_blocking=True)
            self.k[t].copy_(ks[t], non_blocking=True)
            self.v[t].copy_(vs[t], non_blocking=True)
            self.u[t].copy_(us[t], non_blocking=True)
        p0 = torch.as_tensor(pos0, dtype=torch.int32)
        self.pos.copy_(torch.stack([p0 + t for t in range(self.steps)]), non_blocking=True)
        self.resid.copy_(resid, non_blocking=True)
        if n_asked is not None:
            self.n_asked.copy_(torch.as_tensor(n_asked, dtype=torch.int32), non_blocking=True)
        if draws is not None:
            self.draws.copy_(torch.as_tensor(draws, dtype=torch.int32), non_blocking=True)

    def step_attn(self, t):
        tfd.tfd_window_attn(self.q[t], self.k[t], self.v[t], self.pos[t], self.k_ring, self.v_ring,
                            self.window, eps=self.eps, rope_base=self.rope_base, out=self.attn,
                            dev_status=self.status)

    def step_wo(self):
        tfd.tfd_head_gemv(self.wo, tfd.W_FP8_ROW, self.wo_s, self.attn, tfd.OUT_ADD_BF16,
                          y=self.resid)

    def step_w2(self, t):
        tfd.tfd_head_gemv(self.w2, tfd.W_FP8_ROW, self.w2_s, self.u[t], tfd.OUT_ADD_BF16,
                          y=self.resid)

    def step_head(self, t):
        tfd.tfd_head_gemv(self.head, self.head_fmt, self.head_s, self.resid, tfd.OUT_NONE, topk=1,
                          top_vals=self.draft_vals[:, t:t + 1], top_ids=self.drafts[:, t:t + 1],
                          ws=self.ws)

    def enqueue_step(self, t):
        self.step_attn(t)
        self.step_wo()
        self.step_w2(t)
        self.step_head(t)

    def enqueue_accept(self):
        tfd.tfd_accept(self.drafts, self.n_asked, self.draws, n_kept=self.n_kept,
                       asked_hist=self.asked_hist, kept_hist=self.kept_hist,
                       dev_status=self.status)

    def enqueue(self):
        for t in range(self.steps):
            self.enqueue_step(t)
        self.enqueue_accept()

    def launches(self):
        """Kernels one pass launches: 4 per step (attention, wo, w2, head) and the accept."""
        return 4 * self.steps + 1

    def capture(self):
        """Capture one whole pass as a CUDA graph (replayed by run())."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.enqueue()                          # warm: builds and loads the library
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.enqueue()
        return self.graph

    def run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.enqueue()
