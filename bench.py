"""Benchmark of the draft-head decode step on GB300.

Workload (one step): the full-vocabulary bf16 head W [163840 x 4096] (1.34 GB, larger than L2, so
no flush is needed) against 1, 5, 10 and 15 activation rows, each call writing fp32 logits and the
fused top-1 over vocabulary parts plus a join; 1% of the head's rows are planted exact copies.
The metric is achieved HBM GB/s (algorithmic bytes / time) and us per call, timed as CUDA-graph
replays of the step (eager per-call times are reported beside them); the FP8 head
(E4M3 + E8M0 32x32 blocks, and per-row scales) with fused top-64 is reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (the plain fp64 restatement in oracle/) on a bounded
sample of the same workload. Under torchrun every rank runs its own replica (weak scaling); rank 0
prints one JSON line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

VOCAB, HIDDEN = 163840, 4096
ROWS = (1, 5, 10, 15)          # the headline step (the metric's row counts)
ROWS_SWEEP = (1, 5, 10, 15, 16)  # per-row and FP8 figures: 16 rows is the heaviest case
L2_BYTES = 129 * 1000 * 1000
ROTATE_BYTES = 2 * L2_BYTES + 1  # rotated working sets must exceed twice the L2
ROWS_WINDOW = (17, 24, 32)       # decode windows past 16 rows (bf16 head + top-1)
METRIC = "head GEMV+top-k achieved HBM GB/s (% of peak) and us/call at 1/5/10/15 rows"
WORKLOAD = ("full-vocab bf16 head 163840x4096, rows 1/5/10/15, fp32 logits + fused top-1 over "
            "vocabulary parts and a join, 1% planted exact-tie rows")


def bench_config(world):
    """The workload's description, the same on both arms of the bench."""
    return {"workload": WORKLOAD, "vocab": VOCAB, "hidden": HIDDEN, "rows": list(ROWS),
            "rows_sweep": list(ROWS_SWEEP), "rows_window": list(ROWS_WINDOW),
            "l2": "head weights 1.34 GB (FP8 0.67 GB) exceed the 129 MB L2, no flush needed; "
                  "rows_of_path working sets under twice the L2 are rotated over copies whose "
                  "total exceeds it",
            "timing": "value: each step (the four calls at rows 1/5/10/15) replayed from one CUDA "
                      "graph; per_rows (1/5/10/15/16), per_rows_window (17-32 rows) and "
                      "fp8_top64 from graphs of 10 calls, us_eager from single eager launches",
            "parallelism": f"replicas x{world}"}


def bf16_call_bytes(rows):
    """Algorithmic bytes of one bf16 call: weights once, activations, fp32 logits, top-1."""
    return VOCAB * HIDDEN * 2 + rows * HIDDEN * 2 + rows * VOCAB * 4 + rows * 8


def fp8_call_bytes(rows, k=64):
    """FP8 call without logits: codes, scales (655,360 B either form), activations, top-k."""
    return VOCAB * HIDDEN + 655360 + rows * HIDDEN * 2 + rows * k * 8


def profiled_traffic():
    """DRAM bytes per launch of the headline kernel from the committed ncu summary, or None when
    the kernel's sources have changed since that capture."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
        for path, digest in rec["sources_sha256"].items():
            if hashlib.sha256(open(os.path.join(ROOT, path), "rb").read()).hexdigest() != digest:
                return None
        return rec["traffic_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        return None


# ---------------------------------------------------------------------------------------------
# CPU oracle timing (the reported baseline and the reference arm)
# ---------------------------------------------------------------------------------------------
SAMPLE_ROWS = 16384  # vocabulary rows of the oracle's sample (1/10 of the head)


def oracle_sample_worker(seconds):
    """Times the oracle (as it stands) on a slice of the workload; prints one JSON line."""
    import numpy as np

    from oracle import gemv as og
    from oracle.topk import topk
    from synth import inputs

    w = inputs.normal_bf16((SAMPLE_ROWS, HIDDEN), 0.02, 1).float().numpy()
    x = inputs.rows(16).float().numpy()
    t0 = time.perf_counter()
    nbytes = 0
    calls = 0
    while True:
        for r in ROWS:
            y = og.gemv(w, x[:r], og.W_BF16, None, og.OUT_F32)
            topk(y, 1)
            nbytes += SAMPLE_ROWS * HIDDEN * 2 + r * HIDDEN * 2 + r * SAMPLE_ROWS * 4 + r * 8
            calls += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    print(json.dumps({"gbs": nbytes / dt / 1e9, "seconds": dt, "calls": calls,
                      "threads": int(os.environ.get("OPENBLAS_NUM_THREADS", "0") or 0)}))


def cpu_model():
    """The host CPU's model name from lscpu (None if lscpu is missing)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
    except OSError:
        return None
    for line in out.splitlines():
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    return None


def run_oracle_sample(seconds, threads=None):
    """The oracle sample in a fresh process with BLAS limited to ``threads`` (all host cores by
    default): numpy's matrix product splits the vocabulary rows over the threads."""
    threads = threads or os.cpu_count() or 1
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(threads), OMP_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads))
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-worker",
                          str(seconds)], capture_output=True, text=True, env=env, cwd=ROOT)
    if out.returncode != 0:
        raise RuntimeError("oracle timing failed: " + out.stderr[-2000:])
    res = json.loads(out.stdout.strip().splitlines()[-1])
    res["threads"] = threads
    return res


def cpu_baseline(seconds=12.0):
    """The oracle timed on the host: all cores (the reported value) and one thread."""
    r = run_oracle_sample(seconds)
    r1 = run_oracle_sample(seconds / 2, threads=1)
    return {"value": round(r["gbs"], 4), "unit": "GB/s", "cores": r["threads"], "kind": "oracle",
            "single_thread": {"value": round(r1["gbs"], 4), "unit": "GB/s", "cores": 1,
                              "seconds": round(r1["seconds"], 1), "calls": r1["calls"]},
            "nproc": os.cpu_count(), "cpu_model": cpu_model(),
            "sample": f"oracle fp64 GEMV + top-1 on {SAMPLE_ROWS} of the {VOCAB} vocabulary rows "
                      f"at rows 1/5/10/15, repeated for {r['seconds']:.1f} s ({r['calls']} calls) "
                      f"with BLAS over all {r['threads']} host threads; single_thread: the same "
                      f"with one thread"}


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"tfd_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------
def dist_setup(gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The largest of the ranks' values (every rank gets it)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_throughput(bytes_per_rank_step, ms_per_step_max, world):
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time."""
    return bytes_per_rank_step * world / (ms_per_step_max * 1e-3) / 1e9


def _rotating(fn):
    """A list of calls to cycle through: fn itself, or fn's copies when it is a list (each copy
    on its own buffers, so a working set smaller than L2 is read from HBM)."""
    return list(fn) if isinstance(fn, (list, tuple)) else [fn]


def time_calls(fn, iters, stream):
    """Mean device time of one call in ms over iters calls, cycling through fn's copies (CUDA
    events on the launching stream)."""
    import torch
    fns = _rotating(fn)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for i in range(iters):
        fns[i % len(fns)]()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / iters


def time_graph(fn, iters, per_graph=10):
    """Mean device time of one call in ms with the host out of the way: per_graph calls (at least
    one round of fn's copies) captured in one CUDA graph, replayed until about iters calls ran
    (CUDA events on the replaying stream)."""
    import torch
    fns = _rotating(fn)
    per_graph = max(per_graph, len(fns))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for f in fns:
            f()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(per_graph):
            fns[i % len(fns)]()
    reps = max(1, iters // per_graph)
    for _ in range(2):
        g.replay()
    stream = torch.cuda.current_stream()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / (reps * per_graph)


def copies_for(nbytes):
    """How many copies of an nbytes working set make the rotated set exceed twice the L2."""
    return max(1, -(-ROTATE_BYTES // max(1, nbytes)))


def run_ours(args):
    import torch

    from speculative_decoding_draft_row_gb300 import tfd
    from synth import inputs

    rank, world, local = dist_setup(args.gpus)
    stream = torch.cuda.current_stream()
    w, _ = inputs.head(tie_frac=0.01, seed=rank)
    wd = w.cuda()
    del w
    x_host = inputs.rows(32, seed=rank).pin_memory()
    all_rows = ROWS_SWEEP + ROWS_WINDOW
    xs = {r: x_host[:r].cuda() for r in all_rows}
    ys = {r: torch.empty((r, VOCAB), dtype=torch.float32, device="cuda") for r in all_rows}
    tv = {r: torch.empty((r, 1), dtype=torch.float32, device="cuda") for r in all_rows}
    ti = {r: torch.empty((r, 1), dtype=torch.int32, device="cuda") for r in all_rows}
    ws = tfd.zeroed_workspace(tfd.tfd_head_gemv_workspace(32, VOCAB, 1))

    def call(r, x=None):
        tfd.tfd_head_gemv(wd, tfd.W_BF16, None, xs[r] if x is None else x, tfd.OUT_F32, y=ys[r],
                          topk=1, top_vals=tv[r], top_ids=ti[r], ws=ws)

    def step():
        for r in ROWS:
            call(r)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # one step (the four calls) captured as a CUDA graph, as a decode loop replays it
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph):
        step()
    for _ in range(3):
        step_graph.replay()
    torch.cuda.synchronize()
    # ---- timed region: K steps (graph replays), one event pair per step ----
    n = args.steps * len(ROWS)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        evs[0].record(stream)
        for i in range(args.steps):
            step_graph.replay()
            evs[i + 1].record(stream)
        evs[-1].synchronize()
    torch.cuda.synchronize()
    barrier(world)
    total_ms = evs[0].elapsed_time(evs[-1])
    step_bytes = sum(bf16_call_bytes(r) for r in ROWS)
    ms_step = max_over_ranks(total_ms / args.steps, world)
    value = job_throughput(step_bytes, ms_step, world)

    # eager per-call device times (each call launched on its own, an event pair around it)
    eager_reps = 5
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(eager_reps * len(all_rows) + 1)]
    evs[0].record(stream)
    i = 0
    for _ in range(eager_reps):
        for r in all_rows:
            call(r)
            i += 1
            evs[i].record(stream)
    evs[-1].synchronize()
    eager_us = {r: [] for r in all_rows}
    i = 0
    for _ in range(eager_reps):
        for r in all_rows:
            eager_us[r].append(evs[i].elapsed_time(evs[i + 1]) * 1e3)
            i += 1
    # per-call device times with the calls replayed from a CUDA graph (10 calls per graph)
    graph_us = {r: time_graph(lambda r=r: call(r), 100) * 1e3 for r in all_rows}
    pk = peaks()
    peak = pk["hbm_gbs"] if pk else 6800.0
    per_rows, per_rows_window = {}, {}
    for r in all_rows:
        us = graph_us[r]
        gbs = bf16_call_bytes(r) / (us * 1e-6) / 1e9
        (per_rows if r <= 16 else per_rows_window)[str(r)] = {
            "us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
            "us_eager": round(statistics.median(eager_us[r]), 2)}
    # the four launches of a step back to back: bytes per launch over the mean launch duration
    achieved = step_bytes / (total_ms / args.steps * 1e-3) / 1e9

    if args.no_extras:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": round(value, 2), "unit": "GB/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": round(ms_step, 4), "per_rows": per_rows,
                              "partial": "headline calls only (--no-extras)"}), flush=True)
        return
    # ---- e2e: the same calls through the public API with host buffers ----
    top_host = {r: torch.empty((r, 1), dtype=torch.int32).pin_memory() for r in ROWS}
    val_host = {r: torch.empty((r, 1), dtype=torch.float32).pin_memory() for r in ROWS}
    xdev = {r: torch.empty((r, HIDDEN), dtype=torch.bfloat16, device="cuda") for r in ROWS}

    def e2e_step():
        for r in ROWS:
            xdev[r].copy_(x_host[:r], non_blocking=True)
            call(r, xdev[r])
            top_host[r].copy_(ti[r], non_blocking=True)
            val_host[r].copy_(tv[r], non_blocking=True)

    e2e_steps = max(10, args.steps // 4)
    for _ in range(3):
        e2e_step()
    barrier(world)
    e2e_ms = max_over_ranks(time_calls(e2e_step, e2e_steps, stream), world)
    h2d = sum(r * HIDDEN * 2 for r in ROWS)
    d2h = sum(r * 8 for r in ROWS)

    # ---- FP8 head, fused top-64 (reported beside the headline) ----
    fp8 = {}
    for mode, name, aq in ((tfd.W_FP8_BLOCK32, "e4m3_e8m0_32x32", False),
                           (tfd.W_FP8_BLOCK32_IL, "e4m3_e8m0_32x32_interleaved", False),
                           (tfd.W_FP8_ROW, "e4m3_row", False),
                           (tfd.W_FP8_BLOCK32_IL, "e4m3_e8m0_32x32_interleaved_w8a8", True),
                           (tfd.W_FP8_ROW, "e4m3_row_w8a8", True)):
        codes, scales = tfd.tfd_quant_fp8(wd, mode)
        ws64 = tfd.zeroed_workspace(tfd.tfd_head_gemv_workspace(16, VOCAB, 64))
        out = {}
        for r in ROWS_SWEEP:
            v64 = torch.empty((r, 64), dtype=torch.float32, device="cuda")
            i64 = torch.empty((r, 64), dtype=torch.int32, device="cuda")
            f = lambda: tfd.tfd_head_gemv(codes, mode, scales, xs[r], tfd.OUT_NONE, topk=64,
                                          top_vals=v64, top_ids=i64, ws=ws64, act_e4m3=aq)
            for _ in range(3):
                f()
            ms = time_graph(f, 20)
            gbs = fp8_call_bytes(r) / (ms * 1e-3) / 1e9
            out[str(r)] = {"us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                           "frac": round(gbs / peak, 4)}
        fp8[name] = out
        del codes, scales

    draft_pass = measure_pass(wd, stream)
    path_rows = measure_rows_of_path(wd, stream, peak)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) head, N(0,1) rows)",
        "config": bench_config(world),
        "per_rows": per_rows,
        "per_rows_window": per_rows_window,
        "fp8_top64": fp8,
        "pass_5x4": draft_pass,
        "rows_of_path": path_rows,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(),
                     "algorithmic_bytes_per_launch": round(step_bytes / len(ROWS)),
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured)" if pk else "fallback"},
        "e2e": {"value": round(step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": n,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)


PASS_STEPS, PASS_STREAMS, PASS_HEADS, PASS_DIM, PASS_RING, PASS_WINDOW = 5, 4, 32, 128, 528, 511
HIDDEN_FFN = 11008


def pass_bytes(head_bytes):
    """Algorithmic bytes of one 5-step pass: per step the head, wo and w2 (FP8 codes + row scales)
    and the window's K and V rows of every stream and head."""
    wo = HIDDEN * HIDDEN + HIDDEN * 4
    w2 = HIDDEN * HIDDEN_FFN + HIDDEN * 4
    kv = PASS_STREAMS * PASS_HEADS * (PASS_WINDOW + 1) * PASS_DIM * 2 * 2
    return PASS_STEPS * (head_bytes + wo + w2 + kv)


def measure_pass(wd, stream, reps=20):
    """The 5-step x 4-stream draft pass, captured as one CUDA graph; returns ms per pass for the
    bf16 head and for the FP8 (32x32 block) head."""
    import torch

    from speculative_decoding_draft_row_gb300 import tfd
    from speculative_decoding_draft_row_gb300.draft_pass import DraftPass
    from synth import inputs

    wo_c, wo_s = tfd.tfd_quant_fp8(inputs.linear(HIDDEN, HIDDEN, 40).cuda(), tfd.W_FP8_ROW)
    w2_c, w2_s = tfd.tfd_quant_fp8(inputs.linear(HIDDEN, HIDDEN_FFN, 41).cuda(), tfd.W_FP8_ROW)
    kr, vr = inputs.rings(PASS_STREAMS, PASS_RING, PASS_HEADS, PASS_DIM)
    qkv = [inputs.pass_step_qkv(t, PASS_STREAMS, PASS_HEADS, PASS_DIM) for t in range(PASS_STEPS)]
    us = [inputs.normal_bf16((PASS_STREAMS, HIDDEN_FFN), 1.0, 50 + t) for t in range(PASS_STEPS)]
    resid = inputs.normal_bf16((PASS_STREAMS, HIDDEN), 1.0, 60)
    hc, hs = tfd.tfd_quant_fp8(wd, tfd.W_FP8_BLOCK32)
    hci = tfd.tfd_fp8_block32_relayout(hc, True)
    out = {}
    for name, head, fmt, sc in (("bf16_head", wd, tfd.W_BF16, None),
                                ("fp8_block32_head", hc, tfd.W_FP8_BLOCK32, hs),
                                ("fp8_block32_interleaved_head", hci, tfd.W_FP8_BLOCK32_IL, hs)):
        dp = DraftPass(wo_c, wo_s, w2_c, w2_s, head, fmt, sc, kr.clone().cuda(), vr.clone().cuda(),
                       PASS_WINDOW, PASS_STEPS)
        dp.load([q for q, _, _ in qkv], [k for _, k, _ in qkv], [v for _, _, v in qkv], us,
                [511, 511, 511, 511], resid.cuda(), [5] * PASS_STREAMS,
                torch.zeros((PASS_STREAMS, PASS_STEPS), dtype=torch.int32))
        dp.capture()
        for _ in range(3):
            dp.run()
        ms = time_calls(dp.run, reps, stream)
        ms_eager = time_calls(dp.enqueue, reps, stream)
        nb = pass_bytes(head.numel() * head.element_size() + (655360 if sc is not None else 0))
        out[name] = {"ms_graph": round(ms, 4), "ms_eager": round(ms_eager, 4),
                     "gbs": round(nb / (ms * 1e-3) / 1e9, 1), "bytes": nb,
                     "launches": dp.launches()}
    return out


def measure_rows_of_path(wd, stream, peak):
    """The other rows of the step, each timed alone (CUDA-graph replays, mean over repetitions)
    and reported as us per call and algorithmic GB/s against the HBM peak. A row whose working
    set is under twice the L2 cycles through copies (new inputs each call) whose total exceeds it,
    so its bytes come from HBM."""
    import numpy as np
    import torch

    from speculative_decoding_draft_row_gb300 import tfd
    from synth import inputs

    out = {}

    def rec(name, fn, nbytes, reps=20, working_set=None):
        # device time from graph replays; eager calls add the host's launch overhead
        fns = _rotating(fn)
        for f in fns * 2:
            f()
        ms_eager = time_calls(fns, max(reps, len(fns)), stream)
        ms = time_graph(fns, max(reps, 2 * len(fns)))
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 2), "us_eager": round(ms_eager * 1e3, 2),
                     "gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "bytes": nbytes}
        if len(fns) > 1:
            out[name]["rotated"] = {"copies": len(fns), "bytes": len(fns) * working_set}

    # two-stage head, 16 rows: B x, A h, top cand_k of the low-rank logits, exact rescore. Each
    # copy has its own factors (A + B = 86 MB) and activation rows, so its candidates, and the
    # exact-head rows the rescore gathers, differ from the other copies'.
    lr_bytes = 256 * HIDDEN * 2 + VOCAB * 256 * 2
    ncp = copies_for(lr_bytes)
    lr = []
    for c in range(ncp):
        a, b = inputs.low_rank(seed=c)
        lr.append((a.cuda(), b.cuda(), inputs.rows(16, seed=c, tensor_id=92).cuda()))
        del a, b
    h = torch.empty((16, 256), dtype=torch.float32, device="cuda")
    z = torch.empty((16, VOCAB), dtype=torch.float32, device="cuda")
    for ck in (1, 64, 512):
        cv = torch.empty((16, ck), dtype=torch.float32, device="cuda")
        ci = torch.empty((16, ck), dtype=torch.int32, device="cuda")
        tws = tfd.zeroed_workspace(tfd.tfd_head_gemv_workspace(16, VOCAB, ck, 0))
        rws = tfd.zeroed_workspace(tfd.tfd_rescore_workspace(16, ck))
        oi = torch.empty(16, dtype=torch.int32, device="cuda")
        ov = torch.empty(16, dtype=torch.float32, device="cuda")

        def two_stage(ad, bd, x16):
            tfd.tfd_head_gemv(bd, tfd.W_BF16, None, x16, tfd.OUT_F32, y=h)
            tfd.tfd_head_gemv(ad, tfd.W_BF16, None, h, tfd.OUT_F32, y=z, topk=ck, top_vals=cv,
                              top_ids=ci, ws=tws)
            tfd.tfd_rescore(wd, x16, ci, out_ids=oi, out_vals=ov, ws=rws, want_logits=False)

        # what the method must move: B, A, the activations and the gathered exact-head rows
        nbytes = lr_bytes + 16 * HIDDEN * 2 + 16 * ck * HIDDEN * 2
        rec(f"two_stage_cand{ck}", [lambda c=c: two_stage(*lr[c]) for c in range(ncp)], nbytes,
            working_set=nbytes)
    del lr
    # rescore alone: 16 rows x 512 candidate rows of the exact head, new candidates each copy
    rng = np.random.default_rng([0, 91, 0])
    nb_rs = 16 * 512 * HIDDEN * 2 + 16 * HIDDEN * 2 + 16 * 512 * 4
    ncp = copies_for(nb_rs)
    cands = [torch.from_numpy(rng.integers(0, VOCAB, size=(16, 512)).astype(np.int32)).cuda()
             for _ in range(ncp)]
    x16 = inputs.rows(16).cuda()
    rws = tfd.zeroed_workspace(tfd.tfd_rescore_workspace(16, 512))
    oi = torch.empty(16, dtype=torch.int32, device="cuda")
    ov = torch.empty(16, dtype=torch.float32, device="cuda")
    rec("rescore_16x512", [lambda c=c: tfd.tfd_rescore(wd, x16, cands[c], out_ids=oi, out_vals=ov,
                                                       ws=rws, want_logits=False)
                           for c in range(ncp)], nb_rs, working_set=nb_rs)
    del cands
    # standalone top-k of 16 x 163840 fp32 logits (10.5 MB a copy)
    lg_bytes = 16 * VOCAB * 4
    ncp = copies_for(lg_bytes)
    logits = [torch.from_numpy(inputs.normal_f32((16, VOCAB), 1.0, 90, seed=c)).cuda()
              for c in range(ncp)]
    for kk in (64, 512):
        tws = tfd.zeroed_workspace(tfd.tfd_topk_workspace(16, VOCAB, kk))
        cv = torch.empty((16, kk), dtype=torch.float32, device="cuda")
        ci = torch.empty((16, kk), dtype=torch.int32, device="cuda")
        rec(f"topk_16x163840_k{kk}",
            [lambda c=c: tfd.tfd_topk(logits[c], kk, vals=cv, ids=ci, ws=tws) for c in range(ncp)],
            lg_bytes + 16 * kk * 8, working_set=lg_bytes)
    del logits
    # window attention of one pass step: 4 streams x 32 heads, window 511 (512 keys); each copy
    # its own K/V rings (34.6 MB)
    ring_bytes = 2 * PASS_STREAMS * PASS_RING * PASS_HEADS * PASS_DIM * 2
    ncp = copies_for(ring_bytes)
    kr, vr = inputs.rings(PASS_STREAMS, PASS_RING, PASS_HEADS, PASS_DIM)
    rings = [(kr.cuda(), vr.cuda()) for _ in range(ncp)]
    del kr, vr
    q, k, v = (t.cuda() for t in inputs.pass_step_qkv(0))
    pos = torch.full((PASS_STREAMS,), 511, dtype=torch.int32, device="cuda")
    att = torch.empty((PASS_STREAMS, PASS_HEADS * PASS_DIM), dtype=torch.bfloat16, device="cuda")
    rec("window_attn_4x32_w511",
        [lambda c=c: tfd.tfd_window_attn(q, k, v, pos, rings[c][0], rings[c][1], PASS_WINDOW,
                                         out=att) for c in range(ncp)],
        PASS_STREAMS * PASS_HEADS * (PASS_WINDOW + 1) * PASS_DIM * 2 * 2, working_set=ring_bytes)
    krd, vrd = rings[0]
    # the rest of the head layer: RMSNorm of the hidden rows, SwiGLU, a 128-row prompt-chunk absorb
    hid = torch.from_numpy(inputs.normal_f32((PASS_STREAMS, HIDDEN), 1.0, 61)).to(torch.bfloat16).cuda()
    hout = torch.empty_like(hid)
    gam = torch.ones(HIDDEN, dtype=torch.bfloat16, device="cuda")
    rec("rmsnorm_4x4096", lambda: tfd.tfd_rmsnorm(hid, gam, 1e-6, out=hout),
        PASS_STREAMS * HIDDEN * 2 * 2 + HIDDEN * 2)
    gg = torch.from_numpy(inputs.normal_f32((PASS_STREAMS, HIDDEN_FFN), 1.0, 62)).to(torch.bfloat16).cuda()
    uu = torch.from_numpy(inputs.normal_f32((PASS_STREAMS, HIDDEN_FFN), 1.0, 63)).to(torch.bfloat16).cuda()
    so = torch.empty_like(gg)
    rec("swiglu_4x11008", lambda: tfd.tfd_swiglu(gg, uu, out=so), PASS_STREAMS * HIDDEN_FFN * 2 * 3)
    nab = 128
    kab = torch.from_numpy(inputs.normal_f32((PASS_STREAMS * nab * PASS_HEADS, PASS_DIM), 1.0, 64)).to(
        torch.bfloat16).cuda().reshape(PASS_STREAMS, nab, PASS_HEADS, PASS_DIM)
    vab = torch.from_numpy(inputs.normal_f32((PASS_STREAMS * nab * PASS_HEADS, PASS_DIM), 1.0, 65)).to(
        torch.bfloat16).cuda().reshape(PASS_STREAMS, nab, PASS_HEADS, PASS_DIM)
    p0 = torch.zeros(PASS_STREAMS, dtype=torch.int32, device="cuda")
    rec("absorb_4x128rows",
        [lambda c=c: tfd.tfd_absorb(kab, vab, p0, rings[c][0], rings[c][1]) for c in range(ncp)],
        PASS_STREAMS * nab * PASS_HEADS * PASS_DIM * 2 * 4, working_set=ring_bytes)
    # accept of a 5-draft window over 4 streams
    dr = torch.arange(20, dtype=torch.int32, device="cuda").reshape(4, 5)
    na = torch.full((4,), 5, dtype=torch.int32, device="cuda")
    nk = torch.empty(4, dtype=torch.int32, device="cuda")
    rec("accept_4x5", lambda: tfd.tfd_accept(dr, na, dr, n_kept=nk), 4 * 5 * 4 * 2 + 4 * 8)
    # FP8 quantisation of the head (offline step): bf16 in, codes + scales out
    for mode, name in ((tfd.W_FP8_ROW, "quant_row_head"), (tfd.W_FP8_BLOCK32, "quant_block32_head")):
        codes = torch.empty((VOCAB, HIDDEN), dtype=torch.uint8, device="cuda")
        sc = (torch.empty(VOCAB, dtype=torch.float32, device="cuda") if mode == tfd.W_FP8_ROW
              else torch.empty((VOCAB // 32, HIDDEN // 32), dtype=torch.uint8, device="cuda"))
        rec(name, lambda: tfd.tfd_quant_fp8(wd, mode, codes=codes, scales=sc),
            VOCAB * HIDDEN * 3 + sc.numel() * sc.element_size(), reps=5)
        del codes, sc
    return out


def run_head_case(args):
    """A small case for profiling: the head in one format (--head bf16|row|block32|block32il; the
    FP8 forms by default with fused top-64 and no logits, bf16 with fp32 logits and top-1, as the
    headline) at rows 1/5/10/15/16 or --rows, warmup + steps calls of each (the steps from CUDA
    graph replays), one JSON line of us per call."""
    import torch

    from speculative_decoding_draft_row_gb300 import tfd
    from synth import inputs

    torch.cuda.set_device(0)
    fmt = args.head or args.fp8
    mode = {"bf16": tfd.W_BF16, "row": tfd.W_FP8_ROW, "block32": tfd.W_FP8_BLOCK32,
            "block32il": tfd.W_FP8_BLOCK32_IL}[fmt]
    topk = args.topk if args.topk is not None else (1 if mode == tfd.W_BF16 else 64)
    out_mode = tfd.OUT_F32 if mode == tfd.W_BF16 else tfd.OUT_NONE
    if args.shape:  # another matrix than the head: N x K ~ N(0, 0.02)
        n_out, k_in = (int(v) for v in args.shape.split(":"))
        w = inputs.linear(n_out, k_in, 40)
    else:
        w, _ = inputs.head(tie_frac=0.01)
    n_out, k_in = w.shape
    if mode == tfd.W_BF16:
        codes, scales = w.cuda(), None
    else:
        codes, scales = tfd.tfd_quant_fp8(w.cuda(), mode)
    del w
    row_counts = (ROWS_SWEEP if args.rows is None
                  else [1, 4, 8, 9, 12, 16] if args.rows == 0 else [args.rows])
    xs = {r: inputs.rows(32, hidden=k_in)[:r].cuda() for r in row_counts}
    ws = tfd.zeroed_workspace(tfd.tfd_head_gemv_workspace(32, n_out, max(topk, 1)))
    out = {}
    for r in row_counts:
        y = torch.empty((r, n_out), dtype=torch.float32, device="cuda") if out_mode else None
        v = torch.empty((r, max(topk, 1)), dtype=torch.float32, device="cuda")
        i = torch.empty((r, max(topk, 1)), dtype=torch.int32, device="cuda")
        f = lambda: tfd.tfd_head_gemv(codes, mode, scales, xs[r], out_mode, y=y, topk=topk,
                                      top_vals=v if topk else None, top_ids=i if topk else None,
                                      ws=ws, act_e4m3=args.w8a8)
        for _ in range(args.warmup):
            f()
        ms = time_graph(f, args.steps)
        nb = (bf16_call_bytes(r) if mode == tfd.W_BF16 else fp8_call_bytes(r, max(topk, 1)))
        if args.shape:
            nb = n_out * k_in * (2 if mode == tfd.W_BF16 else 1) + r * k_in * 2
        out[str(r)] = {"us": round(ms * 1e3, 2), "gbs": round(nb / (ms * 1e-3) / 1e9, 1)}
    print(json.dumps({"case": f"{fmt}{' w8a8' if args.w8a8 else ''} top-{topk}",
                      "lib": os.environ.get("TFD_LIBRARY", "default"), "per_rows": out}),
          flush=True)


def run_ffma_compare(args):
    """The bf16 head (fp32 logits + top-1) at rows 1/4/8/9/12/16 with the tensor-core MMA step
    (the default build) and with the CUDA-core FFMA step of a -DTFD_GEMV_FFMA=1 build (built on
    first use into _build/ffma; its two-n-tile ring is 4 steps deep to keep it from spilling)."""
    from speculative_decoding_draft_row_gb300 import build
    lib = build.build_library(extra_flags=["-DTFD_GEMV_FFMA=1", "-DTFD_GEMV_DEPTH_NT2=4"],
                              build_dir=os.path.join(build.BUILD_DIR, "ffma"))
    res = {}
    for name, env in (("mma", {}), ("ffma", {"TFD_LIBRARY": lib})):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--head", "bf16", "--rows",
                            "0", "--steps", str(args.steps), "--warmup", str(args.warmup)],
                           env=dict(os.environ, **env), cwd=ROOT, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(r.stderr[-2000:])
        res[name] = json.loads(r.stdout.strip().splitlines()[-1])["per_rows"]
    print(json.dumps({"case": "bf16 head, fp32 logits + top-1: MMA vs FFMA step", "ffma_lib": lib,
                      **res}), flush=True)


def run_case(args):
    """Small isolated cases for profiling: one call of one row of the path, repeated."""
    import torch

    from speculative_decoding_draft_row_gb300 import tfd
    from synth import inputs

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    c = args.case
    if c == "attn":
        kr, vr = inputs.rings(PASS_STREAMS, PASS_RING, PASS_HEADS, PASS_DIM)
        krd, vrd = kr.cuda(), vr.cuda()
        q, k, v = (t.cuda() for t in inputs.pass_step_qkv(0))
        pos = torch.full((PASS_STREAMS,), 511, dtype=torch.int32, device="cuda")
        out = torch.empty((PASS_STREAMS, PASS_HEADS * PASS_DIM), dtype=torch.bfloat16,
                          device="cuda")
        fn = lambda: tfd.tfd_window_attn(q, k, v, pos, krd, vrd, PASS_WINDOW, out=out)
    elif c in ("pass", "passfp8"):
        # one 5-step x 4-stream draft pass (bf16 head, or interleaved block-32 FP8 head), eager
        from speculative_decoding_draft_row_gb300.draft_pass import DraftPass
        w, _ = inputs.head(tie_frac=0.01)
        wd = w.cuda()
        del w
        wo_c, wo_s = tfd.tfd_quant_fp8(inputs.linear(HIDDEN, HIDDEN, 40).cuda(), tfd.W_FP8_ROW)
        w2_c, w2_s = tfd.tfd_quant_fp8(inputs.linear(HIDDEN, HIDDEN_FFN, 41).cuda(), tfd.W_FP8_ROW)
        kr, vr = inputs.rings(PASS_STREAMS, PASS_RING, PASS_HEADS, PASS_DIM)
        qkv = [inputs.pass_step_qkv(t, PASS_STREAMS, PASS_HEADS, PASS_DIM) for t in range(PASS_STEPS)]
        us = [inputs.normal_bf16((PASS_STREAMS, HIDDEN_FFN), 1.0, 50 + t) for t in range(PASS_STEPS)]
        if c == "pass":
            head, fmt, sc = wd, tfd.W_BF16, None
        else:
            hc, sc = tfd.tfd_quant_fp8(wd, tfd.W_FP8_BLOCK32_IL)
            head, fmt = hc, tfd.W_FP8_BLOCK32_IL
            del wd
        dp = DraftPass(wo_c, wo_s, w2_c, w2_s, head, fmt, sc, kr.cuda(), vr.cuda(), PASS_WINDOW,
                       PASS_STEPS)
        dp.load([q for q, _, _ in qkv], [k for _, k, _ in qkv], [v for _, _, v in qkv], us,
                [511] * PASS_STREAMS, inputs.normal_bf16((PASS_STREAMS, HIDDEN), 1.0, 60).cuda(),
                [5] * PASS_STREAMS, torch.zeros((PASS_STREAMS, PASS_STEPS), dtype=torch.int32))
        fn = dp.enqueue
    elif c in ("rows17", "rows24", "rows32"):
        # a 17-32-row decode window on the full bf16 head: fp32 logits + fused top-1
        r = int(c[4:])
        w, _ = inputs.head(tie_frac=0.01)
        wd = w.cuda()
        del w
        xr = inputs.rows(r).cuda()
        y = torch.empty((r, VOCAB), dtype=torch.float32, device="cuda")
        tv = torch.empty((r, 1), dtype=torch.float32, device="cuda")
        ti = torch.empty((r, 1), dtype=torch.int32, device="cuda")
        ws = tfd.zeroed_workspace(tfd.tfd_head_gemv_workspace(r, VOCAB, 1))
        fn = lambda: tfd.tfd_head_gemv(wd, tfd.W_BF16, None, xr, tfd.OUT_F32, y=y, topk=1,
                                       top_vals=tv, top_ids=ti, ws=ws)
        for _ in range(args.warmup):
            fn()
        ms = time_graph(fn, args.steps)
        print(json.dumps({"case": c, "us": round(ms * 1e3, 2),
                          "gbs": round(bf16_call_bytes(r) / (ms * 1e-3) / 1e9, 1)}), flush=True)
        return
    elif c in ("rescore", "topk64", "topk512", "twostage"):
        x16 = inputs.rows(16).cuda()
        if c.startswith("topk"):
            kk = int(c[4:])
            z = torch.from_numpy(inputs.normal_f32((16, VOCAB), 1.0, 90)).cuda()
            ws = tfd.zeroed_workspace(tfd.tfd_topk_workspace(16, VOCAB, kk))
            cv = torch.empty((16, kk), dtype=torch.float32, device="cuda")
            ci = torch.empty((16, kk), dtype=torch.int32, device="cuda")
            fn = lambda: tfd.tfd_topk(z, kk, vals=cv, ids=ci, ws=ws)
        else:
            w, _ = inputs.head(tie_frac=0.01)
            wd = w.cuda()
            cand = torch.from_numpy(
                __import__("numpy").random.default_rng([0, 91, 0]).integers(
                    0, VOCAB, size=(16, 512)).astype("int32")).cuda()
            rws = tfd.zeroed_workspace(tfd.tfd_rescore_workspace(16, 512))
            oi = torch.empty(16, dtype=torch.int32, device="cuda")
            ov = torch.empty(16, dtype=torch.float32, device="cuda")
            if c == "rescore":
                fn = lambda: tfd.tfd_rescore(wd, x16, cand, out_ids=oi, out_vals=ov, ws=rws,
                                             want_logits=False)
            else:
                a, b = inputs.low_rank()
                ad, bd = a.cuda(), b.cuda()
                h = torch.empty((16, 256), dtype=torch.float32, device="cuda")
                z = torch.empty((16, VOCAB), dtype=torch.float32, device="cuda")
                tws = tfd.zeroed_workspace(tfd.tfd_head_gemv_workspace(16, VOCAB, 512, 0))
                cv = torch.empty((16, 512), dtype=torch.float32, device="cuda")
                ci = torch.empty((16, 512), dtype=torch.int32, device="cuda")

                def fn():
                    tfd.tfd_head_gemv(bd, tfd.W_BF16, None, x16, tfd.OUT_F32, y=h)
                    tfd.tfd_head_gemv(ad, tfd.W_BF16, None, h, tfd.OUT_F32, y=z, topk=512,
                                      top_vals=cv, top_ids=ci, ws=tws)
                    tfd.tfd_rescore(wd, x16, ci, out_ids=oi, out_vals=ov, ws=rws,
                                    want_logits=False)
    else:
        raise SystemExit(f"unknown case {c}")
    for _ in range(args.warmup):
        fn()
    ms_eager = time_calls(fn, args.steps, stream)
    ms = time_graph(fn, args.steps)
    print(json.dumps({"case": c, "us": round(ms * 1e3, 2), "us_eager": round(ms_eager * 1e3, 2)}),
          flush=True)


def run_trace(args):
    """Phase stamps of the head GEMV kernel from a build with -DTFD_TRACE=1 (built on first use
    into _build/trace): per block the entry, the staged activations, the end of each group and
    the end of the groups, summarised over the blocks of one call (ns). Reproduces the per-phase
    figures quoted in the profiles."""
    if os.environ.get("TFD_TRACE_CHILD") != "1":
        from speculative_decoding_draft_row_gb300 import build
        lib = build.build_library(extra_flags=["-DTFD_TRACE=1"],
                                  build_dir=os.path.join(build.BUILD_DIR, "trace"))
        env = dict(os.environ, TFD_LIBRARY=lib, TFD_TRACE_CHILD="1")
        sys.exit(subprocess.run([sys.executable, os.path.abspath(__file__), *sys.argv[1:]],
                                env=env, cwd=ROOT).returncode)
    import ctypes

    import numpy as np
    import torch

    from speculative_decoding_draft_row_gb300 import tfd
    from synth import inputs

    torch.cuda.set_device(0)
    spec = args.trace.split(":")
    fmt, rows, topk = spec[0], int(spec[1]), int(spec[2])
    mode = {"bf16": tfd.W_BF16, "row": tfd.W_FP8_ROW, "block32": tfd.W_FP8_BLOCK32,
            "block32il": tfd.W_FP8_BLOCK32_IL}[fmt]
    if len(spec) == 5:  # another matrix: N x K ~ N(0, 0.02)
        w = inputs.linear(int(spec[3]), int(spec[4]), 40)
    else:
        w, _ = inputs.head(tie_frac=0.01)
    n_out, k_in = w.shape
    wd = w.cuda()
    del w
    if mode == tfd.W_BF16:
        codes, scales = wd, None
    else:
        codes, scales = tfd.tfd_quant_fp8(wd, mode)
        del wd
    x = inputs.rows(32, hidden=k_in)[:rows].cuda()
    ws = tfd.zeroed_workspace(tfd.tfd_head_gemv_workspace(rows, n_out, max(topk, 1)))
    buf = torch.zeros((1024, 64), dtype=torch.int64, device="cuda")
    lib = tfd.library()
    lib.tfd_trace_set.argtypes = [ctypes.c_void_p]
    f = lambda: tfd.tfd_head_gemv(codes, mode, scales, x, tfd.OUT_NONE, topk=topk,
                                  ws=ws if topk else None)
    for _ in range(args.warmup):
        f()
    torch.cuda.synchronize()
    lib.tfd_trace_set(buf.data_ptr())
    f()
    torch.cuda.synchronize()
    lib.tfd_trace_set(None)
    t = buf.cpu().numpy()
    used = t[:, 0] > 0
    t = t[used]
    t0 = t[:, 0].min()
    med = lambda v: float(statistics.median(v.tolist())) if len(v) else None
    groups = [(t[b, 2:57][t[b, 2:57] > 0] - t[b, 1]) for b in range(len(t))]
    per_group = [float((g[-1] - 0) / len(g)) for g in groups if len(g)]
    gpu_ms = time_graph(f, 40)
    out = {"case": f"{fmt} {n_out}x{k_in} rows {rows} topk {topk}", "blocks": int(used.sum()),
           "graph_us": round(gpu_ms * 1e3, 2),
           "entry_skew_ns": float(t[:, 0].max() - t0),
           "staging_ns_median": med(t[:, 1] - t[:, 0]), "staging_ns_max": float((t[:, 1] - t[:, 0]).max()),
           "staging_phases_ns_median": [med(t[:, q][t[:, q] > 0] - t[:, 0][t[:, q] > 0])
                                        if (t[:, q] > 0).any() else None for q in (57, 58, 59)],
           "first_group_ns_median": med(t[:, 2] - t[:, 1]),
           "group_ns_median": med(np.array(per_group)),
           "groups_per_block": [int(min(len(g) for g in groups)), int(max(len(g) for g in groups))],
           "groups_done_ns_min": float(t[:, 61].min() - t0), "groups_done_ns_max": float(t[:, 61].max() - t0),
           "join_done_ns": float(t[:, 63].max() - t0) if (t[:, 63] > 0).any() else None}
    print(json.dumps(out), flush=True)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = []
    last = None
    for i in range(args.warmup + args.steps):
        r = run_oracle_sample(2.0)
        if i >= args.warmup:
            per_step.append(r)
        last = r
    gbs = statistics.mean(p["gbs"] for p in per_step)
    ms = statistics.mean(p["seconds"] for p in per_step) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,0.02) head, N(0,1) rows)",
        "config": bench_config(int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": last["threads"],
                         "kind": "oracle",
                         "sample": f"each step: the oracle's fp64 GEMV + top-1 on {SAMPLE_ROWS} of "
                                   f"{VOCAB} vocabulary rows at rows 1/5/10/15, about 2 s"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    if len(sys.argv) > 2 and sys.argv[1] == "--oracle-worker":
        oracle_sample_worker(float(sys.argv[2]))
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8", choices=["row", "block32", "block32il"], default=None,
                    help="profiling case: only the FP8 head with fused top-64")
    ap.add_argument("--head", choices=["bf16", "row", "block32", "block32il"], default=None,
                    help="profiling case: one head format alone (see --rows, --topk, --w8a8)")
    ap.add_argument("--rows", type=int, default=None, choices=list(range(0, 33)),
                    help="with --head/--fp8: one row count instead of 1/5/10/15/16 (0: "
                         "1/4/8/9/12/16)")
    ap.add_argument("--topk", type=int, default=None,
                    help="with --head/--fp8: the fused top-k (default 64 for FP8, 1 for bf16)")
    ap.add_argument("--shape", default=None, metavar="N:K",
                    help="with --head: an N x K matrix ~ N(0, 0.02) instead of the head")
    ap.add_argument("--compare-ffma", action="store_true",
                    help="the bf16 head with the MMA step and with the CUDA-core FFMA step")
    ap.add_argument("--w8a8", action="store_true",
                    help="with --head/--fp8: quantise the activation rows to E4M3 in the call")
    ap.add_argument("--case", choices=["attn", "rescore", "topk64", "topk512", "twostage",
                                       "rows17", "rows24", "rows32", "pass", "passfp8"],
                    default=None,
                    help="profiling case: one row of the path alone")
    ap.add_argument("--trace", default=None, metavar="FMT:ROWS:TOPK[:N:K]",
                    help="phase stamps of one head GEMV call from a -DTFD_TRACE=1 build, e.g. "
                         "row:16:64 (FMT bf16, row, block32 or block32il; N:K another matrix "
                         "than the head)")
    ap.add_argument("--no-extras", action="store_true",
                    help="time the headline calls only (no e2e, FP8 or CPU baseline): a small "
                         "case for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.trace:
        run_trace(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.compare_ffma:
        run_ffma_compare(args)
    elif args.fp8 or args.head:
        run_head_case(args)
    elif args.case:
        run_case(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
