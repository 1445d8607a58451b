"""Failure detection of the bounded device waits, without a GPU fault: a build with
-DTFD_TEST_STALL_EXCHANGE=1 has the second block of each two-block cluster split drop its partial
sums, so the leader's waits run out (about a second) and the call reports TFD_ERR_TIMEOUT in its
device status; the kernel ends, the context stays usable, and the next call (with a fresh status)
computes normally on the default build's code paths that need no exchange.

Both exchanges are covered: the tcgen05 kernel of 17-32 bf16 rows, and the register-ring kernel's
split of two (a 4096 x 4096 row-scaled FP8 matrix at 4 rows, one group per cluster).
The child process loads the planted build through TFD_LIBRARY (one library per process)."""
import os
import subprocess
import sys

import pytest

from helpers import need_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, torch
sys.path.insert(0, sys.argv[1])
from speculative_decoding_draft_row_gb300 import tfd
from synth import inputs
torch.cuda.set_device(0)
out = {}
# tcgen05, 32 rows of bf16
w = inputs.normal_bf16((4096, 4096), 0.02, 1).cuda()
x = inputs.normal_bf16((32, 4096), 1.0, 2).cuda()
st = torch.zeros(1, dtype=torch.int32, device="cuda")
tfd.tfd_head_gemv(w, tfd.W_BF16, None, x, tfd.OUT_F32, topk=1, dev_status=st)
torch.cuda.synchronize()
out["tc32"] = int(st.item())
# the register-ring kernel's split of two: FP8 row scale, 4 rows, output added to bf16
c, s = tfd.tfd_quant_fp8(w, tfd.W_FP8_ROW)
x4 = inputs.normal_bf16((4, 4096), 1.0, 3).cuda()
y = torch.zeros((4, 4096), dtype=torch.bfloat16, device="cuda")
st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
tfd.tfd_head_gemv(c, tfd.W_FP8_ROW, s, x4, tfd.OUT_ADD_BF16, y=y, dev_status=st2)
torch.cuda.synchronize()
out["split2"] = int(st2.item())
# the context is still usable: a call with no exchange (16 rows, no split) succeeds
st3 = torch.zeros(1, dtype=torch.int32, device="cuda")
w16 = inputs.normal_bf16((20480, 4096), 0.02, 4).cuda()
x16 = inputs.normal_bf16((16, 4096), 1.0, 5).cuda()
yy, _, ti = tfd.tfd_head_gemv(w16, tfd.W_BF16, None, x16, tfd.OUT_F32, topk=1, dev_status=st3)
torch.cuda.synchronize()
ref = (x16.float() @ w16.float().T).argmax(1)
out["after"] = int(st3.item())
out["after_top1_ok"] = bool((ti[:, 0].long() == ref).float().mean().item() > 0.9)
print(json.dumps(out))
"""


def test_a_dropped_exchange_times_out_and_reports_it():
    need_gpu()
    from speculative_decoding_draft_row_gb300 import build
    lib = build.build_library(extra_flags=["-DTFD_TEST_STALL_EXCHANGE=1"],
                              build_dir=os.path.join(build.BUILD_DIR, "stall"))
    env = dict(os.environ, TFD_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    out = json.loads(r.stdout.strip().splitlines()[-1])
    timeout = 6  # TFD_ERR_TIMEOUT
    assert out["tc32"] == timeout and out["split2"] == timeout, out
    assert out["after"] == 0 and out["after_top1_ok"], out
