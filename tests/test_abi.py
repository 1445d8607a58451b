"""The C-ABI library builds, loads and exports every symbol include/tfd.h declares; host-side
argument checks refuse bad calls before touching the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_draft_row_gb300 import build, tfd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "tfd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tfd_[a-z0-9_]+)\s*\(", text)))


def test_library_builds_and_exports_every_declared_symbol():
    path = build.build_library()
    assert os.path.exists(path)
    lib = ctypes.CDLL(path)
    names = declared_symbols()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(tfd.SIGNATURES)


def test_status_strings_and_version():
    assert tfd.status_string(0) == "ok"
    assert "workspace" in tfd.status_string(3)
    assert tfd.library().tfd_version() >= 100


def test_workspace_queries():
    lib = tfd.library()
    assert lib.tfd_head_gemv_workspace(1, 163840, 0, 0) == 0
    assert lib.tfd_head_gemv_workspace(1, 163840, 1, 0) > 0
    assert lib.tfd_head_gemv_workspace(16, 163840, 64, 0) >= 16 * 163840 * 4
    assert lib.tfd_head_gemv_workspace(33, 163840, 1, 0) == 0          # rows > 32
    assert lib.tfd_head_gemv_workspace(32, 163840, 64, 0) >= 32 * 163840 * 4
    assert lib.tfd_head_gemv_workspace(1, 100, 513, 0) == 0            # topk > 512
    assert lib.tfd_topk_workspace(16, 163840, 512) > 0
    assert lib.tfd_topk_workspace(1, 10, 11) == 0                      # k > n
    assert lib.tfd_rescore_workspace(16, 512) > 0
    assert lib.tfd_rescore_workspace(16, 513) == 0
    assert lib.tfd_head_gemv_max_k(16, tfd.X_BF16) >= 4096
    assert lib.tfd_head_gemv_max_k(4, tfd.X_BF16) >= 11008
    assert lib.tfd_head_gemv_max_k(16, tfd.X_F32) >= 256
    assert lib.tfd_head_gemv_max_k(32, tfd.X_BF16) >= 4096            # k split over a cluster
    assert lib.tfd_head_gemv_max_k(32, tfd.X_F32) == 0                # fp32 stops at 16 rows
    assert lib.tfd_head_gemv_max_k(16, tfd.X_BF16_E4M3) >= 4096


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced by refused calls


def gemv(**kw):
    a = dict(w=FAKE, wfmt=0, ws_=None, n=4096, k=256, x=FAKE, xfmt=0, rows=1, ldx=256, out=1,
             y=FAKE * 2, ldy=4096, topk=0, parts=0, id_map=None, tv=None, ti=None, ldt=0,
             conf=None, ws=None, wsb=0, st=None, stream=None)
    a.update(kw)
    return tfd.library().tfd_head_gemv(a["w"], a["wfmt"], a["ws_"], a["n"], a["k"], a["x"],
                                       a["xfmt"], a["rows"], a["ldx"], a["out"], a["y"], a["ldy"],
                                       a["topk"], a["parts"], a["id_map"], a["tv"], a["ti"],
                                       a["ldt"], a["conf"], a["ws"], a["wsb"], a["st"],
                                       a["stream"])


@pytest.mark.parametrize("bad,code", [
    (dict(rows=0), 1), (dict(rows=33), 1), (dict(k=250), 1), (dict(k=0), 1), (dict(n=0), 1),
    (dict(wfmt=4), 1), (dict(xfmt=3), 1), (dict(xfmt=2), 1),   # W8A8 needs FP8 weights
    (dict(rows=17, xfmt=1, ldx=256), 2),                         # fp32 activations: 16 rows
    (dict(w=None), 1), (dict(x=None), 1), (dict(w=FAKE + 8), 1), (dict(ldx=100), 1),
    (dict(wfmt=1), 1), (dict(wfmt=2, ws_=FAKE, n=100), 1), (dict(wfmt=3), 1), (dict(out=4), 1),
    (dict(y=None), 1), (dict(ldy=10), 1), (dict(topk=513), 1), (dict(topk=1), 1),
    (dict(topk=1, tv=FAKE, ti=FAKE), 3), (dict(parts=-1), 1), (dict(parts=5000), 1),
    (dict(topk=8, tv=FAKE, ti=FAKE, ldt=4), 1),
    (dict(topk=8, tv=FAKE, ti=FAKE, conf=FAKE * 4), 1),   # confidence only with top-1
    (dict(y=FAKE), 1),  # y overlaps x
    (dict(rows=16, k=65536, ldx=65536, y=FAKE * 64), 2),  # activation tile past shared memory
])
def test_head_gemv_refusals(bad, code):
    assert gemv(**bad) == code


def test_other_refusals():
    lib = tfd.library()
    assert lib.tfd_quant_fp8(FAKE, 64, 250, 1, FAKE, FAKE, None) == 1
    assert lib.tfd_quant_fp8(FAKE, 48, 256, 2, FAKE, FAKE, None) == 1      # n % 32
    assert lib.tfd_quant_fp8(FAKE, 64, 256, 0, FAKE, FAKE, None) == 1      # mode
    assert lib.tfd_quant_fp8(None, 64, 256, 1, FAKE, FAKE, None) == 1
    assert lib.tfd_topk(FAKE, 1, 10, 10, 11, None, FAKE, FAKE, FAKE, 1 << 20, None) == 1
    assert lib.tfd_topk(FAKE, 1, 10, 9, 1, None, FAKE, FAKE, FAKE, 1 << 20, None) == 1  # ld < n
    assert lib.tfd_topk(FAKE, 1, 10000, 10000, 8, None, FAKE, FAKE, None, 0, None) == 3
    assert lib.tfd_rescore(FAKE, 100, 256, FAKE, 1, FAKE, 513, None, FAKE, None, FAKE, 1 << 20,
                           None, None) == 1
    assert lib.tfd_rescore(FAKE, 100, 256, FAKE, 1, FAKE, 8, None, FAKE, None, None, 0, None,
                           None) == 3
    args = [FAKE, FAKE, FAKE, None, None, 1e-6, 10000.0, FAKE, FAKE, FAKE]
    assert lib.tfd_window_attn(*args, 512, 512, 4, 32, 128, FAKE, None, None) == 1   # window 512
    assert lib.tfd_window_attn(*args, 511, 511, 4, 32, 128, FAKE, None, None) == 1   # ring small
    assert lib.tfd_window_attn(*args, 528, 511, 4, 32, 64, FAKE, None, None) == 2    # dim 64
    assert lib.tfd_accept(FAKE, FAKE, FAKE, 4, 0, FAKE, None, None, None, None) == 1
    assert lib.tfd_accept(FAKE, FAKE, FAKE, 4, 5, FAKE, FAKE, None, None, None) == 1
