"""Thin ctypes binding of libtfd.so: one function per C entry point, same names.

Arguments are torch tensors on the current CUDA device (or None for nullable pointers); the binding
only checks dtypes/devices, passes ``data_ptr()`` and sizes, and raises ``TfdError`` on a non-zero
status. Every step of the computation runs in the library's kernels; there is no fallback: if the
library cannot be loaded the import of a function fails with an error.
"""
import ctypes
import os

import torch

from . import build as _build

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_DATA, ERR_TIMEOUT = range(7)
W_BF16, W_FP8_ROW, W_FP8_BLOCK32, W_FP8_BLOCK32_IL = 0, 1, 2, 3
X_BF16, X_F32, X_BF16_E4M3 = 0, 1, 2
OUT_NONE, OUT_F32, OUT_BF16, OUT_ADD_BF16 = 0, 1, 2, 3
MAX_ROWS, MAX_TOPK, MAX_WINDOW = 32, 512, 511

_c = ctypes
_vp, _i64, _i32, _sz, _f32 = _c.c_void_p, _c.c_int64, _c.c_int, _c.c_size_t, _c.c_float

SIGNATURES = {
    "tfd_status_string": (_c.c_char_p, [_i32]),
    "tfd_version": (_i32, []),
    "tfd_quant_fp8": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "tfd_head_gemv_workspace": (_sz, [_i32, _i64, _i32, _i32]),
    "tfd_head_gemv_max_k": (_i64, [_i32, _i32]),
    "tfd_head_gemv": (_i32, [_vp, _i32, _vp, _i64, _i64, _vp, _i32, _i32, _i64, _i32, _vp, _i64,
                             _i32, _i32, _vp, _vp, _vp, _i64, _vp, _vp, _sz, _vp, _vp]),
    "tfd_head_gemv_noalloc": (_i32, [_vp, _i32, _vp, _i64, _i64, _vp, _i32, _i32, _i64, _i32,
                                     _vp, _i64, _i32, _i32, _vp, _vp, _vp, _i64, _vp, _vp, _vp]),
    "tfd_topk_workspace": (_sz, [_i32, _i64, _i32]),
    "tfd_topk": (_i32, [_vp, _i32, _i64, _i64, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tfd_rescore_workspace": (_sz, [_i32, _i32]),
    "tfd_rescore": (_i32, [_vp, _i64, _i64, _vp, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _sz, _vp,
                           _vp]),
    "tfd_window_attn": (_i32, [_vp, _vp, _vp, _vp, _vp, _f32, _f32, _vp, _vp, _vp, _i32, _i32,
                               _i32, _i32, _i32, _vp, _vp, _vp]),
    "tfd_accept": (_i32, [_vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "tfd_fp8_block32_relayout": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp]),
    "tfd_rmsnorm": (_i32, [_vp, _i64, _vp, _f32, _i32, _i64, _vp, _i64, _vp]),
    "tfd_swiglu": (_i32, [_vp, _vp, _i64, _i32, _i64, _vp, _i64, _vp]),
    "tfd_absorb": (_i32, [_vp, _vp, _vp, _f32, _f32, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                          _vp, _vp]),
}

_lib = None


class TfdError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: status {status} ({status_string(status)})")


def library(build=True):
    """The loaded libtfd.so (built first when missing or stale). The environment variable
    TFD_LIBRARY names another build of the library to load instead (it must exist)."""
    global _lib
    if _lib is None:
        path = os.environ.get("TFD_LIBRARY")
        if not path:
            path = _build.build_library() if build else _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"libtfd.so not found at {path}")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def status_string(status):
    return library().tfd_status_string(int(status)).decode()


def _p(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, st):
    if st != OK:
        raise TfdError(fn, st)


def _dev(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tfd tensors must be CUDA tensors")


def zeroed_workspace(nbytes, device=None):
    """A zero-filled device workspace (the calls leave it zeroed again)."""
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device or "cuda")


# ---- entry points ---------------------------------------------------------------------------

def tfd_quant_fp8(w, mode, codes=None, scales=None, stream=None):
    """FP8 codes of a bf16 weight [n][k]: mode W_FP8_ROW (float scales [n]), W_FP8_BLOCK32 or
    W_FP8_BLOCK32_IL (uint8 scales [n/32][k/32]; IL writes the interleaved code layout).
    Returns (codes, scales)."""
    _dev(w)
    n, k = w.shape
    if codes is None:
        codes = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = (torch.empty(n, dtype=torch.float32, device=w.device) if mode == W_FP8_ROW else
                  torch.empty((max(n // 32, 1), max(k // 32, 1)), dtype=torch.uint8,
                              device=w.device))
    st = library().tfd_quant_fp8(_p(w), n, k, mode, _p(codes), _p(scales), _stream(stream))
    _check("tfd_quant_fp8", st)
    return codes, scales


def tfd_head_gemv_workspace(rows, n, topk, parts=0):
    return library().tfd_head_gemv_workspace(rows, n, topk, parts)


def tfd_head_gemv_max_k(rows, xfmt=X_BF16):
    return library().tfd_head_gemv_max_k(rows, xfmt)


def tfd_head_gemv(w, wfmt, w_scales, x, out_mode=OUT_F32, y=None, topk=0, parts=0, id_map=None,
                  top_vals=None, top_ids=None, ws=None, dev_status=None, n=None, top1_conf=None,
                  stream=None, act_e4m3=False):
    """Few-row head GEMV with optional output and fused top-k (top-1 optionally with its softmax
    probability in ``top1_conf`` [rows]). ``act_e4m3`` (FP8 weights, bf16 x): quantise the
    activation rows to E4M3 in the call (W8A8). Returns (y, top_vals, top_ids)."""
    _dev(w, x, y, id_map, ws)
    n = w.shape[0] if n is None else n
    k = w.shape[1]
    rows = x.shape[0]
    xfmt = X_F32 if x.dtype == torch.float32 else (X_BF16_E4M3 if act_e4m3 else X_BF16)
    if y is None and out_mode != OUT_NONE:
        dt = torch.float32 if out_mode == OUT_F32 else torch.bfloat16
        y = torch.empty((rows, n), dtype=dt, device=x.device)
    ldy = y.stride(0) if y is not None else 0
    if topk > 0 and top_vals is None:
        top_vals = torch.empty((rows, topk), dtype=torch.float32, device=x.device)
        top_ids = torch.empty((rows, topk), dtype=torch.int32, device=x.device)
    if ws is None and topk > 0:
        ws = zeroed_workspace(tfd_head_gemv_workspace(rows, n, topk, parts), x.device)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    ldt = top_ids.stride(0) if (topk > 0 and top_ids.dim() == 2) else topk
    if topk > 0 and top_vals.stride(0) != ldt:
        raise ValueError("top_vals and top_ids must share their row stride")
    st = library().tfd_head_gemv(_p(w), wfmt, _p(w_scales), n, k, _p(x), xfmt, rows, x.stride(0),
                                 out_mode, _p(y), ldy, topk, parts, _p(id_map), _p(top_vals),
                                 _p(top_ids), ldt, _p(top1_conf), _p(ws), ws_bytes,
                                 _p(dev_status), _stream(stream))
    _check("tfd_head_gemv", st)
    return y, top_vals, top_ids


NOALLOC_SCRATCH_BYTES = 1048576


def tfd_head_gemv_noalloc(w, wfmt, w_scales, x, out_mode=OUT_F32, y=None, topk=0, parts=0,
                          id_map=None, top_vals=None, top_ids=None, dev_status=None,
                          top1_conf=None, stream=None):
    """tfd_head_gemv on the library's fixed scratch (no workspace argument): for callers that
    cannot allocate device memory. Outputs must be passed in by such callers; the defaults here
    allocate them only for convenience. Returns (y, top_vals, top_ids)."""
    _dev(w, x, y, id_map)
    n, k = w.shape[0], w.shape[1]
    rows = x.shape[0]
    xfmt = X_F32 if x.dtype == torch.float32 else X_BF16
    if y is None and out_mode != OUT_NONE:
        dt = torch.float32 if out_mode == OUT_F32 else torch.bfloat16
        y = torch.empty((rows, n), dtype=dt, device=x.device)
    if topk > 0 and top_vals is None:
        top_vals = torch.empty((rows, topk), dtype=torch.float32, device=x.device)
        top_ids = torch.empty((rows, topk), dtype=torch.int32, device=x.device)
    ldt = top_ids.stride(0) if topk > 0 else 0
    st = library().tfd_head_gemv_noalloc(_p(w), wfmt, _p(w_scales), n, k, _p(x), xfmt, rows,
                                         x.stride(0), out_mode, _p(y),
                                         y.stride(0) if y is not None else 0, topk, parts,
                                         _p(id_map), _p(top_vals), _p(top_ids), ldt,
                                         _p(top1_conf), _p(dev_status), _stream(stream))
    _check("tfd_head_gemv_noalloc", st)
    return y, top_vals, top_ids


def tfd_topk_workspace(rows, n, k):
    return library().tfd_topk_workspace(rows, n, k)


def tfd_topk(logits, k, id_map=None, vals=None, ids=None, ws=None, n=None, stream=None):
    """Top-k of fp32 logits [rows][>= n]. Returns (vals, ids)."""
    _dev(logits, id_map, ws)
    rows = logits.shape[0]
    n = logits.shape[1] if n is None else n
    if vals is None:
        vals = torch.empty((rows, k), dtype=torch.float32, device=logits.device)
        ids = torch.empty((rows, k), dtype=torch.int32, device=logits.device)
    if ws is None:
        ws = zeroed_workspace(tfd_topk_workspace(rows, n, k), logits.device)
    st = library().tfd_topk(_p(logits), rows, n, logits.stride(0), k, _p(id_map), _p(vals),
                            _p(ids), _p(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check("tfd_topk", st)
    return vals, ids


def tfd_rescore_workspace(rows, cand_k):
    return library().tfd_rescore_workspace(rows, cand_k)


def tfd_rescore(w_exact, x, cand, cand_logits=None, out_ids=None, out_vals=None, ws=None,
                dev_status=None, want_logits=True, stream=None):
    """Exact logits of the candidates [rows][cand_k] and their argmax. Returns
    (cand_logits, out_ids, out_vals)."""
    _dev(w_exact, x, cand, ws)
    vocab, k = w_exact.shape
    rows, cand_k = cand.shape
    dev = x.device
    if cand_logits is None and want_logits:
        cand_logits = torch.empty((rows, cand_k), dtype=torch.float32, device=dev)
    if out_ids is None:
        out_ids = torch.empty(rows, dtype=torch.int32, device=dev)
        out_vals = torch.empty(rows, dtype=torch.float32, device=dev)
    if ws is None:
        ws = zeroed_workspace(tfd_rescore_workspace(rows, cand_k), dev)
    st = library().tfd_rescore(_p(w_exact), vocab, k, _p(x), rows, _p(cand), cand_k,
                               _p(cand_logits), _p(out_ids), _p(out_vals), _p(ws),
                               ws.numel() * ws.element_size(), _p(dev_status), _stream(stream))
    _check("tfd_rescore", st)
    return cand_logits, out_ids, out_vals


def tfd_window_attn(q, k_new, v_new, pos, k_ring, v_ring, window, q_gamma=None, k_gamma=None,
                    eps=1e-6, rope_base=10000.0, out=None, dev_status=None, stream=None):
    """qk_norm + RoPE + ring write + window attention. Returns out [streams][heads*dim]."""
    _dev(q, k_new, v_new, pos, k_ring, v_ring)
    streams, heads, dim = q.shape
    ring = k_ring.shape[1]
    if out is None:
        out = torch.empty((streams, heads * dim), dtype=torch.bfloat16, device=q.device)
    st = library().tfd_window_attn(_p(q), _p(k_new), _p(v_new), _p(q_gamma), _p(k_gamma),
                                   float(eps), float(rope_base), _p(pos), _p(k_ring), _p(v_ring),
                                   ring, window, streams, heads, dim, _p(out), _p(dev_status),
                                   _stream(stream))
    _check("tfd_window_attn", st)
    return out


def tfd_accept(drafts, n_asked, draws, n_kept=None, asked_hist=None, kept_hist=None,
               dev_status=None, stream=None):
    """Accept-prefix count. Returns n_kept [streams]."""
    _dev(drafts, n_asked, draws)
    streams, win = drafts.shape
    if n_kept is None:
        n_kept = torch.empty(streams, dtype=torch.int32, device=drafts.device)
    st = library().tfd_accept(_p(drafts), _p(n_asked), _p(draws), streams, win, _p(n_kept),
                              _p(asked_hist), _p(kept_hist), _p(dev_status), _stream(stream))
    _check("tfd_accept", st)
    return n_kept


def tfd_rmsnorm(x, gamma=None, eps=1e-6, out=None, stream=None):
    """RMSNorm of the rows of x [rows][hidden] (bf16). out may be x (in place). Returns out."""
    _dev(x, gamma, out)
    rows, hidden = x.shape
    if out is None:
        out = torch.empty_like(x)
    st = library().tfd_rmsnorm(_p(x), x.stride(0), _p(gamma), float(eps), rows, hidden, _p(out),
                               out.stride(0), _stream(stream))
    _check("tfd_rmsnorm", st)
    return out


def tfd_swiglu(g, u, out=None, stream=None):
    """bf16(bf16(SiLU(g)) * u) of two [rows][cols] bf16 tensors with the same row stride."""
    _dev(g, u, out)
    rows, cols = g.shape
    if u.shape != g.shape or u.stride(0) != g.stride(0):
        raise ValueError("g and u must have the same shape and row stride")
    if out is None:
        out = torch.empty_like(g)
    st = library().tfd_swiglu(_p(g), _p(u), g.stride(0), rows, cols, _p(out), out.stride(0),
                              _stream(stream))
    _check("tfd_swiglu", st)
    return out


def tfd_absorb(k_rows, v_rows, p0, k_ring, v_ring, k_gamma=None, eps=1e-6, rope_base=10000.0,
               dev_status=None, stream=None):
    """Write n rows per stream (k_rows, v_rows [streams][n][heads][dim]) into the rings at positions
    p0[s] .. p0[s] + n - 1. Refuses n > ring."""
    _dev(k_rows, v_rows, p0, k_ring, v_ring, k_gamma)
    streams, n, heads, dim = k_rows.shape
    ring = k_ring.shape[1]
    st = library().tfd_absorb(_p(k_rows), _p(v_rows), _p(k_gamma), float(eps), float(rope_base),
                              _p(p0), n, _p(k_ring), _p(v_ring), ring, streams, heads, dim,
                              _p(dev_status), _stream(stream))
    _check("tfd_absorb", st)


def tfd_fp8_block32_relayout(codes, to_interleaved=True, out=None, stream=None):
    """Block-32 FP8 codes [n][k] between the plain and the interleaved layout. Returns out."""
    _dev(codes, out)
    n, k = codes.shape
    if out is None:
        out = torch.empty_like(codes)
    st = library().tfd_fp8_block32_relayout(_p(codes), n, k, 1 if to_interleaved else 0, _p(out),
                                            _stream(stream))
    _check("tfd_fp8_block32_relayout", st)
    return out
