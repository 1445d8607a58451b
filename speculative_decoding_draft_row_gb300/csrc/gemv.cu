// gemv.cu - the C entry points of the few-row head GEMV (tfd_head_gemv and its workspace and
// size queries); the kernels are in gemv_kernel.cuh, instantiated per weight format in gemv_w*.cu.
//
// Follows the TFE draft head page (#42), commit "pass kernels and FP8 linears": GEMV over bf16 and
// e4m3 weights for up to 16 rows, out bf16 / fp32 / added to bf16, and the top-1 of a vocabulary
// row in parts and a join; the DSpark FP8 head page (#3296), "FP8 draft head".
#include "gemv_kernel.cuh"

TFD_GEMV_EXTERN(TFD_W_BF16)
TFD_GEMV_EXTERN(TFD_W_FP8_ROW)
TFD_GEMV_EXTERN(TFD_W_FP8_BLOCK32)
TFD_GEMV_EXTERN(TFD_W_FP8_BLOCK32_IL)

// Groups taken from a queue in the workspace when there is one (1), or a static split (0).
#ifndef TFD_GEMV_QUEUE
#define TFD_GEMV_QUEUE 1
#endif

namespace {

using namespace tfd_gemv;

// The phase-stamp buffer of TFD_TRACE builds (set by tfd_trace_set; always null otherwise).
uint64_t* g_trace = nullptr;

// Whether a call's activation tile fits shared memory (with k split over a cluster if needed).
bool gemv_fits(int wfmt, int xfmt, int rows, int64_t k) {
  const int nt = rows <= 8 ? 1 : rows <= 16 ? 2 : 4;
  if (nt == 4 && xfmt == TFD_X_F32) return false;
#define TFD_FITS(WF, XF)                                                                       \
  (nt == 1 ? gemv_min_split<WF, XF, 1, 4>(k) : nt == 2 ? gemv_min_split<WF, XF, 2, 4>(k)         \
           : gemv_min_split<WF, XF, 4, 4>(k)) > 0
#define TFD_FITS_X(WF)                                                                         \
  (xfmt == TFD_X_F32 ? TFD_FITS(WF, TFD_X_F32)                                                 \
                     : xfmt == TFD_X_BF16_E4M3 ? TFD_FITS(TFD_W_FP8_ROW, TFD_X_BF16_E4M3)        \
                                               : TFD_FITS(WF, TFD_X_BF16))
  if (wfmt == TFD_W_FP8_ROW) return TFD_FITS_X(TFD_W_FP8_ROW);
  if (wfmt == TFD_W_FP8_BLOCK32) return TFD_FITS_X(TFD_W_FP8_BLOCK32);
  if (wfmt == TFD_W_FP8_BLOCK32_IL) return TFD_FITS_X(TFD_W_FP8_BLOCK32_IL);
  return TFD_FITS_X(TFD_W_BF16);
#undef TFD_FITS_X
#undef TFD_FITS
}

struct GemvWs {
  uint32_t* counter;
  uint64_t* part_keys;
  float2* part_ms;
  float* logits;
  uint32_t* submax;
  uint32_t* part_max;
  void* topk_ws;
  size_t topk_bytes;
};

// Workspace: [counter | part keys for top-1 | fp32 logits for top-k > 1 | sub-group maxima for
// top-k > 1 | part maxima for top-k > 1 | top-k workspace].
size_t gemv_ws_layout(int rows, int64_t n, int topk, bool logits_in_y, char* base, GemvWs* out) {
  size_t off = 256;
  // top-1: per part a key and an online-softmax pair per row
  size_t keys = topk == 1 ? tfd_host::round_up((size_t)kMaxParts * rows * 8, 256) * 2 : 0;
  size_t lg = (topk > 1 && !logits_in_y) ? tfd_host::round_up((size_t)rows * n * 4, 256) : 0;
  size_t sub = topk > 1 ? tfd_host::round_up((size_t)rows * ((n + 15) / 16) * 4, 256) : 0;
  size_t pm = topk > 1 ? tfd_host::round_up((size_t)kMaxParts * rows * 4, 256) : 0;
  size_t tk = topk > 1 ? tfd_internal::topk_workspace(rows, n, topk) : 0;
  if (out) {
    out->counter = reinterpret_cast<uint32_t*>(base);
    out->part_keys = keys ? reinterpret_cast<uint64_t*>(base + off) : nullptr;
    out->part_ms = keys ? reinterpret_cast<float2*>(base + off + keys / 2) : nullptr;
    out->logits = lg ? reinterpret_cast<float*>(base + off + keys) : nullptr;
    out->submax = sub ? reinterpret_cast<uint32_t*>(base + off + keys + lg) : nullptr;
    out->part_max = pm ? reinterpret_cast<uint32_t*>(base + off + keys + lg + sub) : nullptr;
    out->topk_ws = tk ? base + off + keys + lg + sub + pm : nullptr;
    out->topk_bytes = tk;
  }
  if (topk == 0) return 0;
  return off + keys + lg + sub + pm + tk;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
  return pa < pb + nb && pb < pa + na;
}

}  // namespace

extern "C" size_t tfd_head_gemv_workspace(int rows, int64_t n, int topk, int parts) {
  (void)parts;
  if (rows < 1 || rows > TFD_MAX_ROWS || n < 1 || topk < 0 || topk > TFD_MAX_TOPK || topk > n)
    return 0;
  // The fp32 logits of top-k > 1 are counted in the workspace; a call with F32 output keeps them
  // in y instead and needs less.
  return gemv_ws_layout(rows, n, topk, false, nullptr, nullptr);
}

extern "C" int64_t tfd_head_gemv_max_k(int rows, int xfmt) {
  if (rows < 1 || rows > TFD_MAX_ROWS || xfmt < TFD_X_BF16 || xfmt > TFD_X_BF16_E4M3) return 0;
  int64_t best = 0;
  for (int64_t k = 256; k <= (1 << 20); k += 256) {
    bool ok = true;
    for (int wf = xfmt == TFD_X_BF16_E4M3 ? 1 : 0; wf < 4 && ok; ++wf)
      ok = gemv_fits(wf, xfmt, rows, k);
    if (!ok) break;
    best = k;
  }
  return best;
}

// gemv_tc.cu: the tcgen05 form for 17-32 rows of bf16 (sets *taken when it takes the call).
tfd_status gemv_tc_launch(const tfd_gemv::GemvArgs& g, int wfmt, int xfmt, int parts_req,
                          cudaStream_t stream, bool* taken);

extern "C" tfd_status tfd_head_gemv(const void* w, int wfmt, const void* w_scales, int64_t n,
                                    int64_t k, const void* x, int xfmt, int rows, int64_t ldx,
                                    int out_mode, void* y, int64_t ldy, int topk, int parts,
                                    const int32_t* id_map, float* top_vals, int32_t* top_ids,
                                    int64_t ldt, float* top1_conf, void* ws, size_t ws_bytes,
                                    int32_t* dev_status, void* stream) {
  using tfd_host::aligned;
  if (!w || !x) return TFD_ERR_INVALID;
  if (wfmt < TFD_W_BF16 || wfmt > TFD_W_FP8_BLOCK32_IL) return TFD_ERR_INVALID;
  if (xfmt < TFD_X_BF16 || xfmt > TFD_X_BF16_E4M3) return TFD_ERR_INVALID;
  if (xfmt == TFD_X_BF16_E4M3 && wfmt == TFD_W_BF16) return TFD_ERR_INVALID;  // W8A8 only
  if (out_mode < TFD_OUT_NONE || out_mode > TFD_OUT_ADD_BF16) return TFD_ERR_INVALID;
  if (rows < 1 || rows > TFD_MAX_ROWS) return TFD_ERR_INVALID;
  if (n < 1 || n > (int64_t)INT32_MAX || k < 16 || k % 16 != 0) return TFD_ERR_INVALID;
  if (wfmt != TFD_W_BF16 && !w_scales) return TFD_ERR_INVALID;
  if (wfmt == TFD_W_FP8_BLOCK32 && (n % 32 != 0 || k % 32 != 0)) return TFD_ERR_INVALID;
  if (wfmt == TFD_W_FP8_BLOCK32_IL && (n % 32 != 0 || k % 64 != 0)) return TFD_ERR_INVALID;
  const size_t xb = xfmt == TFD_X_F32 ? 4 : 2;
  if (ldx < k || ((size_t)ldx * xb) % 16 != 0) return TFD_ERR_INVALID;
  if (!aligned(w, 16) || !aligned(x, 16)) return TFD_ERR_INVALID;
  if (w_scales && !aligned(w_scales, 4)) return TFD_ERR_INVALID;
  if (topk < 0 || topk > TFD_MAX_TOPK || topk > n) return TFD_ERR_INVALID;
  if (topk > 0 && (!top_vals || !top_ids || !aligned(top_vals, 4) || !aligned(top_ids, 4)))
    return TFD_ERR_INVALID;
  if (ldt == 0) ldt = topk;
  if (topk > 0 && ldt < topk) return TFD_ERR_INVALID;
  if (top1_conf && (topk != 1 || !aligned(top1_conf, 4))) return TFD_ERR_INVALID;
  if (parts < 0 || parts > kMaxParts) return TFD_ERR_INVALID;
  if (id_map && !aligned(id_map, 4)) return TFD_ERR_INVALID;
  const size_t yb = out_mode == TFD_OUT_F32 ? 4 : 2;
  if (out_mode != TFD_OUT_NONE) {
    if (!y || ldy < n || !aligned(y, yb)) return TFD_ERR_INVALID;
    if (overlaps(x, (size_t)rows * ldx * xb, y, (size_t)rows * ldy * yb)) return TFD_ERR_INVALID;
  }
  const bool logits_in_y = out_mode == TFD_OUT_F32;
  GemvWs wl;
  size_t need = gemv_ws_layout(rows, n, topk, logits_in_y, reinterpret_cast<char*>(ws), &wl);
  if (need > 0 && (!ws || ws_bytes < need || !aligned(ws, 16))) return TFD_ERR_WORKSPACE;
  if (!gemv_fits(wfmt, xfmt, rows, k)) return TFD_ERR_UNSUPPORTED;

  GemvArgs a{};
  a.w = w; a.scales = w_scales; a.n = n; a.k = k; a.x = x; a.ldx = ldx; a.rows = rows;
  a.out_mode = out_mode; a.y = y; a.ldy = ldy; a.topk = topk; a.id_map = id_map;
  a.logits = nullptr;
  a.ld_logits = 0;
  a.submax = nullptr;
  a.part_max = nullptr;
  if (topk > 1) {
    a.logits = logits_in_y ? reinterpret_cast<float*>(y) : wl.logits;
    a.ld_logits = logits_in_y ? ldy : n;
    a.submax = wl.submax;
    a.part_max = wl.part_max;
  }
  int parts_used = 0;
  a.parts_used = &parts_used;
  a.trace = g_trace;
  a.status = dev_status;
  // groups taken from a queue in the workspace (bit-identical results; not with the confidence,
  // whose merge order would then follow the blocks' shares)
  a.queue = (TFD_GEMV_QUEUE && wl.counter != nullptr && need > 0 && top1_conf == nullptr)
                ? wl.counter + 1
                : nullptr;
  a.part_keys = wl.part_keys;
  a.counter = wl.counter;
  a.top_vals = top_vals;
  a.top_ids = top_ids;
  a.ldt = ldt;
  a.top1_conf = top1_conf;
  a.part_ms = wl.part_ms;
  a.ngroups = 0;  // set by the launcher for its group size
  cudaStream_t s = tfd_host::as_stream(stream);
  tfd_status st;
  bool taken = false;
  st = gemv_tc_launch(a, wfmt, xfmt, parts, s, &taken);  // 17-32 rows of bf16 on tcgen05
  if (st != TFD_OK) return st;
  if (taken) {
    if (topk <= 1) return st;
    return tfd_internal::topk_launch(a.logits, rows, n, a.ld_logits, topk, id_map, top_vals,
                                     top_ids, ldt, wl.submax, wl.part_max, parts_used, wl.topk_ws,
                                     wl.topk_bytes, s);
  }
  if (wfmt == TFD_W_FP8_ROW) st = gemv_launch_x<TFD_W_FP8_ROW>(a, xfmt, parts, s);
  else if (wfmt == TFD_W_FP8_BLOCK32) st = gemv_launch_x<TFD_W_FP8_BLOCK32>(a, xfmt, parts, s);
  else if (wfmt == TFD_W_FP8_BLOCK32_IL)
    st = gemv_launch_x<TFD_W_FP8_BLOCK32_IL>(a, xfmt, parts, s);
  else st = gemv_launch_x<TFD_W_BF16>(a, xfmt, parts, s);
  if (st != TFD_OK || topk <= 1) return st;
  return tfd_internal::topk_launch(a.logits, rows, n, a.ld_logits, topk, id_map, top_vals, top_ids,
                                   ldt, wl.submax, wl.part_max, parts_used, wl.topk_ws,
                                   wl.topk_bytes, s);
}

#if TFD_TRACE
// TFD_TRACE builds only (not part of the public header): the device buffer, [blocks][64] uint64,
// that the head GEMV kernel writes its phase stamps into; NULL stops the recording.
extern "C" void tfd_trace_set(void* dev_buf) { g_trace = reinterpret_cast<uint64_t*>(dev_buf); }
#endif
