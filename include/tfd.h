/*
 * tfd.h - C ABI of the GB300 (sm_103a) draft-head decode step library, libtfd.so.
 *
 * The library computes the per-round step of an EAGLE-style draft head in a speculative-decoding
 * server: a few-row (1..16 token rows) vocabulary-head GEMV in bf16 or FP8 fused with a
 * split-vocabulary top-1 / top-k, the two-stage head (low-rank top-cand_k then exact rescore), the
 * qk_norm + RoPE ring-window attention, the accept-prefix count, and the FP8 quantisation of the
 * weights these calls read.
 *
 * Conventions shared by every call:
 *  - Pointers named as device buffers are caller-owned device memory on the current CUDA device.
 *    The library allocates nothing in a call and keeps no state between calls.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call only enqueues work
 *    on it and never synchronises; results are ready when the stream reaches them.
 *  - The return value reports host-side argument checks and launch errors. A call that fails a
 *    check returns its status and enqueues nothing.
 *  - Errors that depend on device data (an out-of-range candidate id, an asked count larger than
 *    the window, a negative position) never trap: the kernel skips the offending element and, when
 *    `dev_status` is not NULL, stores TFD_ERR_DEVICE_DATA there with an atomic compare-and-swap
 *    from 0 (the first error stays). The caller zeroes *dev_status before the call.
 *  - Matrices are row-major. Every device pointer must be 16-byte aligned (8-bit and 32-bit scale
 *    arrays: 4-byte aligned), and leading dimensions keep every row 16-byte aligned.
 *  - Top-k outputs are sorted by value descending, then id ascending. Values compare as floats
 *    (-0 == +0); NaN ranks below -inf. Returned values are canonical: -0 comes back as +0 and NaN
 *    as the quiet NaN 0x7FC00000.
 *  - Workspaces: a call that needs one takes `ws`/`ws_bytes` and a `*_workspace()` query returns
 *    the bytes it needs. A workspace holds arrival counters that must start at zero: zero-fill it
 *    once before its first use; every call that completes leaves those counters at zero again.
 *    Two calls that may run at the same time need separate workspaces.
 *
 * Citations name the source page and its section:
 *  [TFE]    "dsv41 Zig: the TFE draft head (TF_DS_DRAFTER=eagle), off by default" (#42)
 *  [DSPARK] "dsv41 metal: the DSpark drafter on an FP8 head, a concurrent propose and resident
 *           buffers" (#3296)
 *  [SUBSET] "nemotron: Super's MTP drafts on the draft vocabulary's FP8 rows ..." (#1011)
 */
#ifndef TFD_H_
#define TFD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TFD_OK = 0,
  TFD_ERR_INVALID = 1,      /* an argument is out of range, NULL, misaligned or aliased */
  TFD_ERR_UNSUPPORTED = 2,  /* valid, but outside what this build implements (e.g. dim != 128) */
  TFD_ERR_WORKSPACE = 3,    /* ws is NULL or ws_bytes is below the *_workspace() size */
  TFD_ERR_CUDA = 4,         /* the CUDA runtime reported an error at launch */
  TFD_ERR_DEVICE_DATA = 5,  /* (device status only) bad ids, counts or positions in device data */
  TFD_ERR_TIMEOUT = 6       /* (device status only) a bounded device wait gave up */
} tfd_status;

/*
 * Weight formats. TFD_W_FP8_BLOCK32_IL holds the same codes and scales as TFD_W_FP8_BLOCK32 with
 * the codes of each row reordered in steps of 64 columns (k % 64 == 0): within step c, bytes
 * 64c + 16t + 8b + e (t = 0..3, b = 0..1, e = 0..7) hold the code of column 64c + 32b + 8t + e,
 * so the 8 codes a GEMV thread takes from each of a step's two 32-wide blocks are one 16-byte
 * load. It is this library's own layout (no counterpart on the pages); tfd_quant_fp8 writes it and
 * tfd_fp8_block32_relayout converts to and from the plain row-major layout.
 */
typedef enum {
  TFD_W_BF16 = 0,
  TFD_W_FP8_ROW = 1,
  TFD_W_FP8_BLOCK32 = 2,
  TFD_W_FP8_BLOCK32_IL = 3
} tfd_wfmt;
/*
 * Activation formats. TFD_X_BF16_E4M3 (FP8 weights only, W8A8): bf16 activations quantised per
 * row inside the call by the weights' row rule, s_r = fl32(amax_r / 448), code = e4m3_rne_sat(
 * fl32(x / s_r)) (a zero row keeps its zeros), and multiplied on the E4M3 tensor-core path; the
 * result is acc * s_r (* the weights' scales) with fp32 accumulation.
 */
typedef enum { TFD_X_BF16 = 0, TFD_X_F32 = 1, TFD_X_BF16_E4M3 = 2 } tfd_xfmt;
typedef enum { TFD_OUT_NONE = 0, TFD_OUT_F32 = 1, TFD_OUT_BF16 = 2, TFD_OUT_ADD_BF16 = 3 } tfd_out;

/* Limits from the pages' statement of the problem. */
/* [TFE] commit "pass kernels and FP8 linears": GEMV for up to 16 rows; windows of up to 32 rows
 * (rows 17-32 take k split over a thread-block cluster where one block's shared memory is too
 * small for the activation tile; fp32 activations stop at 16 rows). */
#define TFD_MAX_ROWS 32
#define TFD_MAX_TOPK 512    /* [TFE] commit "... ocabulary head": cand_k from 1 to 512 */
#define TFD_MAX_WINDOW 511  /* [TFE] commit "... ocabulary head": window up to 511 (512 keys) */

/* A static string naming a status. Never NULL. */
const char* tfd_status_string(int status);

/* Library version (major * 10000 + minor * 100 + patch). */
int tfd_version(void);

/*
 * tfd_quant_fp8 - FP8 E4M3 codes of a bf16 weight W[n][k].
 *   mode TFD_W_FP8_ROW: per row s_n = fl32(amax_n / 448); code = e4m3_rne_sat(fl32(w / s_n)).
 *     [TFE] update "main3x heads, pass kernels, FP8 linears": "scale = row absmax / 448, round to
 *     nearest even, from the bf16 weight". A zero row gets s = 0 and keeps its (signed) zeros.
 *   mode TFD_W_FP8_BLOCK32: per 32x32 block, byte = clamp(e + 127, 0, 254) where 2^e is the
 *     smallest power of two with amax <= 448 * 2^e (an all-zero block stores 0); code =
 *     e4m3_rne_sat(w * 2^-(byte - 127)). [DSPARK] "FP8 draft head": E4M3 codes with E8M0 scales in
 *     32x32 blocks.
 *   mode TFD_W_FP8_BLOCK32_IL: the codes and scales of TFD_W_FP8_BLOCK32, codes written in the
 *     interleaved layout described at tfd_wfmt (k % 64 == 0).
 *   E4M3 is the "fn" form (bias 7, max 448, 0x7F = NaN); encoding is round-to-nearest-even with
 *   saturation to +-448. Weights must be finite.
 * Args:
 *   w_bf16  device, bf16 [n][k] (row stride k).
 *   n, k    n >= 1, k >= 16 and k % 16 == 0; BLOCK32 also needs n % 32 == 0 and k % 32 == 0.
 *   codes   device, uint8 [n][k] (written).
 *   scales  device, ROW: float [n]; BLOCK32: uint8 [n/32][k/32] (written).
 */
tfd_status tfd_quant_fp8(const void* w_bf16, int64_t n, int64_t k, int mode, uint8_t* codes,
                         void* scales, void* stream);

/*
 * tfd_head_gemv - few-row head GEMV acc[r][i] = sum_j W[i][j] * x[r][j] with fp32 accumulation,
 * optional output, and an optional fused top-k over the n outputs of each row.
 *   [TFE] commit "pass kernels and FP8 linears": GEMV over bf16 and e4m3 weights for up to 16 rows
 *   (out bf16, fp32, or added to bf16); the top-1 of a vocabulary row in parts and a join.
 *   [DSPARK] "FP8 draft head": the drafter keeps its top 64 candidates.
 *   FP8 forms keep activations in bf16/fp32 (W8A16): ROW acc = s_i * sum dec(c) x;
 *   BLOCK32 acc = sum over 32-wide k blocks of 2^(byte-127) * (sum dec(c) x).
 * Args:
 *   w        device: bf16 [n][k], or uint8 codes [n][k] for the FP8 forms.
 *   wfmt     tfd_wfmt.
 *   w_scales device: FP8_ROW float [n]; FP8_BLOCK32 uint8 [n/32][k/32]; NULL for bf16.
 *   n, k     outputs per row (>= 1) and reduction length (k >= 16, k % 16 == 0; BLOCK32 also
 *            n % 32 == 0 and k % 32 == 0).
 *   x        device: bf16 or float (xfmt) [rows][ldx], ldx >= k. Float activations are used at
 *            full fp32 precision; TFD_X_BF16_E4M3 (FP8 weights only) quantises bf16 rows to E4M3
 *            first (W8A8, see tfd_xfmt).
 *   rows     1..32 (fp32 activations 1..16). Rows 17-32 go past this page's 16: the subset
 *            page (#1011) runs decode windows of 17 to 32 rows on wider kernels.
 *   out_mode NONE: no output; F32: y float [rows][ldy] = fl32(acc); BF16: y bf16 = bf16(fl32(acc));
 *            ADD_BF16: y bf16 is read as the residual and overwritten with bf16(res + acc), which
 *            may share memory with nothing else read by the call (in place is allowed).
 *   ldy      >= n when out_mode != NONE.
 *   topk     0 = none, else 1..512 (<= n): top_vals/top_ids [rows][ldt] receive the top-k of
 *            each row's fp32 acc (the FP8_ROW scale and BLOCK32 scales applied).
 *   ldt      row stride of top_vals/top_ids (0 = topk; else >= topk), so that the top-1 of each
 *            step of a multi-step pass can land in one column of a [streams][steps] array.
 *   top1_conf device float [rows] or NULL; only with topk == 1: the top-1 "with confidence"
 *            ([TFE] "What this changes": row kernels ... top-1 with confidence), read as the
 *            softmax probability of the pick, 1 / sum_i exp(acc_i - max acc) over the row's n
 *            outputs (NaN and -inf outputs add nothing; a row of only those gives NaN).
 *   parts    the row is scanned in `parts` contiguous ranges whose partial top-k are then joined;
 *            0 = the library's choice. The result does not depend on it.
 *   id_map   device int32 [n] or NULL: the id reported (and compared on ties) for output i is
 *            id_map[i] instead of i (a candidate list or a subset vocabulary, [SUBSET]).
 *   ws       device workspace of tfd_head_gemv_workspace(rows, n, topk, parts) bytes (may be 0).
 *   dev_status device int32 or NULL. A matrix split over a cluster of two blocks (few 64-row
 *            groups, or 17-32 rows of a 4096-wide matrix) exchanges partial sums through bounded
 *            waits; one that gives up (after about a second) stores TFD_ERR_TIMEOUT there and the
 *            call's outputs are then undefined. No other device-data errors exist in this call.
 * Refused: rows outside 1..32 (1..16 for fp32 activations); topk > 512 or > n; x aliasing y; NULL or misaligned pointers;
 *   rows * k too large for the activation tile (TFD_ERR_UNSUPPORTED, see tfd_head_gemv_max_k).
 */
size_t tfd_head_gemv_workspace(int rows, int64_t n, int topk, int parts);
int64_t tfd_head_gemv_max_k(int rows, int xfmt);
tfd_status tfd_head_gemv(const void* w, int wfmt, const void* w_scales, int64_t n, int64_t k,
                         const void* x, int xfmt, int rows, int64_t ldx, int out_mode, void* y,
                         int64_t ldy, int topk, int parts, const int32_t* id_map, float* top_vals,
                         int32_t* top_ids, int64_t ldt, float* top1_conf, void* ws,
                         size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * tfd_head_gemv_noalloc - tfd_head_gemv without a caller workspace, for callers that cannot
 * allocate device memory: serving loops that keep allocator calls off the hot path because
 * cudaMalloc can block or synchronise the whole device in the middle of a decode round, and plugins
 * whose host framework owns all device memory and offers them no allocator.
 *   The pages have no counterpart of this entry point; it is an addition of this library.
 *   Same arguments and results as tfd_head_gemv, minus ws/ws_bytes. The scratch is a fixed device
 *   array of TFD_NOALLOC_SCRATCH_BYTES inside the library, held by every GPU that loads it until
 *   the process exits. A call whose tfd_head_gemv_workspace() size exceeds it returns
 *   TFD_ERR_WORKSPACE and enqueues nothing (top-1 calls always fit; a top-k > 1 call fits only when
 *   its fp32 logits and top-k lists do, i.e. for small n).
 *   The first call on a device looks the array's device address up (once per device, with that
 *   device current; a failed lookup is retried by the next call); make that first call before any
 *   stream capture. Each call clears the part of
 *   the array it uses on `stream` before the GEMV (so a call that then fails an argument check has
 *   already enqueued that clear, which touches only the library's own array). Every call shares
 *   the one array: calls whose work overlaps on the GPU (other streams, other threads) race and
 *   must be serialised by the caller. It calls no cudaMalloc, cudaFree or allocating library.
 */
#define TFD_NOALLOC_SCRATCH_BYTES 1048576
tfd_status tfd_head_gemv_noalloc(const void* w, int wfmt, const void* w_scales, int64_t n,
                                 int64_t k, const void* x, int xfmt, int rows, int64_t ldx,
                                 int out_mode, void* y, int64_t ldy, int topk, int parts,
                                 const int32_t* id_map, float* top_vals, int32_t* top_ids,
                                 int64_t ldt, float* top1_conf, int32_t* dev_status,
                                 void* stream);

/*
 * tfd_topk - top-k of given fp32 logits, ties to the lower (mapped) id; values and ids bit-exact.
 *   [TFE] commit "... ocabulary head": "the top cand_k low-rank logits (fp32, a tie at the k-th
 *   value by the lower token id)", cand_k 1 to 512; "the top-1 kernel through an id map".
 * Args:
 *   logits device float [rows][ld], ld >= n. rows >= 1, n >= 1, 1 <= k <= min(n, 512).
 *   id_map device int32 [n] or NULL (as in tfd_head_gemv).
 *   vals, ids device [rows][k] (written).
 *   ws     device workspace of tfd_topk_workspace(rows, n, k) bytes.
 */
size_t tfd_topk_workspace(int rows, int64_t n, int k);
tfd_status tfd_topk(const float* logits, int rows, int64_t n, int64_t ld, int k,
                    const int32_t* id_map, float* vals, int32_t* ids, void* ws, size_t ws_bytes,
                    void* stream);

/*
 * tfd_rescore - exact logits of each row's candidates from a dense bf16 head, and their argmax.
 *   [TFE] commit "... ocabulary head": the two_stage head drafts "the argmax of their exact logits
 *   from the target's own head, a dense bf16 copy".
 *   e[r][j] = fl32(W_exact[cand[r][j]] . x[r]) with fp32 accumulation; out_ids[r] = the candidate
 *   with the largest e (ties to the lower id). A candidate outside [0, vocab) gets e = NaN (it
 *   ranks last) and sets TFD_ERR_DEVICE_DATA.
 * Args:
 *   w_exact_bf16 device bf16 [vocab][k]; k >= 16, k % 16 == 0.
 *   x_bf16   device bf16 [rows][k]; rows 1..32.
 *   cand     device int32 [rows][cand_k]; cand_k 1..512.
 *   cand_logits device float [rows][cand_k] or NULL.
 *   out_ids  device int32 [rows]; out_vals device float [rows] or NULL.
 *   ws       device workspace of tfd_rescore_workspace(rows, cand_k) bytes.
 */
size_t tfd_rescore_workspace(int rows, int cand_k);
tfd_status tfd_rescore(const void* w_exact_bf16, int64_t vocab, int64_t k, const void* x_bf16,
                       int rows, const int32_t* cand, int cand_k, float* cand_logits,
                       int32_t* out_ids, float* out_vals, void* ws, size_t ws_bytes,
                       int32_t* dev_status, void* stream);

/*
 * tfd_window_attn - one decode position per stream: qk_norm, RoPE, ring write, window attention.
 *   [TFE] commit "... ocabulary head": qk_norm is an RMSNorm on each query and key head before
 *   RoPE; the window goes up to 511 (512 keys). Commit "pass kernels and FP8 linears": single-query
 *   attention over the window in one block. First commits: the head's rows live in a ring.
 *   Per stream s at position p = pos[s] and head h:
 *     q' = rope(rmsnorm(q) * q_gamma, p) (fp32); k' = bf16(rope(rmsnorm(k_new) * k_gamma, p));
 *     k_ring[s][p % ring][h] = k'; v_ring[s][p % ring][h] = v_new;
 *     out[s][h*dim..] = bf16(softmax_j(q' . k_j / sqrt(dim)) . v_j) over positions
 *     j = max(0, p - window) .. p read from the ring.
 *   rmsnorm(v) = v / sqrt(mean(v^2) + eps); RoPE pairs element i with i + dim/2 and turns the pair
 *   by p * rope_base^(-2i/dim). Ring slots of earlier positions must hold their keys and values.
 * Args:
 *   q, k_new, v_new device bf16 [streams][heads][dim]; q_gamma, k_gamma device bf16 [dim] or NULL
 *   (ones); pos device int32 [streams] (a negative position sets TFD_ERR_DEVICE_DATA and that
 *   stream's output is left unwritten); k_ring, v_ring device bf16 [streams][ring][heads][dim];
 *   ring >= window + 1; window 0..511; dim == 128; out device bf16 [streams][heads*dim].
 */
tfd_status tfd_window_attn(const void* q, const void* k_new, const void* v_new,
                           const void* q_gamma, const void* k_gamma, float eps, float rope_base,
                           const int32_t* pos, void* k_ring, void* v_ring, int ring, int window,
                           int streams, int heads, int dim, void* out, int32_t* dev_status,
                           void* stream);

/*
 * tfd_accept - accept-prefix count of a verify round.
 *   [TFE] commit "... rnel test TF_DS_ACCEPT_LOG=N": a draft is kept when it and every earlier
 *   draft equal the round's draws; the log counts drafts asked and kept at each window position.
 *   n_kept[s] = the largest m <= n_asked[s] with drafts[s][i] == draws[s][i] for all i < m.
 *   asked_hist[i] += (i < n_asked[s]) and kept_hist[i] += (i < n_kept[s]) over the streams.
 *   An n_asked outside [0, win] sets TFD_ERR_DEVICE_DATA; that stream keeps 0 and adds nothing.
 * Args:
 *   drafts, draws device int32 [streams][win]; n_asked device int32 [streams]; streams >= 1;
 *   win 1..512; n_kept device int32 [streams]; asked_hist, kept_hist device int64 [win] or NULL
 *   (both or neither), accumulated.
 */
tfd_status tfd_accept(const int32_t* drafts, const int32_t* n_asked, const int32_t* draws,
                      int streams, int win, int32_t* n_kept, int64_t* asked_hist,
                      int64_t* kept_hist, int32_t* dev_status, void* stream);

/*
 * tfd_fp8_block32_relayout - block-32 FP8 codes between the plain row-major layout and the
 *   interleaved layout of TFD_W_FP8_BLOCK32_IL (a permutation of bytes within each row; the
 *   scales are unchanged). No counterpart on the pages: it serves codes made elsewhere.
 * Args:
 *   in, out device uint8 [n][k], not overlapping; n >= 1; k >= 64 and k % 64 == 0; 16-byte
 *   aligned. to_interleaved: 1 plain -> interleaved, 0 interleaved -> plain.
 */
tfd_status tfd_fp8_block32_relayout(const uint8_t* in, int64_t n, int64_t k, int to_interleaved,
                                    uint8_t* out, void* stream);

/*
 * tfd_rmsnorm - RMSNorm of hidden rows.
 *   [TFE] eagle.cu's row kernels include RMSNorm; qk_norm is the same normalisation per head.
 *   out[r][i] = bf16(x[r][i] / sqrt(mean_i(x[r][i]^2) + eps) * gamma[i]), sums in fp32.
 * Args:
 *   x device bf16 [rows][ldx]; out device bf16 [rows][ldo] (may equal x: in place);
 *   gamma device bf16 [hidden] or NULL (ones); rows >= 1; hidden >= 8 and hidden % 8 == 0;
 *   ldx, ldo >= hidden and multiples of 8; eps >= 0; x, out, gamma 16-byte aligned.
 */
tfd_status tfd_rmsnorm(const void* x, int64_t ldx, const void* gamma, float eps, int rows,
                       int64_t hidden, void* out, int64_t ldo, void* stream);

/*
 * tfd_swiglu - SwiGLU of a gate and an up row, SiLU rounded to bf16 before the multiply.
 *   [TFE] the reference "rounds SiLU(g) to bf16 before the multiply", as the silu-mul row kernel
 *   does. out = bf16(bf16(SiLU(g)) * u), SiLU(g) = g / (1 + exp(-g)) in fp32.
 * Args:
 *   g, u device bf16 [rows][ld]; out device bf16 [rows][ldo] (may equal g or u); rows >= 1;
 *   cols >= 8 and cols % 8 == 0; ld, ldo >= cols and multiples of 8; 16-byte aligned.
 */
tfd_status tfd_swiglu(const void* g, const void* u, int64_t ld, int rows, int64_t cols, void* out,
                      int64_t ldo, void* stream);

/*
 * tfd_absorb - write a span of key/value rows into each stream's ring (a prompt chunk or a round).
 *   [TFE] first commits: an absorb of more rows than the ring wrote two rows to one ring row, and
 *   "absorb refuses a larger span"; commit "... ocabulary head": qk_norm before RoPE, and a prompt
 *   chunk gives the head its last ring of rows.
 *   For stream s and row i < n at position p = p0[s] + i:
 *     k_ring[s][p % ring][h] = bf16(rope(rmsnorm(k_rows[s][i][h]) * k_gamma, p));
 *     v_ring[s][p % ring][h] = v_rows[s][i][h];
 *   with the normalisation and rotation of tfd_window_attn.
 * Args:
 *   k_rows, v_rows device bf16 [streams][n][heads][dim]; k_gamma device bf16 [dim] or NULL;
 *   p0 device int32 [streams] (negative, or p0 + n past INT32_MAX: TFD_ERR_DEVICE_DATA and that
 *   stream is left unwritten); 1 <= n <= ring (a longer span is refused with TFD_ERR_INVALID);
 *   k_ring, v_ring device bf16 [streams][ring][heads][dim]; dim == 128.
 */
tfd_status tfd_absorb(const void* k_rows, const void* v_rows, const void* k_gamma, float eps,
                      float rope_base, const int32_t* p0, int n, void* k_ring, void* v_ring,
                      int ring, int streams, int heads, int dim, int32_t* dev_status,
                      void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TFD_H_ */
