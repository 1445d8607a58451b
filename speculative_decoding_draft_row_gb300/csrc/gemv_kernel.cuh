// gemv_kernel.cuh - the few-row vocabulary-head GEMV kernel (bf16, FP8 row-scaled, FP8
// 32x32-block-scaled weights) fused with the output modes and a split-vocabulary top-1, and its
// launchers. Each weight format's kernels are instantiated in a translation unit of their own
// (gemv_w*.cu) so they compile in parallel; gemv.cu holds the C entry points.
//
// Follows the TFE draft head page (#42), commit "pass kernels and FP8 linears": GEMV over bf16 and
// e4m3 weights for up to 16 rows, out bf16 / fp32 / added to bf16, and the top-1 of a vocabulary
// row in parts and a join; the DSpark FP8 head page (#3296), "FP8 draft head": E4M3 codes with
// E8M0 scales in 32x32 blocks, the drafter's top 64 candidates.
//
// Design (GB300, HBM-bound): a 1..32-row GEMV reads every weight byte once, so the kernel is a
// weight stream. Each block is persistent and owns a contiguous range of 64-row groups (one
// "part" of the vocabulary). Its 16 warps split a group as 4 row tiles x 4 k slices; every warp
// streams its 16 rows x k-slice straight from HBM into registers with 16-byte (FP8 block form:
// 8-byte) non-allocating loads kept D steps ahead, and feeds them to warp-level bf16 tensor-core
// MMAs (m16n8k16, fp32 accumulate) whose other operand is the activation tile held in shared
// memory in fragment order (conflict-free 16-byte reads). The MMA removes the per-element FMA
// work that would otherwise cap the CUDA cores at 10-16 rows; FP8 codes are widened to f16 in
// registers (exact), against activations scaled by a power of two into f16 range. The k order
// inside a dot product is permuted consistently between weights and activations so that each
// thread's 16 contiguous bytes are one MMA operand chunk. Weight loads carry an L2 evict-first
// policy, and each block's first group is prefetched into L2 while the activations are staged.
// Per group, the four k-slice partials are summed in a fixed order in shared memory, so every
// output's arithmetic is independent of its index and of the part count.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace tfd_gemv {

// Weight loads kept in flight per warp, in steps, for one and two n-tiles (tuning macros); the
// FP8 forms have their own two-n-tile depth (their decode needs more registers).
#ifndef TFD_GEMV_DEPTH_NT1
#define TFD_GEMV_DEPTH_NT1 4
#endif
#ifndef TFD_GEMV_DEPTH_NT2
#define TFD_GEMV_DEPTH_NT2 8
#endif
#ifndef TFD_GEMV_DEPTH_FP8_NT1
#define TFD_GEMV_DEPTH_FP8_NT1 4
#endif
#ifndef TFD_GEMV_DEPTH_FP8_NT2
#define TFD_GEMV_DEPTH_FP8_NT2 8
#endif
#ifndef TFD_GEMV_DEPTH_BLK_NT2
#define TFD_GEMV_DEPTH_BLK_NT2 4
#endif
#ifndef TFD_GEMV_DEPTH_BLKIL_NT2
#define TFD_GEMV_DEPTH_BLKIL_NT2 4
#endif
// Bytes of a block's first group fetched into L2 while the activations are staged, and the
// number of threads that share the request.
#ifndef TFD_GEMV_PREFETCH
#define TFD_GEMV_PREFETCH 262144
#endif
constexpr int kPrefetchParts = 8;
// Minimum resident blocks per SM asked of the compiler for one n-tile (2 caps registers at 64).
#ifndef TFD_GEMV_MINB_NT1
#define TFD_GEMV_MINB_NT1 1
#endif
// fp32 activations take three planes of MMA operands; their two-n-tile form keeps a shallower ring
#ifndef TFD_GEMV_DEPTH_X32_NT2
#define TFD_GEMV_DEPTH_X32_NT2 4
#endif
// W8A8 with two n-tiles
#ifndef TFD_GEMV_DEPTH_AQ_NT2
#define TFD_GEMV_DEPTH_AQ_NT2 4
#endif
// Fast path for 4096-wide weights (the pages' hidden size) with 4 k-slices and no cluster split:
// each k-slice's steps fully unrolled, every weight and activation address a base plus an
// immediate, the ring's refills following statically into the next group, and no per-step range
// checks (a block takes it when all of its groups lie inside the matrix).
#ifndef TFD_GEMV_FAST
#define TFD_GEMV_FAST 1
#endif
// 4096-wide activations staged with constant geometry by their own instantiation (1), or by the
// general staging loop (0).
#ifndef TFD_GEMV_STAGE4K
#define TFD_GEMV_STAGE4K 1
#endif
// CUDA-core form of the bf16 x bf16 step (off by default): the same operands, multiplied with
// fp32 FMAs instead of tensor-core MMAs. It exists to measure whether the tensor cores pay at this
// row count; the library is built with it only for that measurement.
#ifndef TFD_GEMV_FFMA
#define TFD_GEMV_FFMA 0
#endif
// four n-tiles (17-32 rows)
#ifndef TFD_GEMV_DEPTH_NT4
#define TFD_GEMV_DEPTH_NT4 4
#endif
#ifndef TFD_GEMV_DEPTH_BLK_NT4
#define TFD_GEMV_DEPTH_BLK_NT4 2
#endif
template <int WF, int NT, int XF = TFD_X_BF16>
constexpr int gemv_depth() {
  return NT == 4 ? ((WF == TFD_W_FP8_BLOCK32 || WF == TFD_W_FP8_BLOCK32_IL) ? TFD_GEMV_DEPTH_BLK_NT4
                                                                            : TFD_GEMV_DEPTH_NT4)
       : (XF == TFD_X_F32 && NT == 2) ? TFD_GEMV_DEPTH_X32_NT2
       : (XF == TFD_X_BF16_E4M3 && NT == 2 && WF == TFD_W_FP8_ROW) ? TFD_GEMV_DEPTH_AQ_NT2
       : WF == TFD_W_BF16 ? (NT == 1 ? TFD_GEMV_DEPTH_NT1 : TFD_GEMV_DEPTH_NT2)
       : WF == TFD_W_FP8_ROW ? (NT == 1 ? TFD_GEMV_DEPTH_FP8_NT1 : TFD_GEMV_DEPTH_FP8_NT2)
       : WF == TFD_W_FP8_BLOCK32_IL ? (NT == 1 ? TFD_GEMV_DEPTH_FP8_NT1 : TFD_GEMV_DEPTH_BLKIL_NT2)
                             : (NT == 1 ? TFD_GEMV_DEPTH_FP8_NT1 : TFD_GEMV_DEPTH_BLK_NT2);
}

using namespace tfd;

constexpr int kThreads = 512;
constexpr int kWarps = 16;
constexpr int kMaxParts = 1024;
constexpr int kMaxRowsPad = 32;  // activation rows a call takes (four n-tiles of 8)

template <int WF>
struct WTraits;
template <>
struct WTraits<TFD_W_BF16> {  // 8 bf16 per thread-row load (16 B)
  static constexpr int E = 8, WORDS = 4, ELEM_BYTES = 2;
};
template <>
struct WTraits<TFD_W_FP8_ROW> {  // 16 codes per thread-row load (16 B)
  static constexpr int E = 16, WORDS = 4, ELEM_BYTES = 1;
};
template <>
struct WTraits<TFD_W_FP8_BLOCK32_IL> {  // the same 2 x 8 codes, one 16-byte load (interleaved)
  static constexpr int E = 16, WORDS = 4, ELEM_BYTES = 1;
};
template <>
struct WTraits<TFD_W_FP8_BLOCK32> {  // 2 x 8 codes: 8 from each of the step's two 32-wide blocks
  static constexpr int E = 16, WORDS = 4, ELEM_BYTES = 1;
};

struct GemvArgs {
  const void* w;
  const void* scales;
  int64_t n, k;
  const void* x;
  int64_t ldx;
  int rows;
  int out_mode;
  void* y;
  int64_t ldy;
  int topk;
  const int32_t* id_map;
  float* logits;  // fp32 logits destination for topk > 1 (may equal y), else null
  int64_t ld_logits;
  uint32_t* submax;  // topk > 1: [rows][ceil(n / 16)] value key of each 16-row sub-group's max
  uint32_t* part_max;  // topk > 1: [parts][rows] value key of each part's largest output
  uint64_t* part_keys;  // [parts][rows]
  uint32_t* counter;
  float* top_vals;
  int32_t* top_ids;
  int64_t ldt;  // row stride of top_vals / top_ids
  float* top1_conf;  // [rows] softmax probability of the top-1, or null
  float2* part_ms;   // [parts][rows] per part (max, sum of exp(l - max)) for the confidence
  int parts;
  int64_t ngroups;
  int ssl;  // steps per k slice
  int csplit;  // blocks of a cluster splitting k (1: no cluster); parts counts clusters
  int* parts_used;  // host only (never read by the kernel): the launcher stores the part count
  uint64_t* trace;  // TFD_TRACE builds: [blocks][kTraceSlots] phase stamps, or null
  uint32_t* queue;  // group queue counter (zero between calls), or null for a static split
  int32_t* status;  // device status (TFD_ERR_TIMEOUT from a bounded wait), or null
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A B (a zero accumulator input): starts a block's partial sum without zeroing registers.
__device__ __forceinline__ void mma_f16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1,
                                                uint32_t a2, uint32_t a3, uint32_t b0,
                                                uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// d = A B for E4M3 operands (k = 32), fp32 accumulators starting at zero.
__device__ __forceinline__ void mma_e4m3_16832_z(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// The same MMA accumulating into d (row-scaled codes: no per-block scale between the MMAs).
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> two E4M3 codes (byte 0 = lo, byte 1 = hi), RNE, saturating to +-448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four E4M3 codes -> two f16x2 words (codes 0,1 and codes 2,3). Every E4M3 value is an f16 value,
// so the hardware conversion is exact; one instruction widens two codes.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(v));
}

__device__ __forceinline__ uint16_t f32_to_f16_bits(float f) {
  return __half_as_ushort(__float2half_rn(f));
}
__device__ __forceinline__ float f16_bits_to_f32(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

// Merge of two online-softmax states (max, sum of exp(v - max)).
__device__ __forceinline__ float2 ms_merge(float2 a, float2 b) {
  const float m = fmaxf(a.x, b.x);
  if (m == -INFINITY) return make_float2(-INFINITY, 0.0f);
  return make_float2(m, a.y * expf(a.x - m) + b.y * expf(b.x - m));
}

__device__ __forceinline__ float e8m0_scale(uint32_t byte) {
  return byte == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(byte << 23);
}

// ---- shared-memory barriers of the two-block partial exchange ----
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// The address of this block's shared-memory word `p` in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
// Waits for the phase of parity `par` of a local mbarrier to complete (acquire, cluster scope).
// Gives up after about a second of global time: false, and the caller reports TFD_ERR_TIMEOUT.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t par) {
  const uint32_t ba = smem_addr(bar);
  uint32_t ok;
  uint64_t t0 = 0;
  for (int it = 0;; ++it) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(ba), "r"(par)
        : "memory");
    if (ok) return true;
    uint64_t now;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
    if (it == 0) t0 = now;
    else if (now - t0 > 1000000000ull) return false;
  }
}
// One float4 into block 0's shared memory (cluster address `dst`), counted as 16 bytes of the
// transaction of the mbarrier at cluster address `bar` there. The write needs no fence of its
// own: the barrier's phase completes only once the bytes have landed.
__device__ __forceinline__ void st_async_f4(uint32_t dst, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
      ::"r"(dst), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}

template <int WF>
struct WLoad {
  uint32_t r[2][WTraits<WF>::WORDS];  // rows g and g + 8
  uint32_t scb;                       // the step's two E8M0 scale bytes (FP8_BLOCK32): A | B << 8
};

// An fp32 value split into three parts of the MMA operand type (bf16 for bf16 weights, f16 for
// FP8 weights): hi + mid + lo carries every bit of a normal fp32 value.
template <bool F16>
__device__ __forceinline__ void split3(float v, uint16_t& h0, uint16_t& h1, uint16_t& h2) {
  if (F16) {
    h0 = f32_to_f16_bits(v);
    float r1 = v - f16_bits_to_f32(h0);
    h1 = f32_to_f16_bits(r1);
    float r2 = r1 - f16_bits_to_f32(h1);
    h2 = f32_to_f16_bits(r2);
  } else {
    h0 = f32_to_bf16_bits(v);
    float r1 = v - bf16_bits_to_f32(h0);
    h1 = f32_to_bf16_bits(r1);
    float r2 = r1 - bf16_bits_to_f32(h1);
    h2 = f32_to_bf16_bits(r2);
  }
}

// KSL = k-slices per block: 4 (16 warps = 4 row tiles x 4 k-slices, 64-row groups) or 1 (16 row
// tiles over the whole k range, 256-row groups: for short k, where 4 slices would leave each warp
// only a step or two per group).
template <int WF, int XF, int NT, int KSL = 4>
struct Layout {
  static constexpr int E = WTraits<WF>::E;
  static constexpr bool AQ = XF == TFD_X_BF16_E4M3;  // activations as E4M3 codes (W8A8)
  static constexpr int H = AQ ? 1 : E / 8;           // 16-byte x chunks per (step, nt) per lane
  static constexpr int PL = XF == TFD_X_F32 ? 3 : 1; // activation planes
  static constexpr int MT = 16 / KSL;                // row tiles per block
  __host__ __device__ static size_t x_bytes(int ssl) {
    return (size_t)PL * KSL * ssl * NT * H * 32 * 16;
  }
  __host__ __device__ static size_t red_bytes() {
    return KSL == 1 ? 0 : (size_t)2 * kWarps * NT * 32 * 16;
  }
  __host__ __device__ static size_t best_bytes() {
    // block best keys, join keys, per-row x max and x scale, block (max, sum) pairs, join pairs,
    // per-row part maxima
    return (size_t)MT * kMaxRowsPad * 8 + kMaxRowsPad * kWarps * 8 + 2 * kMaxRowsPad * 4 +
           MT * kMaxRowsPad * 8 + kMaxRowsPad * kWarps * 8 + kMaxRowsPad * 4;
  }
  // group partials of a block for its cluster leader, double-buffered, and (up to two n-tiles)
  // the leader's own partials of its last group (4 k-slices only)
  __host__ __device__ static size_t cpart_bytes() {
    return KSL == 1 ? 0 : (size_t)(NT == 4 ? 2 : 3) * 4 * NT * 32 * 16;
  }
  __host__ __device__ static size_t smem_bytes(int ssl) {
    return x_bytes(ssl) + red_bytes() + cpart_bytes() + best_bytes();
  }
};

// VAR: 0 the general form; 1 a 4096-wide matrix staged by one block (no cluster split) with bf16
// activations: constant staging geometry; 2 that, plus the unrolled check-free weight loop (n a
// multiple of the group rows); 3 the unrolled check-free weight loop of a 4096-wide matrix split
// over a cluster of two (a small matrix, e.g. the attention output projection); 4 the general form
// without a cluster split (none of the split's code, so fewer registers live). The host picks the
// instantiation.
template <int WF, int XF, int NT, int D, int KSL, int VAR = 0>
__global__ void __launch_bounds__(kThreads, NT == 1 ? TFD_GEMV_MINB_NT1 : 1)
gemv_kernel(const GemvArgs a) {
  constexpr bool FASTP = VAR == 2 || VAR == 3;
  constexpr int CSC = VAR == 3 ? 2 : 1;  // the cluster split the fast loop is built for
  using L = Layout<WF, XF, NT, KSL>;
  constexpr int MT = L::MT;
  constexpr int GR = 16 * MT;  // rows per group
  using T = WTraits<WF>;
  constexpr int E = T::E, H = L::H, PL = L::PL, EB = T::ELEM_BYTES;
  constexpr int MMAJ = E / 4;   // k16 MMAs per step per n-tile
  constexpr int STEPK = 4 * E;  // k elements per step (4 threads x E)
  extern __shared__ __align__(16) unsigned char smem[];
  const int ssl = a.ssl;
  const int spad = KSL * ssl;
  uint4* xs = reinterpret_cast<uint4*>(smem);
  float4* red = reinterpret_cast<float4*>(smem + L::x_bytes(ssl));
  float4* cpart = reinterpret_cast<float4*>(smem + L::x_bytes(ssl) + L::red_bytes());
  uint64_t* sbest =
      reinterpret_cast<uint64_t*>(smem + L::x_bytes(ssl) + L::red_bytes() + L::cpart_bytes());
  uint64_t* sjoin = sbest + MT * kMaxRowsPad;
  uint32_t* sxmax = reinterpret_cast<uint32_t*>(sjoin + kMaxRowsPad * kWarps);
  float* sxscale = reinterpret_cast<float*>(sxmax + kMaxRowsPad);
  float2* sms = reinterpret_cast<float2*>(sxscale + kMaxRowsPad);  // [MT][kMaxRowsPad]
  float2* sjms = sms + MT * kMaxRowsPad;                             // [kWarps][kMaxRowsPad]
  uint32_t* spmax = reinterpret_cast<uint32_t*>(sjms + kWarps * kMaxRowsPad);  // [kMaxRowsPad]
  __shared__ int is_last;
  __shared__ __align__(8) uint64_t s_full[2], s_empty[2];  // cluster split of two: the exchange
  // FP8 weights run f16 MMAs: each activation row is scaled by a power of two 2^-e_r into f16 range
  // (max |x| in [2^14, 2^15)), which keeps every bf16 activation exact down to 2^-32 of the row's
  // max; the epilogue multiplies by 2^e_r.
  constexpr bool F16 = WF != TFD_W_BF16;
  // W8A8: activations quantised per row to E4M3 here, E4M3 x E4M3 MMAs (k = 32)
  constexpr bool AQ = XF == TFD_X_BF16_E4M3;
  // block-32 scales (plain or interleaved codes): each step is two 32-wide blocks
  constexpr bool BLK = WF == TFD_W_FP8_BLOCK32 || WF == TFD_W_FP8_BLOCK32_IL;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int mt = warp % MT, ks = warp / MT;
  // trace slots: 0 entry, 1 activations staged, 2 + j end of the block's group j (up to 55),
  // 57/58/59 the 4096-wide staging's loads landed / row scales known / converted (general staging:
  // first barrier passed / chunks stored / converted), 60 the SM,
  // 61 groups done, 62 part keys written, 63 the join done (last block)
  TFD_STAMP(a.trace, 0);
#if TFD_TRACE
  if (a.trace != nullptr && tid == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    a.trace[(int64_t)blockIdx.x * kTraceSlots + 60] = smid;
  }
#endif
  // Split k over a cluster (small matrices, or 17-32 rows of a 4096-wide head): block crank of
  // cluster cid takes k-slices 4 crank .. 4 crank + 3 of every group of the cluster; the leader
  // (crank 0) sums the blocks' partials in rank order and runs the epilogue.
  namespace cg = cooperative_groups;
  const int csplit = (KSL == 1 || VAR == 1 || VAR == 2 || VAR == 4) ? 1 : VAR == 3 ? 2 : a.csplit;
  const int crank = csplit > 1 ? (int)cg::this_cluster().block_rank() : 0;
  const int cid = blockIdx.x / csplit;
  const int kstep0 = crank * KSL * ssl;  // first step of this block's k range
  const int64_t K = a.k, N = a.n;
  const int rows = a.rows;

  // ---- weight stream ----
  // With 4 k-slices a block owns whole 64-row groups. With one k-slice every warp owns whole dot
  // products, so the block owns a range of 16-row tiles [t_begin, t_end) instead (finer balance
  // across blocks: a 256-row group is a large share of a short-k part): warp mt takes tiles
  // t_begin + mt + 16 j, and "group" j starts at row_off + 256 j.
  const int64_t ntiles = (N + 15) / 16;
  const int64_t t_begin = KSL == 1 ? (int64_t)cid * ntiles / a.parts : 0;
  const int64_t t_end = KSL == 1 ? (int64_t)(cid + 1) * ntiles / a.parts : 0;
  const int64_t row_off = t_begin * 16;
  // The block's groups: with one k-slice, 0 .. g_end - 1 of its tile range; with 4 k-slices either
  // the static range g_begin .. g_end - 1, or (a queue in the workspace, no cluster split, more
  // than a ring's depth of steps per k-slice) group cid first and then the next unclaimed group
  // of a queue shared by all blocks (parts + the counter's old value), so faster blocks take more
  // groups and the blocks finish together. Group j of the sequence is published in s_q[j & 3]:
  // the claiming thread (lane 0 of the last warp, never a reducer of the group epilogue when a
  // queue is used, so the atomic's latency is off the critical path) claims groups 1 and 2
  // before the first barrier and group j + 3 just after the barrier that ends group j, which is
  // after every warp has read group j - 1's slot and before any needs group j + 3 (the ring
  // enters group j + 1 during group j).
  constexpr int64_t kNoGroup = (int64_t)1 << 40;
  const bool dyn = KSL == 4 && NT <= 2 && csplit == 1 && a.queue != nullptr &&
                   (ssl + D - 1) / D * D > D;
  const bool claimer = warp == kWarps - 1 && lane == 0;
  const int64_t g_begin = KSL == 1 ? 0 : dyn ? (int64_t)cid : (int64_t)cid * a.ngroups / a.parts;
  const int64_t g_end = KSL == 1 ? (t_end - t_begin + 15) / 16
                      : dyn ? a.ngroups : (int64_t)(cid + 1) * a.ngroups / a.parts;
  __shared__ int64_t s_q[4];
  auto claim = [&]() -> int64_t {
    const int64_t v = (int64_t)a.parts + (int64_t)atomicAdd(a.queue, 1u);
    return v < a.ngroups ? v : kNoGroup;
  };
  auto seq_group = [&](int j) -> int64_t {  // group j of this block's sequence, or kNoGroup
    if (KSL == 4 && dyn) return j == 0 ? ((int64_t)cid < a.ngroups ? (int64_t)cid : kNoGroup) : s_q[j & 3];
    return g_begin + j < g_end ? g_begin + j : kNoGroup;
  };
  auto tile_in = [&](int64_t gi, int tile) {  // the tile exists and is this block's
    return KSL == 1 ? gi < kNoGroup && t_begin + 16 * gi + tile < t_end : gi < a.ngroups;
  };
  const int s_loc = ks * ssl;              // the k-slice's first step in shared memory
  const int s_begin = kstep0 + s_loc;      // ... and in the row
  // The loop runs a multiple of D steps per group so the register ring stays in phase; steps past
  // the slice's own ssl are empty (no loads, zero weights).
  const int ssl_loop = (ssl + D - 1) / D * D;
  const unsigned char* wbase = reinterpret_cast<const unsigned char*>(a.w);
  const int64_t row_bytes = K * EB;
  const uint8_t* blk_scales = reinterpret_cast<const uint8_t*>(a.scales);
  const float* row_scales = reinterpret_cast<const float*>(a.scales);
  const int64_t kblocks = K >> 5;
  const bool sc16 = (kblocks & 1) == 0;  // a step's two scale bytes are 2-byte aligned

  // The thread's first element in a step: its 16 contiguous elements, or (block-32 form) its 8
  // elements of the step's first 32-wide block, the other 8 being 32 further on.
  const int toff = WF == TFD_W_FP8_BLOCK32 ? 8 * t : t * E;
  auto steps_below = [&](int64_t lim) -> int {  // steps s < ssl with (s_begin + s) * STEPK < lim
    int64_t v = lim > 0 ? (lim + STEPK - 1) / STEPK - s_begin : 0;
    return (int)(v < 0 ? 0 : (v > ssl ? ssl : v));
  };
  const int nvalid = steps_below(K - toff);
  const int nvalid_b = WF == TFD_W_FP8_BLOCK32 ? steps_below(K - 32 - toff) : nvalid;

  // Load state: group (and its place in the sequence), step, row pointer and row validity;
  // addresses advance by a constant.
  int ld_j = 0;
  int64_t ld_g = g_begin;
  int ld_s = 0;
  const unsigned char* lp = nullptr;
  const uint8_t* sp = nullptr;
  bool rv0 = false, rv1 = false, rvb = false;
  auto set_group = [&]() {
    const int64_t row = row_off + ld_g * GR + mt * 16 + g;
    const bool in = tile_in(ld_g, mt);
    rv0 = in && row < N;
    rv1 = in && row + 8 < N;
    lp = wbase + row * row_bytes + ((int64_t)s_begin * STEPK + toff) * EB;
    if (BLK) {
      const int64_t rblk = (row_off + ld_g * GR + mt * 16) >> 5;
      rvb = in && rblk * 32 < N;
      sp = blk_scales + rblk * kblocks + 2 * (int64_t)s_begin;
    }
  };
  set_group();
  const uint64_t wpol = l2_stream_policy();
  auto issue = [&](WLoad<WF>& b) {
    // the usual step: both rows and (block-32 form) both blocks in range, no zero fill
    const bool full = rv1 && ld_s < (WF == TFD_W_FP8_BLOCK32 ? nvalid_b : nvalid) &&
                      (!BLK || sc16);
    if (full) {
      if (WF == TFD_W_FP8_BLOCK32) {
        uint2 v = ldg_stream8(lp, wpol);
        b.r[0][0] = v.x; b.r[0][1] = v.y;
        v = ldg_stream8(lp + 32, wpol);
        b.r[0][2] = v.x; b.r[0][3] = v.y;
        v = ldg_stream8(lp + 8 * row_bytes, wpol);
        b.r[1][0] = v.x; b.r[1][1] = v.y;
        v = ldg_stream8(lp + 8 * row_bytes + 32, wpol);
        b.r[1][2] = v.x; b.r[1][3] = v.y;
        b.scb = __ldg(reinterpret_cast<const uint16_t*>(sp));
      } else {
        uint4 v = ldg_stream16(lp, wpol);
        b.r[0][0] = v.x; b.r[0][1] = v.y; b.r[0][2] = v.z; b.r[0][3] = v.w;
        v = ldg_stream16(lp + 8 * row_bytes, wpol);
        b.r[1][0] = v.x; b.r[1][1] = v.y; b.r[1][2] = v.z; b.r[1][3] = v.w;
        if (WF == TFD_W_FP8_BLOCK32_IL) b.scb = __ldg(reinterpret_cast<const uint16_t*>(sp));
      }
      lp += STEPK * EB;
      sp += 2;
      if (++ld_s == ssl_loop) { ld_s = 0; ld_g = seq_group(++ld_j); set_group(); }
      return;
    }
#pragma unroll
    for (int i = 0; i < T::WORDS; ++i) { b.r[0][i] = 0u; b.r[1][i] = 0u; }
    b.scb = 0u;
    if (ld_s < nvalid) {
      if (WF == TFD_W_FP8_BLOCK32) {
        const bool second = ld_s < nvalid_b;
        if (rv0) {
          uint2 v = ldg_stream8(lp, wpol);
          b.r[0][0] = v.x; b.r[0][1] = v.y;
          if (second) { v = ldg_stream8(lp + 32, wpol); b.r[0][2] = v.x; b.r[0][3] = v.y; }
        }
        if (rv1) {
          uint2 v = ldg_stream8(lp + 8 * row_bytes, wpol);
          b.r[1][0] = v.x; b.r[1][1] = v.y;
          if (second) { v = ldg_stream8(lp + 8 * row_bytes + 32, wpol); b.r[1][2] = v.x; b.r[1][3] = v.y; }
        }
        if (rvb) {
          if (sc16) b.scb = __ldg(reinterpret_cast<const uint16_t*>(sp));
          else b.scb = (uint32_t)__ldg(sp) | ((uint32_t)__ldg(sp + 1) << 8);
          if (!second) b.scb &= 0xFFu;
        }
      } else {
        if (rv0) {
          uint4 v = ldg_stream16(lp, wpol);
          b.r[0][0] = v.x; b.r[0][1] = v.y; b.r[0][2] = v.z; b.r[0][3] = v.w;
        }
        if (rv1) {
          uint4 v = ldg_stream16(lp + 8 * row_bytes, wpol);
          b.r[1][0] = v.x; b.r[1][1] = v.y; b.r[1][2] = v.z; b.r[1][3] = v.w;
        }
        // interleaved block-32 (k % 64 == 0): both blocks of a step are in range together
        if (WF == TFD_W_FP8_BLOCK32_IL && rvb) b.scb = __ldg(reinterpret_cast<const uint16_t*>(sp));
      }
    }
    lp += STEPK * EB;
    sp += 2;
    if (++ld_s == ssl_loop) { ld_s = 0; ld_g = seq_group(++ld_j); set_group(); }
  };

  // Fast path (the FASTP instantiations, chosen on the host): k == 4096, 4 k-slices, no cluster
  // split or a split of CSC blocks, n a multiple of the group rows.
  constexpr int FK = 4096;
  constexpr int SSLC = FK / (KSL * STEPK * CSC);  // steps per k-slice at k == FK
  constexpr bool FASTK = FASTP && KSL == 4 && SSLC >= D;
  constexpr int64_t FROWB = (int64_t)FK * EB;
  const bool fast = FASTK && g_begin < g_end;
  // this warp's first byte of group gi in the fast path, and its scale bytes (block-32 forms)
  auto fast_ptr = [&](int64_t gi) {
    return wbase + (gi * GR + mt * 16 + g) * FROWB + ((int64_t)s_begin * STEPK + toff) * EB;
  };
  auto fast_sp = [&](int64_t gi) {
    return blk_scales + ((gi * GR + mt * 16) >> 5) * (FK / 32) + 2 * (int64_t)s_begin;
  };
  auto fload = [&](WLoad<WF>& b, const unsigned char* q, const uint8_t* sq) {
    constexpr int64_t R8 = 8 * FROWB;  // row g + 8
    if (WF == TFD_W_FP8_BLOCK32) {
      uint2 v = ldg_stream8(q, wpol);
      b.r[0][0] = v.x; b.r[0][1] = v.y;
      v = ldg_stream8(q + 32, wpol);
      b.r[0][2] = v.x; b.r[0][3] = v.y;
      v = ldg_stream8(q + R8, wpol);
      b.r[1][0] = v.x; b.r[1][1] = v.y;
      v = ldg_stream8(q + R8 + 32, wpol);
      b.r[1][2] = v.x; b.r[1][3] = v.y;
    } else {
      uint4 v = ldg_stream16(q, wpol);
      b.r[0][0] = v.x; b.r[0][1] = v.y; b.r[0][2] = v.z; b.r[0][3] = v.w;
      v = ldg_stream16(q + R8, wpol);
      b.r[1][0] = v.x; b.r[1][1] = v.y; b.r[1][2] = v.z; b.r[1][3] = v.w;
    }
    if (BLK) b.scb = __ldg(reinterpret_cast<const uint16_t*>(sq));
    else b.scb = 0u;
  };

  // The first D steps of weights are in flight while the activations are staged.
  WLoad<WF> buf[D];
  auto prime = [&]() {
    if constexpr (FASTK) {
      if (fast) {
        const unsigned char* q = fast_ptr(g_begin);
        const uint8_t* sq = BLK ? fast_sp(g_begin) : nullptr;
#pragma unroll
        for (int i = 0; i < D; ++i) fload(buf[i], q + (int64_t)i * STEPK * EB, sq + 2 * i);
      }
    } else {
#pragma unroll
      for (int i = 0; i < D; ++i) issue(buf[i]);
    }
  };
  // The ring's first steps are issued before the activations are staged, except where the staging
  // keeps every row's chunk in registers (the 4096-wide form) and in a cluster split (small
  // matrices, whose staging is most of the call): there the activation loads go first, the L2
  // prefetch below covers the staging, and the ring follows it.
  constexpr bool PRIME_LATE = (VAR == 1 || VAR == 2) && XF == TFD_X_BF16 && !AQ && NT <= 2;
  if (!PRIME_LATE && csplit == 1) prime();
  // Staging the activations takes longer than the ring's loads (every block reads all rows, which
  // all blocks want at once); meanwhile the first TFD_GEMV_PREFETCH bytes of the block's first
  // group are fetched into L2, so the weight stream does not pause.
  auto l2_prefetch = [&]() {
  if (csplit > 1 && g_begin < g_end && tid < GR) {
    // this block's k range of each row of its first group, a row a thread
    const int64_t row = row_off + g_begin * GR + tid;
    const int64_t kb = (int64_t)kstep0 * STEPK;
    const int64_t kl = (int64_t)KSL * ssl * STEPK < K - kb ? (int64_t)KSL * ssl * STEPK : K - kb;
    if (row < N && kl > 0)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(wbase + row * row_bytes + kb * EB),
                   "r"((uint32_t)(kl * EB))
                   : "memory");
  }
  if (csplit == 1 && g_begin < g_end && tid < kPrefetchParts) {
    const int64_t row0 = row_off + g_begin * GR;
    const int64_t gbytes = (N - row0 < GR ? N - row0 : GR) * row_bytes;
    const int64_t pbytes = gbytes < (int64_t)TFD_GEMV_PREFETCH ? gbytes : (int64_t)TFD_GEMV_PREFETCH;
    const int64_t part = (pbytes / kPrefetchParts) & ~(int64_t)15;
    const int64_t off = tid * part;
    const int64_t len = tid == kPrefetchParts - 1 ? (pbytes & ~(int64_t)15) - off : part;
    if (len > 0)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(wbase + row0 * row_bytes + off),
                   "r"((uint32_t)len)
                   : "memory");
  }
  };
  // (the 4096-wide staging and a cluster split's staging issue their activation loads first, so
  // they are not queued behind this)
  if constexpr (VAR == 0 || !(XF == TFD_X_BF16 && !AQ && NT <= 2)) {
    if (csplit == 1) l2_prefetch();
  }

  for (int i = tid; i < MT * kMaxRowsPad; i += kThreads) sbest[i] = 0ull;
  if (csplit == 2) {
    // the exchange's barriers, initialised before either block of the pair can reach them (the
    // pair meets on the cluster barrier before its first group)
    if (tid == 0) {
      mbar_init(&s_full[0], 1);
      mbar_init(&s_full[1], 1);
      mbar_init(&s_empty[0], 4 * NT);
      mbar_init(&s_empty[1], 4 * NT);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  }
  if (tid < kMaxRowsPad) { sxmax[tid] = 0u; spmax[tid] = 0u; }
  if (dyn && claimer) {
    s_q[1] = claim();
    s_q[2] = claim();
  }
  __syncthreads();
  // bf16 activations for FP8 weights: the raw rows are staged in one pass that also takes each
  // row's max |x|; the power-of-two scaling into f16 is applied afterwards in shared memory.
  constexpr bool ONEPASS_C = F16 && XF == TFD_X_BF16 && !AQ;
  // 4096-wide bf16 activations staged whole by one block: 512 chunks of 8 a row, one per thread,
  // so thread tid owns k = 8 tid .. 8 tid + 7 of every row (constant geometry, every row's load in
  // flight at once, conversions in registers)
  constexpr bool STAGE4K_C = (VAR == 1 || VAR == 2) && XF == TFD_X_BF16 && !AQ && NT <= 2 && kThreads * 8 == 4096;
  constexpr bool stage4k = STAGE4K_C;
  // (in a cluster split each block scales by the max over its own k range, and its partial sums
  // are scaled back before the cluster sums them: power-of-two scalings are exact, so the logits
  // are the same bits as with one scale for the whole row)
  const bool onepass = ONEPASS_C && !stage4k;
  constexpr bool STAGER_C = !STAGE4K_C && (VAR == 0 || VAR == 3 || VAR == 4) &&
                            XF == TFD_X_BF16 && !AQ && NT == 1 && KSL == 4;
  // (measured faster where the general loop would take two passes; slower for one)
  const bool stager = STAGER_C && spad * STEPK / 8 > kThreads && spad * STEPK / 8 <= 2 * kThreads;
  if constexpr (!STAGE4K_C) TFD_STAMP(a.trace, 57);  // general staging: after the first barrier
  if (F16 && !onepass && !stage4k) {
    if (F16) {
      // per-row max |x| over the whole row (non-negative floats order like their bit patterns): the
      // chunks of all rows taken together, U loads in flight per thread; a warp whose lanes share a
      // row takes its maximum and makes one shared atomic, otherwise each lane makes its own
      constexpr int U = XF == TFD_X_F32 ? 4 : 8;
      const int chunks = (int)(K / 8);
      const int total = rows * chunks;
      for (int base = 0; base < total; base += U * kThreads) {  // the same trip count in every lane
        float m[U];
        int rr[U];
        if (XF != TFD_X_F32) {
          uint4 v[U];
  #pragma unroll
          for (int u = 0; u < U; ++u) {
            const int idx = base + u * kThreads + tid;
            const bool ok = idx < total;
            rr[u] = ok ? idx / chunks : 0;
            v[u] = ok ? *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.x) +
                                                       (int64_t)rr[u] * a.ldx + 8 * (idx - rr[u] * chunks))
                      : make_uint4(0u, 0u, 0u, 0u);
          }
  #pragma unroll
          for (int u = 0; u < U; ++u) {
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            m[u] = 0.0f;
  #pragma unroll
            for (int i = 0; i < 4; ++i) m[u] = fmaxf(m[u], fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
          }
        } else {
          float4 v[U][2];
  #pragma unroll
          for (int u = 0; u < U; ++u) {
            const int idx = base + u * kThreads + tid;
            const bool ok = idx < total;
            rr[u] = ok ? idx / chunks : 0;
            const float4* p = reinterpret_cast<const float4*>(
                reinterpret_cast<const float*>(a.x) + (int64_t)rr[u] * a.ldx + 8 * (idx - rr[u] * chunks));
            v[u][0] = ok ? p[0] : make_float4(0.f, 0.f, 0.f, 0.f);
            v[u][1] = ok ? p[1] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
  #pragma unroll
          for (int u = 0; u < U; ++u) {
            m[u] = 0.0f;
  #pragma unroll
            for (int h = 0; h < 2; ++h)
              m[u] = fmaxf(m[u], fmaxf(fmaxf(fabsf(v[u][h].x), fabsf(v[u][h].y)),
                                       fmaxf(fabsf(v[u][h].z), fabsf(v[u][h].w))));
          }
        }
  #pragma unroll
        for (int u = 0; u < U; ++u) {
          const int r0 = __shfl_sync(0xffffffffu, rr[u], 0);
          if (__all_sync(0xffffffffu, rr[u] == r0)) {
            const float mw = warp_max(m[u]);
            if (lane == 0) atomicMax(&sxmax[r0], __float_as_uint(mw));
          } else {
            atomicMax(&sxmax[rr[u]], __float_as_uint(m[u]));
          }
        }
      }
      __syncthreads();
    }
  }
  auto row_scales_from_max = [&]() {
    if (tid < kMaxRowsPad) {
      if (AQ) {  // the row's E4M3 scale s = amax / 448 (IEEE division): epilogue factor and divisor
        const float sx = __fdiv_rn(__uint_as_float(sxmax[tid]), 448.0f);
        sxscale[tid] = sx;
        sxmax[tid] = __float_as_uint(sx);
      } else {
        int e = 0;
        const uint32_t ef = (sxmax[tid] >> 23) & 0xFFu;
        if (F16 && sxmax[tid] != 0u && ef != 0xFFu) {
          e = (int)ef - 127 - 14;
          e = e < -110 ? -110 : (e > 110 ? 110 : e);
        }
        sxscale[tid] = __uint_as_float((uint32_t)(e + 127) << 23);  // 2^e
        sxmax[tid] = (uint32_t)(127 - e) << 23;                       // bits of 2^-e
      }
    }
    __syncthreads();
  };
  if (!onepass && !stage4k) row_scales_from_max();
  // ---- activations -> shared memory, in MMA B-fragment order ----
  if constexpr (STAGE4K_C) {
    const int k0 = 8 * tid;
    const int s = k0 / STEPK;
    const int rem = k0 - s * STEPK;
    const int tt = BLK ? (rem & 31) >> 3 : rem / E;
    const int hf = BLK ? rem >> 5 : (rem - tt * E) >> 3;
    uint4 v[8 * NT];
#pragma unroll
    for (int r = 0; r < 8 * NT; ++r)
      v[r] = r < rows ? *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.x) +
                                                        (int64_t)r * a.ldx + k0)
                      : make_uint4(0u, 0u, 0u, 0u);
    l2_prefetch();
#if TFD_TRACE
    if (a.trace != nullptr && tid == 0) {  // slot 56: a value of the loads, so slot 57 waits for them
      uint32_t z = 0u;
#pragma unroll
      for (int r = 0; r < 8 * NT; ++r) z ^= v[r].x;
      a.trace[(int64_t)blockIdx.x * kTraceSlots + 56] = z;
    }
#endif
    TFD_STAMP(a.trace, 57);
    if (F16) {
      // each row's max |x| (non-negative floats order like their bit patterns): a warp maximum,
      // one shared atomic per warp and row
#pragma unroll
      for (int r = 0; r < 8 * NT; ++r) {
        if (r < rows) {  // block-uniform
          const uint32_t w[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
          uint32_t m = 0u;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            m = max(m, max((w[i] << 16) & 0x7FFFFFFFu, w[i] & 0x7FFF0000u));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0 && m != 0u) atomicMax(&sxmax[r], m);
        }
      }
      __syncthreads();
      row_scales_from_max();
      TFD_STAMP(a.trace, 58);
      // scaled by the row's 2^-e into f16 (exact for every bf16 down to 2^-32 of the row's max)
#pragma unroll
      for (int r = 0; r < 8 * NT; ++r) {
        const float inv = __uint_as_float(sxmax[r]);
        const uint32_t w[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          asm("cvt.rn.f16x2.f32 %0, %1, %2;"
              : "=r"(o[j])
              : "f"(bf16_hi(w[j]) * inv), "f"(bf16_lo(w[j]) * inv));
        }
        v[r] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    TFD_STAMP(a.trace, 59);
#pragma unroll
    for (int r = 0; r < 8 * NT; ++r) xs[((s * NT + (r >> 3)) * H + hf) * 32 + (r & 7) * 4 + tt] = v[r];
  } else if (STAGER_C && stager) {
    // one n-tile, a block k range of 513-1024 chunks a row (small matrices, e.g. the pass's
    // 11008-wide projection): like the 4096-wide form, every chunk a thread owns (two) loaded at
    // once for all rows, the block's row maxima and f16 conversion in registers, one store a slot
    constexpr int CPT = 2;
    const int cpr = spad * STEPK / 8;
    uint4 v[CPT][8];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = tid + i * kThreads;
      const int64_t kg = (int64_t)kstep0 * STEPK + 8 * c;
      const bool kin = c < cpr && kg < K;
#pragma unroll
      for (int r = 0; r < 8; ++r)
        v[i][r] = (kin && r < rows) ? *reinterpret_cast<const uint4*>(
                                          reinterpret_cast<const uint16_t*>(a.x) + (int64_t)r * a.ldx + kg)
                                    : make_uint4(0u, 0u, 0u, 0u);
    }
    if (csplit > 1) l2_prefetch();
    TFD_STAMP(a.trace, 57);
    if (F16) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r < rows) {  // block-uniform
          uint32_t m = 0u;
#pragma unroll
          for (int i = 0; i < CPT; ++i) {
            const uint32_t w[4] = {v[i][r].x, v[i][r].y, v[i][r].z, v[i][r].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) m = max(m, max((w[j] << 16) & 0x7FFFFFFFu, w[j] & 0x7FFF0000u));
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0 && m != 0u) atomicMax(&sxmax[r], m);
        }
      }
      __syncthreads();
      row_scales_from_max();
      TFD_STAMP(a.trace, 58);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float inv = __uint_as_float(sxmax[r]);
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
          const uint32_t w[4] = {v[i][r].x, v[i][r].y, v[i][r].z, v[i][r].w};
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o[j]) : "f"(bf16_hi(w[j]) * inv), "f"(bf16_lo(w[j]) * inv));
          v[i][r] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    TFD_STAMP(a.trace, 59);
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = tid + i * kThreads;
      if (c < cpr) {
        const int k0 = 8 * c;
        const int s = k0 / STEPK;
        const int rem = k0 - s * STEPK;
        const int tt = BLK ? (rem & 31) >> 3 : rem / E;
        const int hf = BLK ? rem >> 5 : (rem - tt * E) >> 3;
#pragma unroll
        for (int r = 0; r < 8; ++r) xs[(s * H + hf) * 32 + r * 4 + tt] = v[i][r];
      }
    }
  } else
  // Chunk (r, c) (8 consecutive k of activation row r at column c of this block's k range) goes to
  // one 16-byte fragment slot. Thread tid takes columns tid, tid + 512, ... (a block-uniform loop),
  // so each column's place in the fragment order is computed once with compile-time divisions;
  // XU rows of a column are loaded before any is stored; rows past `rows` only get zeros.
  {
    const int cpr = spad * STEPK / 8;  // chunks per row of this block's k range
    constexpr int NR = 8 * NT;         // activation rows of the tile
    constexpr int XU = XF == TFD_X_F32 ? 4 : 8;
    for (int c0 = 0; c0 < cpr; c0 += kThreads) {
      const int c = c0 + tid;
      const bool cin = c < cpr;
      const int k0 = c * 8;  // within the block's k range
      const int s = k0 / STEPK;
      const int rem = k0 - s * STEPK;
      // A thread's 16-element chunk is contiguous, except in the block-32 form, where it is 8
      // elements of each 32-wide scale block of the step (so every MMA stays inside one block).
      const int tt = BLK ? (rem & 31) >> 3 : rem / E;
      const int hf = BLK ? rem >> 5 : (rem - tt * E) >> 3;
      const int64_t kg = (int64_t)kstep0 * STEPK + k0;  // in the whole row
      const bool kin = cin && kg < K;
#pragma unroll
      for (int r0 = 0; r0 < NR; r0 += XU) {
        if (r0 >= rows) {  // block-uniform: padding rows are zeros
#pragma unroll
          for (int u = 0; u < XU; ++u) {
            const int r = r0 + u;
            if (r >= NR || !cin) continue;
            const int ln = (r & 7) * 4 + tt, nt = r >> 3;
            if (AQ) reinterpret_cast<uint2*>(xs)[((s * NT + nt) * 32 + ln) * 2 + hf] = make_uint2(0u, 0u);
            else
#pragma unroll
              for (int pl = 0; pl < PL; ++pl)
                xs[(((pl * spad + s) * NT + nt) * H + hf) * 32 + ln] = make_uint4(0u, 0u, 0u, 0u);
          }
          continue;
        }
        uint4 raw[XU][XF == TFD_X_F32 ? 2 : 1];
#pragma unroll
        for (int u = 0; u < XU; ++u) {
          const int r = r0 + u;
          const bool ok = kin && r < rows && r < NR;
          if (XF == TFD_X_F32) {
            const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(a.x) +
                                                            (int64_t)r * a.ldx + kg);
            raw[u][0] = ok ? p[0] : make_uint4(0u, 0u, 0u, 0u);
            raw[u][XF == TFD_X_F32 ? 1 : 0] = ok ? p[1] : make_uint4(0u, 0u, 0u, 0u);
          } else {
            raw[u][0] = ok ? *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.x) +
                                                           (int64_t)r * a.ldx + kg)
                           : make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int u = 0; u < XU; ++u) {
          const int r = r0 + u;
          if (r >= NR) continue;
          const int ln = (r & 7) * 4 + tt;
          const int nt = r >> 3;
          const uint4 v = raw[u][0];
          if (ONEPASS_C && onepass) {  // block-uniform
            // raw bf16 bits in the f16 slot; the row's max |x| (non-negative floats order like
            // their bit patterns): a warp maximum and one shared atomic per warp
            uint32_t m = 0u;
            if (cin) {
              xs[((s * NT + nt) * H + hf) * 32 + ln] = v;
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int i = 0; i < 4; ++i)
                m = max(m, max((w[i] << 16) & 0x7FFFFFFFu, w[i] & 0x7FFF0000u));
            }
            if (r < rows) {  // block-uniform
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
              if (lane == 0 && m != 0u) atomicMax(&sxmax[r], m);
            }
            continue;
          }
          if (!cin) continue;
          if (AQ) {
            // 8 codes: code = e4m3(fl32(x / s)), s = 0 for a zero row (its codes are zero)
            const float inv = __uint_as_float(sxmax[r]);
            const uint32_t uw[4] = {v.x, v.y, v.z, v.w};
            uint32_t q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float lo = bf16_lo(uw[i]), hi = bf16_hi(uw[i]);
              if (inv > 0.0f) { lo = __fdiv_rn(lo, inv); hi = __fdiv_rn(hi, inv); }
              q[i] = f32x2_to_e4m3x2(lo, hi);
            }
            reinterpret_cast<uint2*>(xs)[((s * NT + nt) * 32 + ln) * 2 + hf] =
                make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
          } else if (XF == TFD_X_BF16 && !F16) {
            xs[((s * NT + nt) * H + hf) * 32 + ln] = v;
          } else {
            const float inv = F16 ? __uint_as_float(sxmax[r]) : 1.0f;
            float f[8];
            if (XF == TFD_X_BF16) {
              const uint32_t uw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) { f[2 * i] = bf16_lo(uw[i]); f[2 * i + 1] = bf16_hi(uw[i]); }
            } else {
              const uint4 v2 = raw[u][XF == TFD_X_F32 ? 1 : 0];
              f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
              f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
              f[4] = __uint_as_float(v2.x); f[5] = __uint_as_float(v2.y);
              f[6] = __uint_as_float(v2.z); f[7] = __uint_as_float(v2.w);
            }
            uint16_t h[3][8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (PL == 1) h[0][e] = f32_to_f16_bits(f[e] * inv);   // bf16 x, FP8 weights
              else split3<F16>(f[e] * inv, h[0][e], h[1][e], h[2][e]);
            }
#pragma unroll
            for (int pl = 0; pl < PL; ++pl) {
              uint4 o;
              o.x = h[pl][0] | ((uint32_t)h[pl][1] << 16);
              o.y = h[pl][2] | ((uint32_t)h[pl][3] << 16);
              o.z = h[pl][4] | ((uint32_t)h[pl][5] << 16);
              o.w = h[pl][6] | ((uint32_t)h[pl][7] << 16);
              xs[(((pl * spad + s) * NT + nt) * H + hf) * 32 + ln] = o;
            }
          }
        }
      }
    }
    if constexpr (!STAGE4K_C) {
      if (csplit > 1) l2_prefetch();
    }
    TFD_STAMP(a.trace, 58);  // this thread's chunks stored
    if (ONEPASS_C && onepass) {
      __syncthreads();  // every row's max |x| and every raw chunk is in shared memory
      row_scales_from_max();
      // each slot scaled by its row's 2^-e and rounded to f16 (exact for every bf16 down to
      // 2^-32 of the row's max); a slot's row is (lane slot / 4) + 8 n-tile
      const int slots = spad * NT * H * 32;
      for (int i = tid; i < slots; i += kThreads) {
        const int ln = i & 31;
        const int nt = (i / (H * 32)) % NT;
        const int r = nt * 8 + (ln >> 2);
        if (r >= rows) continue;  // padding rows hold zeros already
        const float inv = __uint_as_float(sxmax[r]);
        const uint4 v = xs[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o[j]) : "f"(bf16_hi(w[j]) * inv), "f"(bf16_lo(w[j]) * inv));
        xs[i] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    TFD_STAMP(a.trace, 59);
  }
  __syncthreads();
  if (PRIME_LATE || csplit > 1) prime();
  TFD_STAMP(a.trace, 1);

  // One step: MMA j of the step takes elements [4j, 4j + 4) of each thread's chunk. All activation
  // fragments of the step are read first; each weight fragment is widened just before its MMAs.
  // Block-32 form: the step is two 32-wide blocks (MMAs 0-1 and 2-3), each summed on its own and
  // added to the accumulator times its scale; its activation fragments are read per block, which
  // keeps fewer registers live.
  // CUDA-core form: per thread the partial dot products of its two weight rows (g, g + 8) with
  // every activation row over its k elements, reduced over the four lanes of a row at the end of
  // the k-slice into the MMA accumulator layout.
  constexpr bool FFMA = TFD_GEMV_FFMA && WF == TFD_W_BF16 && XF == TFD_X_BF16;
  float accf[2][FFMA ? 8 * NT : 1];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int c = 0; c < (FFMA ? 8 * NT : 1); ++c) accf[i][c] = 0.0f;
  auto compute = [&](const WLoad<WF>& b, int sg, float (&acc)[NT][4]) {
    if constexpr (FFMA) {
      float wv[2][8];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          wv[i][2 * e] = bf16_lo(b.r[i][e]);
          wv[i][2 * e + 1] = bf16_hi(b.r[i][e]);
        }
#pragma unroll
      for (int c = 0; c < 8 * NT; ++c) {
        if (c < rows) {  // warp-uniform
          // x[c][the thread's 8 k elements of this step]: the B fragment slot of (c, t)
          const uint4 v = xs[(sg * NT + (c >> 3)) * 32 + (c & 7) * 4 + t];
          const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = bf16_lo(xw[e]), x1 = bf16_hi(xw[e]);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              accf[i][c] = fmaf(wv[i][2 * e], x0, accf[i][c]);
              accf[i][c] = fmaf(wv[i][2 * e + 1], x1, accf[i][c]);
            }
          }
        }
      }
      (void)acc;
    } else if constexpr (AQ) {
      // MMA j (k = 32) takes codes [8j, 8j + 8) of each thread's 16: one scale block in the block-32
      // forms, where each MMA starts from zero and is added in fp32 times its block's scale; the
      // row-scaled form accumulates in the MMAs.
      uint4 xq[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) xq[nt] = xs[(sg * NT + nt) * 32 + lane];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float sc = BLK ? e8m0_scale((b.scb >> (8 * j)) & 0xFFu) : 1.0f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (BLK) {
            float c[4];
            mma_e4m3_16832_z(c, b.r[0][2 * j], b.r[1][2 * j], b.r[0][2 * j + 1], b.r[1][2 * j + 1],
                             j == 0 ? xq[nt].x : xq[nt].z, j == 0 ? xq[nt].y : xq[nt].w);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][i] = fmaf(sc, c[i], acc[nt][i]);
          } else {  // one scale per row: the MMAs accumulate in place
            mma_e4m3_16832(acc[nt], b.r[0][2 * j], b.r[1][2 * j], b.r[0][2 * j + 1],
                           b.r[1][2 * j + 1], j == 0 ? xq[nt].x : xq[nt].z,
                           j == 0 ? xq[nt].y : xq[nt].w);
          }
        }
      }
    } else if constexpr (BLK) {
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t xq[NT][PL][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int pl = 0; pl < PL; ++pl) {
            const uint4 v = xs[(((pl * spad + sg) * NT + nt) * H + hb) * 32 + lane];
            xq[nt][pl][0] = v.x; xq[nt][pl][1] = v.y; xq[nt][pl][2] = v.z; xq[nt][pl][3] = v.w;
          }
        float c[NT][4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          uint32_t A0, A1, A2, A3;
          e4m3x4_to_f16x2(b.r[0][2 * hb + jj], A0, A2);
          e4m3x4_to_f16x2(b.r[1][2 * hb + jj], A1, A3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int pl = 0; pl < PL; ++pl) {
              if (jj == 0 && pl == 0)  // the block's first MMA starts its partial sum
                mma_f16_16816_z(c[nt], A0, A1, A2, A3, xq[nt][pl][0], xq[nt][pl][1]);
              else
                mma_f16_16816(c[nt], A0, A1, A2, A3, xq[nt][pl][2 * jj], xq[nt][pl][2 * jj + 1]);
            }
        }
        const float sc = e8m0_scale((b.scb >> (8 * hb)) & 0xFFu);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[nt][i] = fmaf(sc, c[nt][i], acc[nt][i]);
      }
    } else {
    uint32_t xw[NT][PL][4 * H];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int pl = 0; pl < PL; ++pl)
#pragma unroll
        for (int hf = 0; hf < H; ++hf) {
          uint4 v = xs[(((pl * spad + sg) * NT + nt) * H + hf) * 32 + lane];
          xw[nt][pl][4 * hf] = v.x; xw[nt][pl][4 * hf + 1] = v.y;
          xw[nt][pl][4 * hf + 2] = v.z; xw[nt][pl][4 * hf + 3] = v.w;
        }
    float c[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[nt][i] = acc[nt][i];
#pragma unroll
    for (int j = 0; j < MMAJ; ++j) {
      uint32_t A0, A1, A2, A3;
      if (WF == TFD_W_BF16) {
        A0 = b.r[0][2 * j]; A1 = b.r[1][2 * j]; A2 = b.r[0][2 * j + 1]; A3 = b.r[1][2 * j + 1];
      } else {
        e4m3x4_to_f16x2(b.r[0][j], A0, A2);
        e4m3x4_to_f16x2(b.r[1][j], A1, A3);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int pl = 0; pl < PL; ++pl) {
          if (F16) mma_f16_16816(c[nt], A0, A1, A2, A3, xw[nt][pl][2 * j], xw[nt][pl][2 * j + 1]);
          else mma_bf16_16816(c[nt], A0, A1, A2, A3, xw[nt][pl][2 * j], xw[nt][pl][2 * j + 1]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = c[nt][i];
    }
  };

  // Epilogue of one output value: scale, store, rank.
  // slot = 2 * n-tile + (act & 1); with 4 k-slices a reducer warp handles one n-tile
  constexpr int BS = KSL == 1 ? 2 * NT : 2;
  uint64_t best[BS];
#pragma unroll
  for (int i = 0; i < BS; ++i) best[i] = 0ull;
  // online softmax state (max, sum of exp(v - max)) of this thread's outputs, for the confidence
  float2 ms[BS];
#pragma unroll
  for (int i = 0; i < BS; ++i) ms[i] = make_float2(-INFINITY, 0.0f);
  const bool want_conf = a.topk == 1 && a.top1_conf != nullptr;
  // Returns the stored value (NaN outside the output).
  auto epi = [&](int64_t row, int act, float v, int slot, float rsc) -> float {
    if (row >= N || act >= rows) return __uint_as_float(0x7FC00000u);
    if (F16 && !(ONEPASS_C && onepass && csplit > 1)) v *= sxscale[act];  // else scaled per block
    if (WF == TFD_W_FP8_ROW) v *= rsc;
    const int64_t yi = (int64_t)act * a.ldy + row;
    if (a.out_mode == TFD_OUT_F32) {
      reinterpret_cast<float*>(a.y)[yi] = v;
    } else if (a.out_mode == TFD_OUT_BF16) {
      reinterpret_cast<uint16_t*>(a.y)[yi] = f32_to_bf16_bits(v);
    } else if (a.out_mode == TFD_OUT_ADD_BF16) {
      uint16_t* yp = reinterpret_cast<uint16_t*>(a.y) + yi;
      *yp = f32_to_bf16_bits(bf16_bits_to_f32(*yp) + v);
    }
    if (a.topk == 1) {
      const int32_t id = a.id_map ? __ldg(a.id_map + row) : (int32_t)row;
      best[slot] = umax64(best[slot], make_key(v, id));
      if (want_conf && v > -INFINITY) {  // NaN and -inf add nothing
        if (v > ms[slot].x) {
          ms[slot].y = ms[slot].y * expf(ms[slot].x - v) + 1.0f;
          ms[slot].x = v;
        } else {
          ms[slot].y += expf(v - ms[slot].x);
        }
      }
    } else if (a.logits != nullptr && a.logits != a.y) {
      a.logits[(int64_t)act * a.ld_logits + row] = v;
    }
    return v;
  };

  // Epilogue of one finished MMA tile (rows g, g + 8 of tile `tile` of group gi; activations act0,
  // act0 + 1), and the tile's sub-group maximum for a later top-k.
  // row scales of the warp's own tile in the current group, loaded at the group's start (fast path)
  float rs_pref[2] = {0.0f, 0.0f};
  auto finish_tile = [&](int64_t gi, int tile, int act0, float4 v, int slot0) {
    if (!tile_in(gi, tile)) return;  // warp-uniform: the tile belongs to the next block
    const int64_t row_lo = row_off + gi * GR + tile * 16 + g;
    float rs0 = 1.0f, rs1 = 1.0f;
    if (WF == TFD_W_FP8_ROW) {
      if (FASTK && CSC == 1 && tile == mt) {  // (a split's leader finishes the previous group)
        rs0 = rs_pref[0];
        rs1 = rs_pref[1];
      } else {
        rs0 = row_lo < N ? __ldg(row_scales + row_lo) : 0.0f;
        rs1 = row_lo + 8 < N ? __ldg(row_scales + row_lo + 8) : 0.0f;
      }
    }
    const float o0 = epi(row_lo, act0, v.x, slot0, rs0);
    const float o1 = epi(row_lo, act0 + 1, v.y, slot0 + 1, rs0);
    const float o2 = epi(row_lo + 8, act0, v.z, slot0, rs1);
    const float o3 = epi(row_lo + 8, act0 + 1, v.w, slot0 + 1, rs1);
    if (a.submax != nullptr) {
      // the 16 rows of this MMA tile are one sub-group: rows g and g + 8 of the eight lanes that
      // share t
      uint32_t m0 = max(value_key(o0), value_key(o2));
      uint32_t m1 = max(value_key(o1), value_key(o3));
#pragma unroll
      for (int o = 4; o <= 16; o <<= 1) {
        m0 = max(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        m1 = max(m1, __shfl_xor_sync(0xffffffffu, m1, o));
      }
      const int64_t sg = row_off / 16 + gi * MT + tile;
      const int64_t S = (N + 15) / 16;
      if (g == 0 && sg < S) {
        if (act0 < rows) a.submax[(int64_t)act0 * S + sg] = m0;
        if (act0 + 1 < rows) a.submax[(int64_t)(act0 + 1) * S + sg] = m1;
        if (a.part_max != nullptr) {  // the part's maximum of each row
          if (act0 < rows) atomicMax(&spmax[act0], m0);
          if (act0 + 1 < rows) atomicMax(&spmax[act0 + 1], m1);
        }
      }
    }
  };

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
  int rb = 0;
  const int mr = warp & 3, nr = warp >> 2;  // reducer role of warps < 4 * NT
  // Cluster split of more than two: the blocks meet on a split cluster barrier, one group behind.
  // At the end of group j every block waits for the barrier phase of group j - 1 (long complete
  // unless a block lags by a whole group), the leader then sums group j - 1's partials from every
  // block's shared memory, and each block stores its partials of group j and arrives. A block
  // writes a partial buffer again two groups on, after its wait has seen the leader's arrival
  // behind its read. (The leader's arrival is relaxed: it has consumed the values it read. A
  // release would first wait for every load the block has in flight, the weight ring included.)
  // Cluster split of two: no cluster barrier per group. The second block writes its partials of
  // group j straight into the leader's buffer j & 1 with asynchronous stores counted by the
  // leader's mbarrier s_full[j & 1]; the leader keeps its own partials in registers, waits on
  // s_full one group later, sums, and each of its reducer warps then arrives on the second block's
  // s_empty[j & 1], which the second block waits for before it writes that buffer again.
  // the leader's own partial of its last group (split of two): in registers at four n-tiles
  // (shared memory is full there), else after the two exchange buffers (fewer registers live)
  float4 vown = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float4* cown = cpart + 2 * 4 * NT * 32;
  auto take2 = [&](int64_t gp, int jp) {  // the leader's sum of the pair's group jp (group gp)
    if (warp < 4 * NT) {
      const int pb = jp & 1;
      if (!mbar_wait(&s_full[pb], (uint32_t)(jp >> 1) & 1u)) set_dev_status(a.status, TFD_ERR_TIMEOUT);
      const float4 u = cpart[(pb * 4 * NT + warp) * 32 + lane];
      // rank order: the leader's partial, then the second block's
      float4 v = NT == 4 ? vown : cown[warp * 32 + lane];
      v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
      __syncwarp();  // every lane of the warp has consumed its slot
      if (lane == 0)
        asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                         cluster_addr(&s_empty[pb], 1))
                     : "memory");
      finish_tile(gp, mr, nr * 8 + 2 * t, v, 0);
    }
  };
  auto cluster_take = [&](int64_t gp, int pb) {
    if (crank == 0 && warp < 4 * NT) {
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int q = 0; q < csplit; ++q) {  // blocks in rank order
        const float4 u = cg::this_cluster().map_shared_rank(cpart, q)[(pb * 4 * NT + warp) * 32 + lane];
        v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
      }
      finish_tile(gp, mr, nr * 8 + 2 * t, v, 0);
    }
  };
  // The end of group gi: k-slice partials summed, epilogue.
  auto group_end = [&](int64_t gi, int j) {
    if constexpr (FFMA) {
      // sum over the four lanes of each weight row, then lane t keeps columns 2t, 2t + 1 of each
      // n-tile, as the MMA accumulator holds them
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int c = 0; c < 8 * NT; ++c) {
          accf[i][c] += __shfl_xor_sync(0xffffffffu, accf[i][c], 1);
          accf[i][c] += __shfl_xor_sync(0xffffffffu, accf[i][c], 2);
        }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = q >> 1, h = q & 1;
          float v = accf[i][nt * 8 + h];
#pragma unroll
          for (int tt = 1; tt < 4; ++tt)
            if (t == tt) v = accf[i][nt * 8 + 2 * tt + h];
          acc[nt][q] = v;
        }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int c = 0; c < 8 * NT; ++c) accf[i][c] = 0.0f;
    }
    if constexpr (KSL == 1) {  // the warp holds whole dot products: epilogue straight away
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        finish_tile(gi, mt, nt * 8 + 2 * t, make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]),
                    2 * nt);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
      }
    } else {
    // k-slice partials -> shared memory; fixed-order sum; epilogue.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      red[((rb * kWarps + warp) * NT + nt) * 32 + lane] =
          make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
    }
    __syncthreads();
    if (dyn && claimer) s_q[(j + 3) & 3] = claim();
    // (a split's groups are consecutive: the previous one is gi - 1)
    if (csplit > 2 && j > 0) {
      asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
      cluster_take(gi - 1, rb ^ 1);
    }
    if (csplit == 2 && j > 0 && crank == 0) take2(gi - 1, j - 1);
    if (csplit == 2 && crank == 0 && tid == 0)  // group j's bytes from the second block
      asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                       smem_addr(&s_full[j & 1])),
                   "r"(4 * NT * 32 * 16)
                   : "memory");
    if (warp < 4 * NT) {
      // warp index = ks * 4 + mt, so the partials of row tile mr are warps mr, 4+mr, 8+mr, 12+mr.
      float4 v = red[((rb * kWarps + mr) * NT + nr) * 32 + lane];
#pragma unroll
      for (int ksi = 1; ksi < 4; ++ksi) {
        float4 u = red[((rb * kWarps + ksi * 4 + mr) * NT + nr) * 32 + lane];
        v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
      }
      if (csplit == 1) finish_tile(gi, mr, nr * 8 + 2 * t, v, 0);
      else {
        if (ONEPASS_C && onepass) {  // this block's own activation scale, before the cluster sum
          const int act0 = nr * 8 + 2 * t;
          v.x *= sxscale[act0]; v.z *= sxscale[act0];
          v.y *= sxscale[act0 + 1]; v.w *= sxscale[act0 + 1];
        }
        if (csplit == 2) {
          if (crank == 0) {
            if (NT == 4) vown = v;
            else cown[warp * 32 + lane] = v;  // read by this thread at the next group's end
          } else {
            const int b = j & 1;  // written again two groups on, once the leader has read it
            if (j >= 2 && !mbar_wait(&s_empty[b], (uint32_t)((j >> 1) - 1) & 1u))
              set_dev_status(a.status, TFD_ERR_TIMEOUT);
            if (!TFD_TEST_STALL_EXCHANGE)
              st_async_f4(cluster_addr(cpart + (b * 4 * NT + warp) * 32 + lane, 0), v,
                          cluster_addr(&s_full[b], 0));
          }
        } else {
          cpart[(rb * 4 * NT + warp) * 32 + lane] = v;
        }
      }
    }
    if (csplit > 2) {
      if (crank == 0) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
      else asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    }
    }
    rb ^= 1;
    TFD_STAMP(a.trace, 2 + (j < 55 ? j : 55));
  };
  // (split of two: both blocks' exchange barriers are initialised)
  if (csplit == 2) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if constexpr (FASTK) {
    for (int j = 0;; ++j) {
      const int64_t gi = seq_group(j);
      if (gi >= kNoGroup) break;  // block-uniform
      const int64_t gn = seq_group(j + 1);
      const bool nxt = gn < kNoGroup;  // warp-uniform
      const unsigned char* q = fast_ptr(gi);
      const unsigned char* qn = fast_ptr(nxt ? gn : gi);
      const uint8_t* sq = BLK ? fast_sp(gi) : nullptr;
      const uint8_t* sqn = BLK ? fast_sp(nxt ? gn : gi) : nullptr;
      if (WF == TFD_W_FP8_ROW && CSC == 1) {
        rs_pref[0] = __ldg(row_scales + gi * GR + mt * 16 + g);
        rs_pref[1] = __ldg(row_scales + gi * GR + mt * 16 + g + 8);
      }
#pragma unroll
      for (int st = 0; st < SSLC; ++st) {
        compute(buf[st % D], s_loc + st, acc);
        const int s2 = st + D;  // the step this ring slot takes next
        if (s2 < SSLC)
          fload(buf[st % D], q + (int64_t)s2 * STEPK * EB, sq + 2 * s2);
        else if (nxt)
          fload(buf[st % D], qn + (int64_t)(s2 - SSLC) * STEPK * EB, sqn + 2 * (s2 - SSLC));
      }
      group_end(gi, j);
    }
  } else {
    for (int j = 0;; ++j) {
      const int64_t gi = seq_group(j);
      if (gi >= kNoGroup) break;  // block-uniform
      for (int s0 = 0; s0 < ssl_loop; s0 += D) {
#pragma unroll
        for (int st = 0; st < D; ++st) {
          // an empty step (past ssl) reads any valid activation slot: its weights are zero
          compute(buf[st], s_loc + (s0 + st < ssl ? s0 + st : 0), acc);
          issue(buf[st]);
        }
      }
      group_end(gi, j);
    }
  }
  if (csplit > 1) {
    if (g_begin < g_end) {  // the last group's partials
      if (csplit == 2) {
        if (crank == 0) take2(g_end - 1, (int)(g_end - 1 - g_begin));
      } else {
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        cluster_take(g_end - 1, rb ^ 1);
      }
    }
    cg::this_cluster().sync();  // the leader has read every block's last partial
    if (crank != 0) return;
  }

  TFD_STAMP(a.trace, 61);
  if (dyn && a.topk != 1) {
    // the last block to finish (every claim of every block is done) zeroes the queue
    __threadfence();
    if (tid == 0 && atomicAdd(a.counter, 1u) == (uint32_t)(a.parts - 1)) {
      *a.counter = 0u;
      *a.queue = 0u;
    }
  }
  if (a.part_max != nullptr) {
    __syncthreads();  // every tile's maximum is in spmax
    if (tid < rows) a.part_max[(int64_t)cid * rows + tid] = spmax[tid];
  }
  if (a.topk != 1) return;
  // ---- top-1: block best per row, then the last block to finish joins the parts ----
  if (KSL == 1 || warp < 4 * NT) {
    // the tile this warp finished, and its n-tiles: (mr, nr) with 4 k-slices, (mt, all) with one
    const int tile = KSL == 1 ? mt : mr;
#pragma unroll
    for (int sl = 0; sl < BS; ++sl) {
      const int nt = KSL == 1 ? sl >> 1 : nr;
      const int c = sl & 1;
      uint64_t key = best[sl];
      key = umax64(key, shfl_xor_u64(key, 4));
      key = umax64(key, shfl_xor_u64(key, 8));
      key = umax64(key, shfl_xor_u64(key, 16));
      if (g == 0) sbest[tile * kMaxRowsPad + nt * 8 + 2 * t + c] = key;
      if (want_conf) {
        float2 q = ms[sl];
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1)
          q = ms_merge(q, make_float2(__shfl_xor_sync(0xffffffffu, q.x, o),
                                      __shfl_xor_sync(0xffffffffu, q.y, o)));
        if (g == 0) sms[tile * kMaxRowsPad + nt * 8 + 2 * t + c] = q;
      }
    }
  }
  __syncthreads();
  if (tid < kMaxRowsPad) {  // tiles merged in a fixed order
    uint64_t m = sbest[tid];
    for (int i = 1; i < MT; ++i) m = umax64(m, sbest[i * kMaxRowsPad + tid]);
    if (tid < rows) a.part_keys[(int64_t)cid * rows + tid] = m;
    if (want_conf) {
      float2 q = sms[tid];
      for (int i = 1; i < MT; ++i) q = ms_merge(q, sms[i * kMaxRowsPad + tid]);
      if (tid < rows) a.part_ms[(int64_t)cid * rows + tid] = q;
    }
  }
  if (tid < kMaxRowsPad) sjoin[tid] = 0ull;
  __threadfence();
  __syncthreads();
  TFD_STAMP(a.trace, 62);
  if (tid == 0) is_last = (atomicAdd(a.counter, 1u) == (uint32_t)(a.parts - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  {
    // every part's key of every row in flight at once (8 loads a thread), then a shared maximum
    // per row (the maximum of keys does not depend on the order)
    constexpr int U = 8;
    const int tot = a.parts * rows;  // key i = part i / rows, row i % rows
    for (int i0 = 0; i0 < tot; i0 += U * kThreads) {
      uint64_t kk[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kThreads + tid;
        kk[u] = i < tot ? __ldcg(a.part_keys + i) : 0ull;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kThreads + tid;
        if (i < tot) atomicMax(reinterpret_cast<unsigned long long*>(&sjoin[i % rows]),
                               (unsigned long long)kk[u]);
      }
    }
  }
  if (want_conf) {
    // parts are merged in a fixed order: p = tid, tid + 512, ..., then lanes, then warps
    for (int r = 0; r < rows; ++r) {
      float2 q = make_float2(-INFINITY, 0.0f);
      for (int p = tid; p < a.parts; p += kThreads)
        q = ms_merge(q, __ldcg(a.part_ms + (int64_t)p * rows + r));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        q = ms_merge(q, make_float2(__shfl_xor_sync(0xffffffffu, q.x, o),
                                    __shfl_xor_sync(0xffffffffu, q.y, o)));
      if (lane == 0) sjms[warp * kMaxRowsPad + r] = q;
    }
  }
  __syncthreads();
  if (tid < rows) {
    const uint64_t key = sjoin[tid];
    a.top_vals[tid * a.ldt] = key_value(key);
    a.top_ids[tid * a.ldt] = key_id(key);
    if (want_conf) {
      float2 q = make_float2(-INFINITY, 0.0f);
      for (int w = 0; w < kWarps; ++w) q = ms_merge(q, sjms[w * kMaxRowsPad + tid]);
      a.top1_conf[tid] = q.y > 0.0f ? 1.0f / q.y : __uint_as_float(0x7FC00000u);
    }
  }
  if (tid == 0) {  // leave the workspace zeroed
    *a.counter = 0u;
    if (dyn) *a.queue = 0u;
  }
  TFD_STAMP(a.trace, 63);
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------

constexpr size_t kSmemLimit = 232448 - 1024;   // sm_100-class dynamic shared memory, minus slack

template <int WF, int XF, int NT, int KSL = 4>
size_t gemv_smem(int64_t k, int* ssl_out) {
  constexpr int E = WTraits<WF>::E;
  int64_t steps = (k + 4 * E - 1) / (4 * E);
  int64_t ssl = (steps + KSL - 1) / KSL;
  if (ssl_out) *ssl_out = (int)ssl;
  return Layout<WF, XF, NT, KSL>::smem_bytes((int)ssl);
}

// The smallest cluster split (1, 2, 4 or 8 blocks sharing a group's k range) whose share of the
// activation tile fits a block's shared memory, or 0 if none does (one k-slice: no split).
template <int WF, int XF, int NT, int KSL>
int gemv_min_split(int64_t k) {
  constexpr int E = WTraits<WF>::E;
  const int64_t steps = (k + 4 * E - 1) / (4 * E);
  for (int c = 1; c <= (KSL == 4 ? 8 : 1); c *= 2) {
    const int64_t ssl = (steps + (int64_t)KSL * c - 1) / ((int64_t)KSL * c);
    if (Layout<WF, XF, NT, KSL>::smem_bytes((int)ssl) <= kSmemLimit) return c;
  }
  return 0;
}

template <int WF, int XF, int NT, int KSL>
tfd_status gemv_launch_k(GemvArgs a, int parts_req, cudaStream_t stream) {
  int ssl = 0;
  size_t smem = gemv_smem<WF, XF, NT, KSL>(a.k, &ssl);
  // Up to 16 rows a 4096-wide tile fits one block; 32 rows of it need k split over a cluster.
  const int cmin = gemv_min_split<WF, XF, NT, KSL>(a.k);
  if (cmin == 0) return TFD_ERR_UNSUPPORTED;
  if (cmin > 1) {
    constexpr int E = WTraits<WF>::E;
    const int64_t steps = (a.k + 4 * E - 1) / (4 * E);
    smem = Layout<WF, XF, NT, KSL>::smem_bytes((int)((steps + 4 * cmin - 1) / (4 * cmin)));
  }
  const int64_t group_rows = 16 * (16 / KSL);
  a.ngroups = (a.n + group_rows - 1) / group_rows;
  auto kern = gemv_kernel<WF, XF, NT, gemv_depth<WF, NT, XF>(), KSL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit) !=
      cudaSuccess)
    return TFD_ERR_CUDA;
  int parts = parts_req;
  int csplit = cmin;
  if (parts <= 0) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem) != cudaSuccess)
      return TFD_ERR_CUDA;
    if (occ < 1) occ = 1;
    const int64_t slots = (int64_t)tfd_host::sm_count() * occ;
    if (KSL == 4 && a.ngroups * 2 <= slots) {
      // Too few groups for the SMs: split k over a cluster of 2, 4 or 8 blocks, keeping at least
      // a ring's depth of steps per k-slice.
      constexpr int E = WTraits<WF>::E;
      constexpr int D = gemv_depth<WF, NT, XF>();
      const int64_t steps = (a.k + 4 * E - 1) / (4 * E);
      int64_t c = slots / a.ngroups;
      if (c > steps / (4 * D)) c = steps / (4 * D);
      const int want = c >= 8 ? 8 : c >= 4 ? 4 : c >= 2 ? 2 : 1;
      csplit = want > cmin ? want : cmin;
    }
    int64_t p = slots / csplit;
    if (p > a.ngroups) p = a.ngroups;
    if (p > kMaxParts) p = kMaxParts;
    if (p < 1) p = 1;
    parts = (int)p;
  }
  a.parts = parts;
  a.csplit = csplit;
  if (a.parts_used != nullptr) *a.parts_used = parts;
  if (csplit == 1) {
    a.ssl = ssl;
#if TFD_GEMV_STAGE4K
    // (not the block-32 forms at two n-tiles: they spill in that instantiation)
    if constexpr (XF == TFD_X_BF16 && KSL == 4 &&
                  (NT == 1 || (NT == 2 && (WF == TFD_W_BF16 || WF == TFD_W_FP8_ROW)))) {
      if (a.k == 4096) {  // staged by one block with constant geometry
        auto k4 = gemv_kernel<WF, XF, NT, gemv_depth<WF, NT, XF>(), KSL, 1>;
#if TFD_GEMV_FAST
        // measured faster for one n-tile of bf16 and row-scaled FP8 weights only (the block-32
        // forms spill when unrolled; two n-tiles gained nothing)
        if constexpr (KSL == 4 && NT == 1 && (WF == TFD_W_BF16 || WF == TFD_W_FP8_ROW) &&
                      4096 / (KSL * 4 * WTraits<WF>::E) >= gemv_depth<WF, NT, XF>()) {
          // whole 64-row groups: the unrolled, check-free instantiation
          if (a.n % (16 * (16 / KSL)) == 0) k4 = gemv_kernel<WF, XF, NT, gemv_depth<WF, NT, XF>(), KSL, 2>;
        }
#endif
        if (cudaFuncSetAttribute(k4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemLimit) != cudaSuccess)
          return TFD_ERR_CUDA;
        k4<<<parts, kThreads, smem, stream>>>(a);
        return tfd_host::launch_status();
      }
    }
#endif
    auto k1 = kern;
    // the FP8 block-32 forms at two n-tiles and the W8A8 forms: the general loop without the
    // split's code (measured slower with it)
    if constexpr (KSL == 4 && NT <= 2 &&
                  ((XF == TFD_X_BF16 && NT == 2 &&
                    (WF == TFD_W_FP8_BLOCK32 || WF == TFD_W_FP8_BLOCK32_IL)) ||
                   XF == TFD_X_BF16_E4M3)) {
      k1 = gemv_kernel<WF, XF, NT, gemv_depth<WF, NT, XF>(), KSL, 4>;
      if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit) !=
          cudaSuccess)
        return TFD_ERR_CUDA;
    }
    k1<<<parts, kThreads, smem, stream>>>(a);
    return tfd_host::launch_status();
  }
  constexpr int E = WTraits<WF>::E;
  const int64_t steps = (a.k + 4 * E - 1) / (4 * E);
  a.ssl = (int)((steps + 4 * csplit - 1) / (4 * csplit));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(parts * csplit));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout<WF, XF, NT, KSL>::smem_bytes(a.ssl);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)csplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kc = kern;
#if TFD_GEMV_FAST
  // a 4096-wide matrix of whole 64-row groups split over two blocks: the unrolled, check-free
  // weight loop (one n-tile of row-scaled FP8 weights; four n-tiles measured slower with it)
  if constexpr (XF == TFD_X_BF16 && KSL == 4 &&
                ((NT == 1 && WF == TFD_W_FP8_ROW)) &&
                4096 / (KSL * 4 * E * 2) >= gemv_depth<WF, NT, XF>()) {
    if (csplit == 2 && a.k == 4096 && a.n % (16 * (16 / KSL)) == 0) {
      kc = gemv_kernel<WF, XF, NT, gemv_depth<WF, NT, XF>(), KSL, 3>;
      if (cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit) !=
          cudaSuccess)
        return TFD_ERR_CUDA;
    }
  }
#endif
  if (cudaLaunchKernelEx(&cfg, kc, a) != cudaSuccess) return TFD_ERR_CUDA;
  return tfd_host::launch_status();
}

// bf16 weights with a short k (fewer than D steps per k-slice, e.g. the 256-wide second GEMV of
// the two-stage head) and enough rows for every SM run with one k-slice and 256-row groups.
template <int WF, int XF, int NT>
tfd_status gemv_launch_t(GemvArgs a, int parts_req, cudaStream_t stream) {
  if constexpr (WF == TFD_W_BF16 && NT <= 2) {
    constexpr int D = gemv_depth<WF, NT, XF>();
    const int64_t steps = (a.k + 4 * WTraits<WF>::E - 1) / (4 * WTraits<WF>::E);
    if ((steps + 3) / 4 < D && (a.n + 255) / 256 >= tfd_host::sm_count())
      return gemv_launch_k<WF, XF, NT, 1>(a, parts_req, stream);
  }
  return gemv_launch_k<WF, XF, NT, 4>(a, parts_req, stream);
}

// Rows 1-8: one n-tile; 9-16: two; 17-32: four (fp32 activations, three operand planes each,
// stop at 16 rows).
template <int WF, int XF>
tfd_status gemv_launch_nt(GemvArgs a, int parts, cudaStream_t s) {
  if (a.rows <= 8) return gemv_launch_t<WF, XF, 1>(a, parts, s);
  if (a.rows <= 16) return gemv_launch_t<WF, XF, 2>(a, parts, s);
  if constexpr (XF != TFD_X_F32) return gemv_launch_t<WF, XF, 4>(a, parts, s);
  return TFD_ERR_UNSUPPORTED;
}

template <int WF>
tfd_status gemv_launch_x(GemvArgs a, int xfmt, int parts, cudaStream_t s) {
  if constexpr (WF != TFD_W_BF16) {
    if (xfmt == TFD_X_BF16_E4M3) return gemv_launch_nt<WF, TFD_X_BF16_E4M3>(a, parts, s);
  }
  if (xfmt == TFD_X_BF16_E4M3) return TFD_ERR_INVALID;
  return xfmt == TFD_X_F32 ? gemv_launch_nt<WF, TFD_X_F32>(a, parts, s)
                           : gemv_launch_nt<WF, TFD_X_BF16>(a, parts, s);
}

}  // namespace tfd_gemv

// The launchers each gemv_w*.cu instantiates (and gemv.cu only declares).
#define TFD_GEMV_EXTERN(WF)                                                                    \
  extern template tfd_status tfd_gemv::gemv_launch_x<WF>(tfd_gemv::GemvArgs, int, int,          \
                                                         cudaStream_t);
#define TFD_GEMV_INSTANTIATE(WF)                                                               \
  template tfd_status tfd_gemv::gemv_launch_x<WF>(tfd_gemv::GemvArgs, int, int, cudaStream_t);

