// attn.cu - one decode position per stream: qk_norm (RMSNorm per head), RoPE, the ring write of
// the new key/value row, and single-query attention over the window read back from the ring.
//
// Follows the TFE draft head page (#42): commit "... ocabulary head" (qk_norm is an RMSNorm on each
// query and key head before RoPE; the window goes up to 511, 512 keys), commit "pass kernels and
// FP8 linears" (single-query window attention in one block, a thread a key and the values split
// over the warps), and the first commits (the head's rows live in a ring; no write of more rows
// than the ring holds). Readings: half-split RoPE pairs (i, i + dim/2) turned by
// p * base^(-2i/dim); the key is rounded to bf16 when written to the ring; the query stays fp32.
//
// A cluster of 4 blocks per (head, stream) splits the window's keys; each block keeps its K rows
// (in registers) and V rows (asynchronous copies into shared memory) in flight at once, 128 keys
// x 256 B each, and the partial softmax states are combined in distributed shared memory.
#include <cooperative_groups.h>

#include <cmath>

#include "common.cuh"

namespace {

using namespace tfd;
namespace cg = cooperative_groups;

constexpr int kDim = 128;
constexpr int kThreads = 256;
constexpr int kCluster = 4;                       // blocks per (head, stream)
constexpr int kMaxKeys = TFD_MAX_WINDOW + 1;      // 512
constexpr int kKeysPerBlock = kMaxKeys / kCluster;  // 128
constexpr int kKeysPerHalfWarp = kKeysPerBlock / 16;  // 8: 16 half-warps per block

__device__ __forceinline__ float block_reduce(float v, float* sred, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = is_max ? warp_max(v) : warp_sum(v);
  __syncthreads();
  if (lane == 0) sred[warp] = v;
  __syncthreads();
  float r = sred[0];
  for (int i = 1; i < kThreads / 32; ++i) r = is_max ? fmaxf(r, sred[i]) : r + sred[i];
  return r;
}

// Each pair's frequency base^(-2i/dim) in turns (1 turn = 2 pi), as a 64-bit binary fraction:
// t_i = frac(base^(-2i/dim) / (2 pi)) * 2^64. For an integer position p, p * t_i mod 2^64 is the
// angle p * base^(-2i/dim) reduced to one turn, exact up to the rounding of t_i (2^-53 relative),
// so the reduction needs no floating-point arithmetic on the device.
struct RopeTurns {
  uint64_t t[kDim / 2];
};

// Lane l of a warp holds elements 4l..4l+3 of a 128-vector: RMSNorm with gamma, then RoPE with
// the angle reduced to [-pi, pi) before the fp32 sine and cosine.
// The sines and cosines of this lane's four pairs at position p (lane l holds pairs
// 4 (l mod 16) .. + 3), shared by every head at that position.
__device__ __forceinline__ void rope_sincos(int p, const RopeTurns& turns, float (&sn)[4],
                                            float (&cs)[4]) {
  const int lane = threadIdx.x & 31;
  const float turn_unit = 1.4629180792671596e-9f;  // 2 pi / 2^32
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * (lane & 15) + j;  // pair index 0..63
    const uint64_t ph = (uint64_t)(uint32_t)p * turns.t[i];  // mod 2^64: the reduced angle
    const float red = (float)(int32_t)(ph >> 32) * turn_unit;
    sincosf(red, &sn[j], &cs[j]);
  }
}

// RMSNorm with gamma, then the rotation by the given sines and cosines.
__device__ __forceinline__ void norm_rope_sc(float (&x)[4], const uint16_t* gamma, float eps,
                                             const float (&sn)[4], const float (&cs)[4]) {
  const int lane = threadIdx.x & 31;
  float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / (float)kDim + eps);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float gm = gamma ? bf16_bits_to_f32(gamma[4 * lane + j]) : 1.0f;
    x[j] = x[j] * inv * gm;
  }
  float other[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) other[j] = __shfl_xor_sync(0xffffffffu, x[j], 16);
  const bool first_half = lane < 16;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // first half holds a = x[i] (partner b = x[i+64]); second half holds b (partner a).
    x[j] = first_half ? (x[j] * cs[j] - other[j] * sn[j]) : (other[j] * sn[j] + x[j] * cs[j]);
  }
}

__device__ __forceinline__ void norm_rope(float (&x)[4], const uint16_t* gamma, float eps, int p,
                                          const RopeTurns& turns) {
  float sn[4], cs[4];
  rope_sincos(p, turns, sn, cs);
  norm_rope_sc(x, gamma, eps, sn, cs);
}

struct AttnPartial {
  float m, l;          // block max score and sum of exp(score - m)
  float acc[kDim];     // sum of exp(score - m) * v
};

// Cluster of 4 blocks per (head, stream): block r of the cluster scores keys [128r, 128r + 128) of
// the window with all their K and V rows in flight at once, keeps a softmax partial (max, sum,
// weighted values), and block 0 combines the four partials read through distributed shared memory
// in a fixed order. Block 0 also writes the new key/value row to the ring; every block computes
// the current key itself, so no block reads the row another block writes.
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 4)
window_attn_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k_new,
                   const uint16_t* __restrict__ v_new, const uint16_t* __restrict__ q_gamma,
                   const uint16_t* __restrict__ k_gamma, float eps, const RopeTurns turns,
                   const int32_t* __restrict__ pos, uint16_t* k_ring, uint16_t* v_ring, int ring,
                   int window, int heads, uint16_t* __restrict__ out, int32_t* dev_status) {
  __shared__ float qn[kDim];
  __shared__ float kcur[kDim];
  __shared__ float vcur[kDim];
  __shared__ float scores[kKeysPerBlock];
  __shared__ float sred[kThreads / 32];
  __shared__ float red_o[16][kDim];
  __shared__ AttnPartial part;
  __shared__ __align__(16) uint16_t vsm[kKeysPerBlock][kDim];  // V rows, copied asynchronously
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int h = blockIdx.x / kCluster, s = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p = pos[s];
  const bool bad = p < 0;  // uniform over the cluster: every block returns after the barriers
  if (bad && crank == 0 && tid == 0) set_dev_status(dev_status, TFD_ERR_DEVICE_DATA);
  const int pp = bad ? 0 : p;
  const int slot = pp % ring;
  const int64_t head_off = ((int64_t)s * heads + h) * kDim;
  const int64_t ring_row = (((int64_t)s * ring + slot) * heads + h) * kDim;
  const int p0 = pp - window > 0 ? pp - window : 0;
  const int nk = pp - p0 + 1;
  const int lo = crank * kKeysPerBlock;              // this block's keys: window index lo..hi-1
  const int hi = lo + kKeysPerBlock < nk ? lo + kKeysPerBlock : nk;
  const int hw = tid >> 4, hl = tid & 15;            // half-warp per key, 8 dims per lane

  // issue this block's K rows (into registers) and V rows (asynchronous copies into shared
  // memory, zero-filled for rows that are not past positions) before the prologue math; each
  // thread later reads back only the V bytes it copied itself
  uint4 kv[kKeysPerHalfWarp];
#pragma unroll
  for (int u = 0; u < kKeysPerHalfWarp; ++u) {
    const int i = lo + hw + 16 * u;
    const bool past = !bad && i < hi && p0 + i < pp;
    const int64_t row = (((int64_t)s * ring + (p0 + i) % ring) * heads + h) * kDim + hl * 8;
    kv[u] = past ? *reinterpret_cast<const uint4*>(k_ring + row) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&vsm[hw + 16 * u][hl * 8]);
    const uint16_t* src = past ? v_ring + row : v_ring;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(past ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  if (!bad && warp < 2) {
    const uint16_t* src = (warp == 0 ? q : k_new) + head_off + 4 * lane;
    uint2 raw = *reinterpret_cast<const uint2*>(src);
    float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    norm_rope(x, warp == 0 ? q_gamma : k_gamma, eps, pp, turns);
    if (warp == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) qn[4 * lane + j] = x[j];
    } else {
      uint16_t b[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) { b[j] = f32_to_bf16_bits(x[j]); kcur[4 * lane + j] = bf16_bits_to_f32(b[j]); }
      if (crank == 0) {
        uint2 o;
        o.x = b[0] | ((uint32_t)b[1] << 16);
        o.y = b[2] | ((uint32_t)b[3] << 16);
        *reinterpret_cast<uint2*>(k_ring + ring_row + 4 * lane) = o;
      }
    }
  } else if (!bad && warp == 2) {
    const uint2 raw = *reinterpret_cast<const uint2*>(v_new + head_off + 4 * lane);
    vcur[4 * lane] = bf16_lo(raw.x);
    vcur[4 * lane + 1] = bf16_hi(raw.x);
    vcur[4 * lane + 2] = bf16_lo(raw.y);
    vcur[4 * lane + 3] = bf16_hi(raw.y);
    if (crank == 0) *reinterpret_cast<uint2*>(v_ring + ring_row + 4 * lane) = raw;
  }
  __syncthreads();

  // scores of this block's keys (the current key from registers of the prologue, via kcur)
  float qv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) qv[j] = qn[hl * 8 + j];
  const float inv_sqrt_d = 1.0f / sqrtf((float)kDim);
#pragma unroll
  for (int u = 0; u < kKeysPerHalfWarp; ++u) {
    const int i = lo + hw + 16 * u;
    float d = 0.0f;
    if (!bad && i < hi && p0 + i == pp) {
#pragma unroll
      for (int j = 0; j < 8; ++j) d = fmaf(qv[j], kcur[hl * 8 + j], d);
    } else {
      const uint32_t w[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        d = fmaf(qv[2 * j], bf16_lo(w[j]), d);
        d = fmaf(qv[2 * j + 1], bf16_hi(w[j]), d);
      }
    }
#pragma unroll
    for (int m = 8; m > 0; m >>= 1) d += __shfl_xor_sync(0xffffffffu, d, m);
    if (hl == 0 && i < hi) scores[i - lo] = d * inv_sqrt_d;
  }
  __syncthreads();
  const int nb = hi > lo ? hi - lo : 0;
  float mx = -INFINITY;
  for (int i = tid; i < nb; i += kThreads) mx = fmaxf(mx, scores[i]);
  mx = block_reduce(mx, sred, true);
  float sum = 0.0f;
  for (int i = tid; i < nb; i += kThreads) {
    const float e = expf(scores[i] - mx);
    scores[i] = e;
    sum += e;
  }
  sum = block_reduce(sum, sred, false);  // its barriers also publish scores[]
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // this thread's V copies have landed
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
#pragma unroll
  for (int u = 0; u < kKeysPerHalfWarp; ++u) {
    const int i = lo + hw + 16 * u;
    if (i < hi) {
      const float e = scores[i - lo];
      if (p0 + i == pp) {
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(e, vcur[hl * 8 + j], acc[j]);
      } else {
        const uint4 vq = *reinterpret_cast<const uint4*>(&vsm[hw + 16 * u][hl * 8]);
        const uint32_t w[4] = {vq.x, vq.y, vq.z, vq.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] = fmaf(e, bf16_lo(w[j]), acc[2 * j]);
          acc[2 * j + 1] = fmaf(e, bf16_hi(w[j]), acc[2 * j + 1]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) red_o[hw][hl * 8 + j] = acc[j];
  __syncthreads();
  if (tid < kDim) {
    float o = 0.0f;
    for (int g = 0; g < 16; ++g) o += red_o[g][tid];
    part.acc[tid] = o;
  }
  if (tid == 0) { part.m = mx; part.l = sum; }
  cluster.sync();  // every block's partial is written
  if (crank == 0 && !bad && tid < kDim) {
    float mm = -INFINITY;
    for (int r = 0; r < kCluster; ++r) mm = fmaxf(mm, cluster.map_shared_rank(&part, r)->m);
    float l = 0.0f, o = 0.0f;
    for (int r = 0; r < kCluster; ++r) {
      const AttnPartial* pr = cluster.map_shared_rank(&part, r);
      if (pr->m == -INFINITY) continue;  // a block with no keys
      const float f = expf(pr->m - mm);
      l += pr->l * f;
      o += pr->acc[tid] * f;
    }
    out[head_off + tid] = f32_to_bf16_bits(o / l);
  }
  cluster.sync();  // keep every block's shared memory alive until block 0 has read it
}

// Absorb: one warp per (stream, row, 4 heads), the 4 key and value rows loaded up front. A key
// row gets the same qk_norm, rotation and bf16 rounding as the window attention's current key, so
// a row absorbed at p equals the row the attention writes at p; a value row is copied.
constexpr int kAbsorbHeads = 4;

__global__ void __launch_bounds__(256)
absorb_kernel(const uint16_t* __restrict__ k_rows, const uint16_t* __restrict__ v_rows,
              const uint16_t* __restrict__ k_gamma, float eps, const RopeTurns turns,
              const int32_t* __restrict__ p0, int n, uint16_t* k_ring, uint16_t* v_ring, int ring,
              int streams, int heads, int32_t* dev_status) {
  const int lane = threadIdx.x & 31;
  const int hgroups = (heads + kAbsorbHeads - 1) / kAbsorbHeads;
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= (int64_t)streams * n * hgroups) return;  // warp-uniform
  const int h0 = (int)(w % hgroups) * kAbsorbHeads;
  const int64_t si = w / hgroups;
  const int i = (int)(si % n);
  const int s = (int)(si / n);
  const int pb = p0[s];
  if (pb < 0 || pb > 2147483647 - (n - 1)) {
    if (i == 0 && h0 == 0 && lane == 0) set_dev_status(dev_status, TFD_ERR_DEVICE_DATA);
    return;
  }
  const int p = pb + i;
  const int64_t src = (((int64_t)s * n + i) * heads + h0) * kDim + 4 * lane;
  const int64_t dst = (((int64_t)s * ring + p % ring) * heads + h0) * kDim + 4 * lane;
  uint2 kraw[kAbsorbHeads], vraw[kAbsorbHeads];
#pragma unroll
  for (int j = 0; j < kAbsorbHeads; ++j) {
    if (h0 + j < heads) {
      kraw[j] = *reinterpret_cast<const uint2*>(k_rows + src + j * kDim);
      vraw[j] = *reinterpret_cast<const uint2*>(v_rows + src + j * kDim);
    }
  }
  float sn[4], cs[4];
  rope_sincos(p, turns, sn, cs);  // one position: the same rotation for every head
#pragma unroll
  for (int j = 0; j < kAbsorbHeads; ++j) {
    if (h0 + j >= heads) break;  // warp-uniform
    float x[4] = {bf16_lo(kraw[j].x), bf16_hi(kraw[j].x), bf16_lo(kraw[j].y), bf16_hi(kraw[j].y)};
    norm_rope_sc(x, k_gamma, eps, sn, cs);
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(x[0]) | ((uint32_t)f32_to_bf16_bits(x[1]) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(x[2]) | ((uint32_t)f32_to_bf16_bits(x[3]) << 16);
    *reinterpret_cast<uint2*>(k_ring + dst + j * kDim) = o;
    *reinterpret_cast<uint2*>(v_ring + dst + j * kDim) = vraw[j];
  }
}

// The turn table of a RoPE base, computed in double on the host (kept for the last base used by
// this thread).
const RopeTurns& rope_turns(float base) {
  thread_local float cached_base = -1.0f;
  thread_local RopeTurns cached;
  if (cached_base != base) {
    const double two_pi = 6.283185307179586476925286766559;
    for (int i = 0; i < kDim / 2; ++i) {
      const double f = std::pow((double)base, -2.0 * i / kDim);
      double turns = f / two_pi;
      turns -= std::floor(turns);
      cached.t[i] = (uint64_t)std::ldexp(turns, 64);
    }
    cached_base = base;
  }
  return cached;
}

}  // namespace

extern "C" tfd_status tfd_window_attn(const void* q, const void* k_new, const void* v_new,
                                      const void* q_gamma, const void* k_gamma, float eps,
                                      float rope_base, const int32_t* pos, void* k_ring,
                                      void* v_ring, int ring, int window, int streams, int heads,
                                      int dim, void* out, int32_t* dev_status, void* stream) {
  using tfd_host::aligned;
  if (!q || !k_new || !v_new || !pos || !k_ring || !v_ring || !out) return TFD_ERR_INVALID;
  if (streams < 1 || streams > 65535 || heads < 1 || heads > 65535) return TFD_ERR_INVALID;
  if (window < 0 || window > TFD_MAX_WINDOW || ring < window + 1) return TFD_ERR_INVALID;
  if (!(eps >= 0.0f) || !(rope_base > 0.0f)) return TFD_ERR_INVALID;
  if (dim != kDim) return TFD_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_ring, 16) ||
      !aligned(v_ring, 16) || !aligned(out, 16) || !aligned(pos, 4))
    return TFD_ERR_INVALID;
  if ((q_gamma && !aligned(q_gamma, 2)) || (k_gamma && !aligned(k_gamma, 2))) return TFD_ERR_INVALID;
  if ((int64_t)heads * 4 > 2147483647) return TFD_ERR_INVALID;
  dim3 grid(heads * 4, streams);
  window_attn_kernel<<<grid, kThreads, 0, tfd_host::as_stream(stream)>>>(
      reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint16_t*>(k_new),
      reinterpret_cast<const uint16_t*>(v_new), reinterpret_cast<const uint16_t*>(q_gamma),
      reinterpret_cast<const uint16_t*>(k_gamma), eps, rope_turns(rope_base), pos,
      reinterpret_cast<uint16_t*>(k_ring), reinterpret_cast<uint16_t*>(v_ring), ring, window,
      heads, reinterpret_cast<uint16_t*>(out), dev_status);
  return tfd_host::launch_status();
}

extern "C" tfd_status tfd_absorb(const void* k_rows, const void* v_rows, const void* k_gamma,
                                 float eps, float rope_base, const int32_t* p0, int n,
                                 void* k_ring, void* v_ring, int ring, int streams, int heads,
                                 int dim, int32_t* dev_status, void* stream) {
  using tfd_host::aligned;
  if (!k_rows || !v_rows || !p0 || !k_ring || !v_ring) return TFD_ERR_INVALID;
  if (streams < 1 || heads < 1 || ring < 1) return TFD_ERR_INVALID;
  if (n < 1 || n > ring) return TFD_ERR_INVALID;  // a span longer than the ring is refused
  if (!(eps >= 0.0f) || !(rope_base > 0.0f)) return TFD_ERR_INVALID;
  if (dim != kDim) return TFD_ERR_UNSUPPORTED;
  if (!aligned(k_rows, 16) || !aligned(v_rows, 16) || !aligned(k_ring, 16) ||
      !aligned(v_ring, 16) || !aligned(p0, 4) || (k_gamma && !aligned(k_gamma, 2)))
    return TFD_ERR_INVALID;
  const int64_t warps = (int64_t)streams * n * ((heads + kAbsorbHeads - 1) / kAbsorbHeads);
  if ((warps + 7) / 8 > 2147483647) return TFD_ERR_INVALID;
  absorb_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, tfd_host::as_stream(stream)>>>(
      reinterpret_cast<const uint16_t*>(k_rows), reinterpret_cast<const uint16_t*>(v_rows),
      reinterpret_cast<const uint16_t*>(k_gamma), eps, rope_turns(rope_base), p0, n,
      reinterpret_cast<uint16_t*>(k_ring), reinterpret_cast<uint16_t*>(v_ring), ring, streams,
      heads, dev_status);
  return tfd_host::launch_status();
}
