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
// One block per (head, stream): its 512 keys x 128 dims of K and V (256 KB) are read once with
// 16-byte loads, half a warp per key row.
#include "common.cuh"

namespace {

using namespace tfd;

constexpr int kDim = 128;
constexpr int kThreads = 256;
constexpr int kMaxKeys = TFD_MAX_WINDOW + 1;

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

// Lane l of a warp holds elements 4l..4l+3 of a 128-vector: RMSNorm with gamma, then RoPE.
__device__ __forceinline__ void norm_rope(float (&x)[4], const uint16_t* gamma, float eps, int p,
                                          float base) {
  const int lane = threadIdx.x & 31;
  float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / (float)kDim + eps);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float gm = gamma ? bf16_bits_to_f32(gamma[4 * lane + j]) : 1.0f;
    x[j] = x[j] * inv * gm;
  }
  float other[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) other[j] = __shfl_xor_sync(0xffffffffu, x[j], 16);
  const bool first_half = lane < 16;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * (lane & 15) + j;  // pair index 0..63
    const double ang = (double)p * pow((double)base, -2.0 * (double)i / (double)kDim);
    double sd, cd;
    sincos(ang, &sd, &cd);
    const float c = (float)cd, s = (float)sd;
    // first half holds a = x[i] (partner b = x[i+64]); second half holds b (partner a).
    x[j] = first_half ? (x[j] * c - other[j] * s) : (other[j] * s + x[j] * c);
  }
}

__global__ void __launch_bounds__(kThreads)
window_attn_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k_new,
                   const uint16_t* __restrict__ v_new, const uint16_t* __restrict__ q_gamma,
                   const uint16_t* __restrict__ k_gamma, float eps, float rope_base,
                   const int32_t* __restrict__ pos, uint16_t* k_ring, uint16_t* v_ring, int ring,
                   int window, int heads, uint16_t* __restrict__ out, int32_t* dev_status) {
  __shared__ float qn[kDim];
  __shared__ float scores[kMaxKeys];
  __shared__ float sred[kThreads / 32];
  __shared__ float red_o[16][kDim];
  const int h = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p = pos[s];
  if (p < 0) {
    if (tid == 0) set_dev_status(dev_status, TFD_ERR_DEVICE_DATA);
    return;
  }
  const int slot = p % ring;
  const int64_t head_off = ((int64_t)s * heads + h) * kDim;
  const int64_t ring_row = (((int64_t)s * ring + slot) * heads + h) * kDim;

  if (warp < 2) {
    const uint16_t* src = (warp == 0 ? q : k_new) + head_off + 4 * lane;
    uint2 raw = *reinterpret_cast<const uint2*>(src);
    float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    norm_rope(x, warp == 0 ? q_gamma : k_gamma, eps, p, rope_base);
    if (warp == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) qn[4 * lane + j] = x[j];
    } else {
      uint2 o;
      o.x = f32_to_bf16_bits(x[0]) | ((uint32_t)f32_to_bf16_bits(x[1]) << 16);
      o.y = f32_to_bf16_bits(x[2]) | ((uint32_t)f32_to_bf16_bits(x[3]) << 16);
      *reinterpret_cast<uint2*>(k_ring + ring_row + 4 * lane) = o;
    }
  } else if (warp == 2) {
    *reinterpret_cast<uint2*>(v_ring + ring_row + 4 * lane) =
        *reinterpret_cast<const uint2*>(v_new + head_off + 4 * lane);
  }
  __syncthreads();

  const int p0 = p - window > 0 ? p - window : 0;
  const int nk = p - p0 + 1;
  const int hw = tid >> 4, hl = tid & 15;  // half-warp per key, 8 dims per lane
  float qv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) qv[j] = qn[hl * 8 + j];
  const float inv_sqrt_d = 1.0f / sqrtf((float)kDim);
  // Trip counts depend on nk only, so both halves of a warp run the same iterations (the
  // half-warp shuffles below need the whole warp).
  for (int ib = 0; ib < nk; ib += 16 * 4) {
    const int i0 = ib + hw;
    uint4 kv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + 16 * u;
      if (i < nk) {
        const int sl = (p0 + i) % ring;
        kv[u] = *reinterpret_cast<const uint4*>(
            k_ring + (((int64_t)s * ring + sl) * heads + h) * kDim + hl * 8);
      } else {
        kv[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint32_t w[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
      float d = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        d = fmaf(qv[2 * j], bf16_lo(w[j]), d);
        d = fmaf(qv[2 * j + 1], bf16_hi(w[j]), d);
      }
#pragma unroll
      for (int m = 8; m > 0; m >>= 1) d += __shfl_xor_sync(0xffffffffu, d, m);
      const int i = i0 + 16 * u;
      if (hl == 0 && i < nk) scores[i] = d * inv_sqrt_d;
    }
  }
  __syncthreads();
  float mx = -INFINITY;
  for (int i = tid; i < nk; i += kThreads) mx = fmaxf(mx, scores[i]);
  mx = block_reduce(mx, sred, true);
  float sum = 0.0f;
  for (int i = tid; i < nk; i += kThreads) {
    float e = expf(scores[i] - mx);
    scores[i] = e;
    sum += e;
  }
  sum = block_reduce(sum, sred, false);  // its first barrier also publishes scores[]

  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  for (int ib = 0; ib < nk; ib += 16 * 4) {
    const int i0 = ib + hw;
    uint4 vv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + 16 * u;
      if (i < nk) {
        const int sl = (p0 + i) % ring;
        vv[u] = *reinterpret_cast<const uint4*>(
            v_ring + (((int64_t)s * ring + sl) * heads + h) * kDim + hl * 8);
      } else {
        vv[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + 16 * u;
      const float e = i < nk ? scores[i] : 0.0f;
      uint32_t w[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[2 * j] = fmaf(e, bf16_lo(w[j]), acc[2 * j]);
        acc[2 * j + 1] = fmaf(e, bf16_hi(w[j]), acc[2 * j + 1]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) red_o[hw][hl * 8 + j] = acc[j];
  __syncthreads();
  if (tid < kDim) {
    float o = 0.0f;
    for (int g = 0; g < 16; ++g) o += red_o[g][tid];
    out[((int64_t)s * heads + h) * kDim + tid] = f32_to_bf16_bits(o / sum);
  }
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
  dim3 grid(heads, streams);
  window_attn_kernel<<<grid, kThreads, 0, tfd_host::as_stream(stream)>>>(
      reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint16_t*>(k_new),
      reinterpret_cast<const uint16_t*>(v_new), reinterpret_cast<const uint16_t*>(q_gamma),
      reinterpret_cast<const uint16_t*>(k_gamma), eps, rope_base, pos,
      reinterpret_cast<uint16_t*>(k_ring), reinterpret_cast<uint16_t*>(v_ring), ring, window,
      heads, reinterpret_cast<uint16_t*>(out), dev_status);
  return tfd_host::launch_status();
}
