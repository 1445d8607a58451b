// layer.cu - the rest of the head layer's row kernels: RMSNorm of hidden rows and SwiGLU.
//
// Follows the TFE draft head page (#42): eagle.cu's row kernels ("RMSNorm, RoPE, window attention,
// SwiGLU, top-1 with confidence"), and the commit that splits eagle.zig (the reference "rounds
// SiLU(g) to bf16 before the multiply").
//
// Both are HBM-bound row sweeps with 16-byte loads and stores. RMSNorm: one block per row; the sum
// of squares is taken per thread over its chunks, then over the warp and over the warps in a fixed
// order, and the row is read again (from L1/L2) to write it. SwiGLU: a grid-stride sweep, eight
// elements per thread and step.
#include "common.cuh"

namespace {

using namespace tfd;

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
rmsnorm_kernel(const uint16_t* __restrict__ x, int64_t ldx, const uint16_t* __restrict__ gamma,
               float eps, int64_t hidden, uint16_t* out, int64_t ldo) {
  __shared__ float swarp[kNormThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint16_t* xr = x + (int64_t)blockIdx.x * ldx;
  uint16_t* orow = out + (int64_t)blockIdx.x * ldo;
  const int64_t chunks = hidden / 8;
  float ss = 0.0f;
  for (int64_t c = tid; c < chunks; c += kNormThreads) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + 8 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) swarp[warp] = ss;
  __syncthreads();  // also: every read of the row is done before any write (in place)
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += swarp[w];
  const float inv = 1.0f / sqrtf(tot / (float)hidden + eps);
  for (int64_t c = tid; c < chunks; c += kNormThreads) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + 8 * c);
    uint4 gv = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);  // bf16 ones
    if (gamma) gv = *reinterpret_cast<const uint4*>(gamma + 8 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint16_t lo = f32_to_bf16_bits(bf16_lo(w[j]) * inv * bf16_lo(gw[j]));
      const uint16_t hi = f32_to_bf16_bits(bf16_hi(w[j]) * inv * bf16_hi(gw[j]));
      o[j] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *reinterpret_cast<uint4*>(orow + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// SiLU in fp32 without overflow: g * sigmoid(g), the exponential taken of -|g|.
__device__ __forceinline__ float silu(float g) {
  const float e = expf(-fabsf(g));
  const float sig = g >= 0.0f ? 1.0f / (1.0f + e) : e / (1.0f + e);
  return g * sig;
}

__global__ void __launch_bounds__(256)
swiglu_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ u, int64_t ld,
              int rows, int64_t cols, uint16_t* out, int64_t ldo) {
  const int64_t per_row = cols / 8;
  const int64_t total = per_row * rows;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row, c = i - r * per_row;
    const uint4 gv = *reinterpret_cast<const uint4*>(g + r * ld + 8 * c);
    const uint4 uv = *reinterpret_cast<const uint4*>(u + r * ld + 8 * c);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // s = bf16(SiLU(g)); s * u is exact in fp32 (8 x 8 significant bits); one rounding to bf16
      const float slo = bf16_bits_to_f32(f32_to_bf16_bits(silu(bf16_lo(gw[j]))));
      const float shi = bf16_bits_to_f32(f32_to_bf16_bits(silu(bf16_hi(gw[j]))));
      o[j] = (uint32_t)f32_to_bf16_bits(slo * bf16_lo(uw[j])) |
             ((uint32_t)f32_to_bf16_bits(shi * bf16_hi(uw[j])) << 16);
    }
    *reinterpret_cast<uint4*>(out + r * ldo + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

extern "C" tfd_status tfd_rmsnorm(const void* x, int64_t ldx, const void* gamma, float eps,
                                  int rows, int64_t hidden, void* out, int64_t ldo,
                                  void* stream) {
  using tfd_host::aligned;
  if (!x || !out) return TFD_ERR_INVALID;
  if (rows < 1 || rows > 2147483647 || hidden < 8 || hidden % 8 != 0) return TFD_ERR_INVALID;
  if (ldx < hidden || ldo < hidden || ldx % 8 != 0 || ldo % 8 != 0) return TFD_ERR_INVALID;
  if (!(eps >= 0.0f)) return TFD_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(out, 16) || (gamma && !aligned(gamma, 16))) return TFD_ERR_INVALID;
  if (out != x) {  // partial overlap is not a supported form of in-place
    const uintptr_t a0 = (uintptr_t)x, a1 = a0 + (uintptr_t)(((rows - 1) * ldx + hidden) * 2);
    const uintptr_t b0 = (uintptr_t)out, b1 = b0 + (uintptr_t)(((rows - 1) * ldo + hidden) * 2);
    if (a0 < b1 && b0 < a1) return TFD_ERR_INVALID;
  } else if (ldx != ldo) {
    return TFD_ERR_INVALID;
  }
  rmsnorm_kernel<<<rows, kNormThreads, 0, tfd_host::as_stream(stream)>>>(
      reinterpret_cast<const uint16_t*>(x), ldx, reinterpret_cast<const uint16_t*>(gamma), eps,
      hidden, reinterpret_cast<uint16_t*>(out), ldo);
  return tfd_host::launch_status();
}

extern "C" tfd_status tfd_swiglu(const void* g, const void* u, int64_t ld, int rows, int64_t cols,
                                 void* out, int64_t ldo, void* stream) {
  using tfd_host::aligned;
  if (!g || !u || !out) return TFD_ERR_INVALID;
  if (rows < 1 || cols < 8 || cols % 8 != 0 || ld < cols || ldo < cols) return TFD_ERR_INVALID;
  if (ld % 8 != 0 || ldo % 8 != 0) return TFD_ERR_INVALID;
  if (!aligned(g, 16) || !aligned(u, 16) || !aligned(out, 16)) return TFD_ERR_INVALID;
  if ((out == g || out == u) && ldo != ld) return TFD_ERR_INVALID;
  const int64_t total = (int64_t)rows * (cols / 8);
  int sms = tfd_host::sm_count();
  if (sms < 1) sms = 1;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  swiglu_kernel<<<(unsigned)blocks, 256, 0, tfd_host::as_stream(stream)>>>(
      reinterpret_cast<const uint16_t*>(g), reinterpret_cast<const uint16_t*>(u), ld, rows, cols,
      reinterpret_cast<uint16_t*>(out), ldo);
  return tfd_host::launch_status();
}
