// quant.cu - FP8 E4M3 codes of a bf16 weight: per-row fp32 scale (amax/448) or E8M0 scales per
// 32x32 block.
//
// Follows the TFE draft head page (#42), update "main3x heads, pass kernels, FP8 linears" (e4m3
// with an fp32 scale a row: scale = row absmax / 448, round to nearest even, from the bf16 weight)
// and the DSpark FP8 head page (#3296), "FP8 draft head" (E4M3 codes with E8M0 scales in 32x32
// blocks, made from the bf16 head at load). The exponent rule of the block scale is the smallest
// power of two that keeps the block's max |w| within 448 (no code saturates).
//
// Numerics: the scale is an IEEE fp32 division and so is each quotient (compiled without fast
// math); the fp32 -> E4M3 step is the hardware's round-to-nearest-even saturating conversion.
#include "common.cuh"

namespace {

using namespace tfd;

// Two floats -> two E4M3 codes (byte 0 = lo, byte 1 = hi), RNE, saturating to +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One warp per row: amax, s = amax / 448, codes = e4m3(w / s). k % 16 == 0.
__global__ void __launch_bounds__(256) quant_row_kernel(const uint16_t* __restrict__ w, int64_t n,
                                                        int64_t k, uint8_t* __restrict__ codes,
                                                        float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= n) return;
  const uint16_t* wr = w + row * k;
  float amax = 0.0f;
  for (int64_t c = (int64_t)lane * 8; c < k; c += 256) {
    uint4 v = *reinterpret_cast<const uint4*>(wr + c);
    uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[i])), fabsf(bf16_hi(u[i]))));
  }
  amax = warp_max(amax);
  const float s = __fdiv_rn(amax, 448.0f);
  if (lane == 0) scales[row] = s;
  uint8_t* cr = codes + row * k;
  for (int64_t c = (int64_t)lane * 8; c < k; c += 256) {
    uint4 v = *reinterpret_cast<const uint4*>(wr + c);
    uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float a0 = bf16_lo(u[2 * i]), a1 = bf16_hi(u[2 * i]);
      float a2 = bf16_lo(u[2 * i + 1]), a3 = bf16_hi(u[2 * i + 1]);
      if (s > 0.0f) {
        a0 = __fdiv_rn(a0, s); a1 = __fdiv_rn(a1, s);
        a2 = __fdiv_rn(a2, s); a3 = __fdiv_rn(a3, s);
      }
      out[i] = e4m3x2(a0, a1) | (e4m3x2(a2, a3) << 16);
    }
    *reinterpret_cast<uint2*>(cr + c) = make_uint2(out[0], out[1]);
  }
}

// Block of 32 rows x 256 columns (8 scale blocks); thread = (row, 32-column block). IL: the codes
// go to the interleaved layout (piece t of block b of 64-column step c at 64c + 16t + 8b).
template <bool IL>
__global__ void __launch_bounds__(256) quant_block_kernel(const uint16_t* __restrict__ w,
                                                          int64_t n, int64_t k,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
  __shared__ float samax[32][9];
  __shared__ uint32_t sbyte[8];
  const int r = threadIdx.x >> 3;   // row within the 32-row block
  const int cb = threadIdx.x & 7;   // 32-column block within the 256 columns
  const int64_t row = (int64_t)blockIdx.y * 32 + r;
  const int64_t col0 = (int64_t)blockIdx.x * 256 + cb * 32;
  const bool active = col0 < k;
  uint32_t u[16];
  float amax = 0.0f;
  if (active) {
    const uint4* p = reinterpret_cast<const uint4*>(w + row * k + col0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 v = p[i];
      u[4 * i] = v.x; u[4 * i + 1] = v.y; u[4 * i + 2] = v.z; u[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[i])), fabsf(bf16_hi(u[i]))));
  }
  samax[r][cb] = amax;
  __syncthreads();
  if (threadIdx.x < 8) {
    float m = 0.0f;
    for (int i = 0; i < 32; ++i) m = fmaxf(m, samax[i][threadIdx.x]);
    // smallest e with m <= 448 * 2^e: with m = f * 2^E (1 <= f < 2), e = E - 8 + (f > 1.75).
    uint32_t b = __float_as_uint(m);
    uint32_t ef = b >> 23;
    int byte = 0;
    if (m > 0.0f && ef != 0u) {
      int e = (int)ef - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
      byte = e + 127;
      byte = byte < 0 ? 0 : (byte > 254 ? 254 : byte);
    }
    sbyte[threadIdx.x] = (uint32_t)byte;
    const int64_t kb = (int64_t)blockIdx.x * 8 + threadIdx.x;
    if (kb * 32 < k) scales[(int64_t)blockIdx.y * (k >> 5) + kb] = (uint8_t)byte;
  }
  __syncthreads();
  if (!active) return;
  // 2^-(byte - 127) as an fp32 (2^-127 is the subnormal 0x00400000).
  const uint32_t byte = sbyte[cb];
  const float inv = byte == 254u ? __uint_as_float(0x00400000u) : __uint_as_float((254u - byte) << 23);
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a0 = bf16_lo(u[2 * i]) * inv, a1 = bf16_hi(u[2 * i]) * inv;
    float a2 = bf16_lo(u[2 * i + 1]) * inv, a3 = bf16_hi(u[2 * i + 1]) * inv;
    out[i] = e4m3x2(a0, a1) | (e4m3x2(a2, a3) << 16);
  }
  if (IL) {
    uint8_t* rp = codes + row * k + (col0 & ~(int64_t)63) + 8 * ((col0 >> 5) & 1);
#pragma unroll
    for (int t = 0; t < 4; ++t)
      *reinterpret_cast<uint2*>(rp + 16 * t) = make_uint2(out[2 * t], out[2 * t + 1]);
  } else {
    uint4* cp = reinterpret_cast<uint4*>(codes + row * k + col0);
    cp[0] = make_uint4(out[0], out[1], out[2], out[3]);
    cp[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

// One thread per 16 bytes of interleaved layout: piece t of 64-column step c, i.e. plain bytes
// 64c + 8t .. +8 (block 0) and 64c + 32 + 8t .. +8 (block 1).
__global__ void __launch_bounds__(256) relayout_kernel(const uint8_t* __restrict__ in, int64_t n,
                                                       int64_t k, bool to_il,
                                                       uint8_t* __restrict__ out) {
  const int64_t per_row = k / 16;
  const int64_t total = n * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / per_row, q = i - row * per_row;
    const int64_t c = q >> 2, t = q & 3;
    const int64_t il = row * k + 64 * c + 16 * t;
    const int64_t p0 = row * k + 64 * c + 8 * t, p1 = p0 + 32;
    if (to_il) {
      const uint2 a = *reinterpret_cast<const uint2*>(in + p0);
      const uint2 b = *reinterpret_cast<const uint2*>(in + p1);
      *reinterpret_cast<uint4*>(out + il) = make_uint4(a.x, a.y, b.x, b.y);
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(in + il);
      *reinterpret_cast<uint2*>(out + p0) = make_uint2(v.x, v.y);
      *reinterpret_cast<uint2*>(out + p1) = make_uint2(v.z, v.w);
    }
  }
}

}  // namespace

extern "C" tfd_status tfd_quant_fp8(const void* w_bf16, int64_t n, int64_t k, int mode,
                                    uint8_t* codes, void* scales, void* stream) {
  using tfd_host::aligned;
  if (!w_bf16 || !codes || !scales) return TFD_ERR_INVALID;
  if (n < 1 || k < 16 || k % 16 != 0) return TFD_ERR_INVALID;
  if (!aligned(w_bf16, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return TFD_ERR_INVALID;
  cudaStream_t s = tfd_host::as_stream(stream);
  if (mode == TFD_W_FP8_ROW) {
    dim3 grid((unsigned)((n + 7) / 8));
    quant_row_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint16_t*>(w_bf16), n, k, codes,
                                         reinterpret_cast<float*>(scales));
    return tfd_host::launch_status();
  }
  if (mode == TFD_W_FP8_BLOCK32 || mode == TFD_W_FP8_BLOCK32_IL) {
    const bool il = mode == TFD_W_FP8_BLOCK32_IL;
    if (n % 32 != 0 || k % (il ? 64 : 32) != 0 || n / 32 > 65535) return TFD_ERR_INVALID;
    dim3 grid((unsigned)((k + 255) / 256), (unsigned)(n / 32));
    auto kern = il ? quant_block_kernel<true> : quant_block_kernel<false>;
    kern<<<grid, 256, 0, s>>>(reinterpret_cast<const uint16_t*>(w_bf16), n, k, codes,
                              reinterpret_cast<uint8_t*>(scales));
    return tfd_host::launch_status();
  }
  return TFD_ERR_INVALID;
}

extern "C" tfd_status tfd_fp8_block32_relayout(const uint8_t* in, int64_t n, int64_t k,
                                               int to_interleaved, uint8_t* out, void* stream) {
  using tfd_host::aligned;
  if (!in || !out || n < 1 || k < 64 || k % 64 != 0) return TFD_ERR_INVALID;
  if (to_interleaved != 0 && to_interleaved != 1) return TFD_ERR_INVALID;
  if (!aligned(in, 16) || !aligned(out, 16)) return TFD_ERR_INVALID;
  const uintptr_t a = (uintptr_t)in, b = (uintptr_t)out, len = (uintptr_t)(n * k);
  if (a < b + len && b < a + len) return TFD_ERR_INVALID;
  const int64_t total = n * (k / 16);
  int sms = tfd_host::sm_count();
  if (sms < 1) sms = 1;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
  relayout_kernel<<<(unsigned)blocks, 256, 0, tfd_host::as_stream(stream)>>>(
      in, n, k, to_interleaved == 1, out);
  return tfd_host::launch_status();
}
