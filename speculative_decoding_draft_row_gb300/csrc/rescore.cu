// rescore.cu - exact logits of each row's candidates from a dense bf16 head, and their argmax.
//
// Follows the TFE draft head page (#42), commit "... ocabulary head": a two_stage head drafts the
// argmax of the candidates' exact logits from the target's own head, a dense bf16 copy; cand_k is
// 1 to 512. The work is a gather GEMV: one warp per candidate streams its 8 KB head row with
// 16-byte loads and a fixed lane-strided fp32 sum, so a candidate's logit does not depend on where
// it sits in the list; the last block of a row to finish takes the argmax over its blocks' bests.
#include "common.cuh"

namespace {

using namespace tfd;

constexpr int kWarpsPerBlock = 8;
constexpr int kUnroll = 4;

struct RescoreWs {
  uint32_t* counters;  // [rows]
  uint64_t* best;      // [rows][blocks]
};

size_t rescore_ws_layout(int rows, int blocks, char* base, RescoreWs* out) {
  size_t c = tfd_host::round_up((size_t)rows * 4, 256);
  size_t b = tfd_host::round_up((size_t)rows * blocks * 8, 256);
  if (out) {
    out->counters = reinterpret_cast<uint32_t*>(base);
    out->best = reinterpret_cast<uint64_t*>(base + c);
  }
  return c + b;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
rescore_kernel(const uint16_t* __restrict__ w, int64_t vocab, int64_t k,
               const uint16_t* __restrict__ x, const int32_t* __restrict__ cand, int cand_k,
               float* __restrict__ cand_logits, int32_t* __restrict__ out_ids,
               float* __restrict__ out_vals, RescoreWs ws, int32_t* dev_status) {
  __shared__ uint64_t sbest[kWarpsPerBlock];
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y;
  const int j = blockIdx.x * kWarpsPerBlock + warp;
  const uint16_t* xr = x + (int64_t)r * k;
  uint64_t key = 0ull;
  if (j < cand_k) {
    const int32_t c = cand[(int64_t)r * cand_k + j];
    float e;
    if (c < 0 || (int64_t)c >= vocab) {
      e = __uint_as_float(0x7FC00000u);
      set_dev_status(dev_status, TFD_ERR_DEVICE_DATA);
    } else {
      const uint16_t* wr = w + (int64_t)c * k;
      const uint64_t pol = l2_stream_policy();
      float acc = 0.0f;
      int64_t base = (int64_t)lane * 8;
      for (; base + (kUnroll - 1) * 256 < k; base += kUnroll * 256) {
        uint4 wv[kUnroll], xv[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          wv[u] = ldg_stream16(wr + base + u * 256, pol);
          xv[u] = __ldg(reinterpret_cast<const uint4*>(xr + base + u * 256));
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          uint32_t a[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
          uint32_t b[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc = fmaf(bf16_lo(a[i]), bf16_lo(b[i]), acc);
            acc = fmaf(bf16_hi(a[i]), bf16_hi(b[i]), acc);
          }
        }
      }
      for (; base < k; base += 256) {
        uint4 wv = ldg_stream16(wr + base, pol);
        uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr + base));
        uint32_t a[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t b[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc = fmaf(bf16_lo(a[i]), bf16_lo(b[i]), acc);
          acc = fmaf(bf16_hi(a[i]), bf16_hi(b[i]), acc);
        }
      }
      e = warp_sum(acc);
    }
    if (cand_logits && lane == 0) cand_logits[(int64_t)r * cand_k + j] = e;
    key = make_key(e, c);
  }
  if (lane == 0) sbest[warp] = key;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t m = 0ull;
    for (int i = 0; i < kWarpsPerBlock; ++i) m = umax64(m, sbest[i]);
    ws.best[(int64_t)r * gridDim.x + blockIdx.x] = m;
    __threadfence();
    is_last = (atomicAdd(&ws.counters[r], 1u) == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  uint64_t m = 0ull;
  for (unsigned b = threadIdx.x; b < gridDim.x; b += blockDim.x)
    m = umax64(m, __ldcg(ws.best + (int64_t)r * gridDim.x + b));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = umax64(m, shfl_xor_u64(m, o));
  if (lane == 0) sbest[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t mm = 0ull;
    for (int i = 0; i < kWarpsPerBlock; ++i) mm = umax64(mm, sbest[i]);
    out_ids[r] = key_id(mm);
    if (out_vals) out_vals[r] = key_value(mm);
    ws.counters[r] = 0u;  // leave the workspace zeroed
  }
}

}  // namespace

extern "C" size_t tfd_rescore_workspace(int rows, int cand_k) {
  if (rows < 1 || rows > TFD_MAX_ROWS || cand_k < 1 || cand_k > TFD_MAX_TOPK) return 0;
  int blocks = (cand_k + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return rescore_ws_layout(rows, blocks, nullptr, nullptr);
}

extern "C" tfd_status tfd_rescore(const void* w_exact_bf16, int64_t vocab, int64_t k,
                                  const void* x_bf16, int rows, const int32_t* cand, int cand_k,
                                  float* cand_logits, int32_t* out_ids, float* out_vals, void* ws,
                                  size_t ws_bytes, int32_t* dev_status, void* stream) {
  using tfd_host::aligned;
  if (!w_exact_bf16 || !x_bf16 || !cand || !out_ids) return TFD_ERR_INVALID;
  if (vocab < 1 || vocab > (int64_t)INT32_MAX || k < 16 || k % 16 != 0) return TFD_ERR_INVALID;
  if (rows < 1 || rows > TFD_MAX_ROWS || cand_k < 1 || cand_k > TFD_MAX_TOPK) return TFD_ERR_INVALID;
  if (!aligned(w_exact_bf16, 16) || !aligned(x_bf16, 16) || !aligned(cand, 4) ||
      !aligned(out_ids, 4))
    return TFD_ERR_INVALID;
  if ((cand_logits && !aligned(cand_logits, 4)) || (out_vals && !aligned(out_vals, 4)) ||
      (dev_status && !aligned(dev_status, 4)))
    return TFD_ERR_INVALID;
  const int blocks = (cand_k + kWarpsPerBlock - 1) / kWarpsPerBlock;
  RescoreWs w;
  size_t need = rescore_ws_layout(rows, blocks, reinterpret_cast<char*>(ws), &w);
  if (!ws || ws_bytes < need || !aligned(ws, 16)) return TFD_ERR_WORKSPACE;
  dim3 grid(blocks, rows);
  rescore_kernel<<<grid, kWarpsPerBlock * 32, 0, tfd_host::as_stream(stream)>>>(
      reinterpret_cast<const uint16_t*>(w_exact_bf16), vocab, k,
      reinterpret_cast<const uint16_t*>(x_bf16), cand, cand_k, cand_logits, out_ids, out_vals, w,
      dev_status);
  return tfd_host::launch_status();
}
