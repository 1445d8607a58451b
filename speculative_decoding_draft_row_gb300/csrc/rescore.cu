// rescore.cu - exact logits of each row's candidates from a dense bf16 head, and their argmax.
//
// Follows the TFE draft head page (#42), commit "... ocabulary head": a two_stage head drafts the
// argmax of the candidates' exact logits from the target's own head, a dense bf16 copy; cand_k is
// 1 to 512. The work is a gather GEMV: one warp per candidate streams its 8 KB head row with
// 16-byte loads (a whole 4096-element chunk of them in flight, the row's activations in shared
// memory) and a fixed lane-strided fp32 sum, so a candidate's logit does not depend on where it
// sits in the list; the last block of a row to finish takes the argmax over its blocks' bests.
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

// Rows up to this width keep the activation row in shared memory (the block's 8 warps score 8
// candidates of one row) and issue a whole chunk of kChunk 16-byte weight loads per lane at once.
constexpr int64_t kSmemK = 16384;
constexpr int kChunk = 16;

// One candidate's dot product with the shared-memory activation row: kChunk loads a lane in flight
// (4096 elements a warp), then the fixed lane-strided fp32 sum, in the same order as the
// global-memory form below (element base + 256 u of lane l, u ascending), so both forms give the
// same bits.
__device__ __forceinline__ float dot_smem_x(const uint16_t* __restrict__ wr, const uint16_t* xs,
                                            int64_t k, int lane, uint64_t pol) {
  float acc = 0.0f;
  for (int64_t c0 = 0; c0 < k; c0 += (int64_t)kChunk * 256) {  // warp-uniform
    uint4 wv[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int64_t e = c0 + (int64_t)u * 256 + lane * 8;
      wv[u] = e < k ? ldg_stream16(wr + e, pol) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int64_t e = c0 + (int64_t)u * 256 + lane * 8;
      if (e < k) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + e);
        const uint32_t a[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
        const uint32_t b[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc = fmaf(bf16_lo(a[i]), bf16_lo(b[i]), acc);
          acc = fmaf(bf16_hi(a[i]), bf16_hi(b[i]), acc);
        }
      }
    }
  }
  return acc;
}

template <bool SMEM_X>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
rescore_kernel(const uint16_t* __restrict__ w, int64_t vocab, int64_t k,
               const uint16_t* __restrict__ x, const int32_t* __restrict__ cand, int cand_k,
               float* __restrict__ cand_logits, int32_t* __restrict__ out_ids,
               float* __restrict__ out_vals, RescoreWs ws, int32_t* dev_status) {
  extern __shared__ __align__(16) uint16_t xs_dyn[];
  __shared__ uint64_t sbest[kWarpsPerBlock];
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y;
  const int j = blockIdx.x * kWarpsPerBlock + warp;
  const uint16_t* xr = x + (int64_t)r * k;
  int32_t c = 0;
  if (j < cand_k) c = cand[(int64_t)r * cand_k + j];  // issued before the activations are staged
  if (SMEM_X) {
    for (int64_t e = (int64_t)threadIdx.x * 8; e < k; e += kWarpsPerBlock * 32 * 8)
      *reinterpret_cast<uint4*>(xs_dyn + e) = __ldg(reinterpret_cast<const uint4*>(xr + e));
    __syncthreads();
  }
  uint64_t key = 0ull;
  if (j < cand_k) {
    float e;
    if (c < 0 || (int64_t)c >= vocab) {
      e = __uint_as_float(0x7FC00000u);
      set_dev_status(dev_status, TFD_ERR_DEVICE_DATA);
    } else if (SMEM_X) {
      e = warp_sum(dot_smem_x(w + (int64_t)c * k, xs_dyn, k, lane, l2_stream_policy()));
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
  if (k <= kSmemK) {
    const size_t smem = (size_t)k * 2;
    if (cudaFuncSetAttribute(rescore_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kSmemK * 2)) != cudaSuccess)
      return TFD_ERR_CUDA;
    rescore_kernel<true><<<grid, kWarpsPerBlock * 32, smem, tfd_host::as_stream(stream)>>>(
        reinterpret_cast<const uint16_t*>(w_exact_bf16), vocab, k,
        reinterpret_cast<const uint16_t*>(x_bf16), cand, cand_k, cand_logits, out_ids, out_vals,
        w, dev_status);
    return tfd_host::launch_status();
  }
  rescore_kernel<false><<<grid, kWarpsPerBlock * 32, 0, tfd_host::as_stream(stream)>>>(
      reinterpret_cast<const uint16_t*>(w_exact_bf16), vocab, k,
      reinterpret_cast<const uint16_t*>(x_bf16), cand, cand_k, cand_logits, out_ids, out_vals, w,
      dev_status);
  return tfd_host::launch_status();
}
