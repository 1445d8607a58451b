// topk.cu - split top-k over given fp32 logits: each (row, part) block keeps the exact top-k of a
// contiguous range, and the last block of a row to finish joins the parts' lists.
//
// Follows the TFE draft head page (#42): commit "... ocabulary head" (top cand_k of fp32 logits,
// 1..512, a tie at the k-th value going to the lower token id; the top-1 through an id map) and
// commit "pass kernels and FP8 linears" (a vocabulary row scanned in parts and joined).
#include "select.cuh"

namespace {

using namespace tfd;

struct TopkPlan {
  int parts;
  int64_t chunk;
};

// Parts per row: enough blocks to fill the GPU (about 320 in all), each part at least
// max(4k, 1024) long, and at most 16384 keys for the join. Independent of the device.
TopkPlan topk_plan(int rows, int64_t n, int k) {
  int64_t p = (320 + rows - 1) / rows;
  int64_t min_len = 4LL * k > 1024 ? 4LL * k : 1024;
  int64_t by_len = n / min_len;
  if (by_len < 1) by_len = 1;
  if (p > by_len) p = by_len;
  int64_t by_join = 16384 / k;
  if (by_join < 1) by_join = 1;
  if (p > by_join) p = by_join;
  if (p < 1) p = 1;
  int64_t chunk = (n + p - 1) / p;
  p = (n + chunk - 1) / chunk;
  return TopkPlan{(int)p, chunk};
}

struct TopkWs {
  uint32_t* counters;  // [rows]
  int* counts;         // [rows][parts]
  uint64_t* keys;      // [rows][parts][k]
};

size_t topk_ws_layout(int rows, int parts, int k, char* base, TopkWs* out) {
  size_t off = 0;
  size_t c_bytes = tfd_host::round_up((size_t)rows * 4, 256);
  size_t n_bytes = tfd_host::round_up((size_t)rows * parts * 4, 256);
  size_t k_bytes = tfd_host::round_up((size_t)rows * parts * k * 8, 256);
  if (out) {
    out->counters = reinterpret_cast<uint32_t*>(base + off);
    out->counts = reinterpret_cast<int*>(base + off + c_bytes);
    out->keys = reinterpret_cast<uint64_t*>(base + off + c_bytes + n_bytes);
  }
  return c_bytes + n_bytes + k_bytes;
}

__global__ void __launch_bounds__(kSelectThreads)
topk_kernel(const float* __restrict__ logits, int64_t n, int64_t ld, int k,
            const int32_t* __restrict__ id_map, float* __restrict__ vals,
            int32_t* __restrict__ ids, int64_t ld_out, TopkWs ws, int parts, int64_t chunk) {
  __shared__ SelectSmem sm;
  __shared__ int is_last;
  const int tid = threadIdx.x;
  const int p = blockIdx.x;
  const int r = blockIdx.y;
  const int64_t lo = (int64_t)p * chunk;
  const int64_t hi = lo + chunk < n ? lo + chunk : n;
  const int cnt = hi > lo ? (int)(hi - lo) : 0;
  const float* row = logits + (int64_t)r * ld;

  auto part_key = [&](int i) -> uint64_t {
    int64_t j = lo + i;
    return make_key(row[j], id_map ? id_map[j] : (int32_t)j);
  };
  block_select_topk(cnt, k, part_key, sm);
  const int kk = cnt < k ? cnt : k;
  uint64_t* dst = ws.keys + ((int64_t)r * parts + p) * k;
  for (int i = tid; i < kk; i += kSelectThreads) dst[i] = sm.out[i];
  if (tid == 0) ws.counts[r * parts + p] = kk;
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(&ws.counters[r], 1u) == (uint32_t)(parts - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  const uint64_t* rowkeys = ws.keys + (int64_t)r * parts * k;
  const int* rowcounts = ws.counts + r * parts;
  auto join_key = [&](int i) -> uint64_t {
    int q = i / k;
    int j = i - q * k;
    return j < __ldcg(rowcounts + q) ? __ldcg(rowkeys + i) : 0ull;
  };
  block_select_topk(parts * k, k, join_key, sm);
  for (int i = tid; i < k; i += kSelectThreads) {
    vals[(int64_t)r * ld_out + i] = key_value(sm.out[i]);
    ids[(int64_t)r * ld_out + i] = key_id(sm.out[i]);
  }
  if (tid == 0) ws.counters[r] = 0u;  // leave the workspace zeroed
}

}  // namespace

namespace tfd_internal {

size_t topk_workspace(int rows, int64_t n, int k) {
  if (rows < 1 || n < 1 || k < 1 || k > TFD_MAX_TOPK || k > n) return 0;
  TopkPlan pl = topk_plan(rows, n, k);
  return topk_ws_layout(rows, pl.parts, k, nullptr, nullptr);
}

tfd_status topk_launch(const float* logits, int rows, int64_t n, int64_t ld, int k,
                       const int32_t* id_map, float* vals, int32_t* ids, int64_t ld_out, void* ws,
                       size_t ws_bytes, cudaStream_t stream) {
  TopkPlan pl = topk_plan(rows, n, k);
  TopkWs w;
  size_t need = topk_ws_layout(rows, pl.parts, k, reinterpret_cast<char*>(ws), &w);
  if (ws == nullptr || ws_bytes < need) return TFD_ERR_WORKSPACE;
  dim3 grid(pl.parts, rows);
  topk_kernel<<<grid, kSelectThreads, 0, stream>>>(logits, n, ld, k, id_map, vals, ids, ld_out,
                                                   w, pl.parts, pl.chunk);
  return tfd_host::launch_status();
}

}  // namespace tfd_internal

extern "C" size_t tfd_topk_workspace(int rows, int64_t n, int k) {
  return tfd_internal::topk_workspace(rows, n, k);
}

extern "C" tfd_status tfd_topk(const float* logits, int rows, int64_t n, int64_t ld, int k,
                               const int32_t* id_map, float* vals, int32_t* ids, void* ws,
                               size_t ws_bytes, void* stream) {
  using tfd_host::aligned;
  if (!logits || !vals || !ids) return TFD_ERR_INVALID;
  if (rows < 1 || rows > 65535 || n < 1 || n > (int64_t)INT32_MAX || ld < n) return TFD_ERR_INVALID;
  if (k < 1 || k > TFD_MAX_TOPK || k > n) return TFD_ERR_INVALID;
  if (!aligned(logits, 4) || !aligned(vals, 4) || !aligned(ids, 4)) return TFD_ERR_INVALID;
  if (id_map && !aligned(id_map, 4)) return TFD_ERR_INVALID;
  if (ws && !aligned(ws, 16)) return TFD_ERR_INVALID;
  return tfd_internal::topk_launch(logits, rows, n, ld, k, id_map, vals, ids, k, ws, ws_bytes,
                                   tfd_host::as_stream(stream));
}
