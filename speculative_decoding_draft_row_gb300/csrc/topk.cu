// topk.cu - split top-k over given fp32 logits: each (row, part) block stages a contiguous range
// of 8192 keys in shared memory and selects its top k there; the last block of a row to finish
// stages the union of the parts' lists in shared memory and selects the row's top k from it. A
// selection is one histogram pass to a boundary bin, a gather of the keys at or above it, and a
// rank count (each key's rank is the number of keys that beat it: the rank-count top-k of the
// subset page (#1011), "tf_super_topk_few").
//
// Follows the TFE draft head page (#42): commit "... ocabulary head" (top cand_k of fp32 logits,
// 1..512, a tie at the k-th value going to the lower token id; the top-1 through an id map) and
// commit "pass kernels and FP8 linears" (a vocabulary row scanned in parts and joined).
#include "select.cuh"

namespace {

using namespace tfd;

constexpr int kCap = 16384;  // keys a block holds in shared memory (a part, or the join's union)
constexpr int kPartLen = 8192;  // keys per part

struct TopkPlan {
  int parts;
  int64_t chunk;
  int64_t cap;  // shared-memory keys per block: max(chunk, parts * k), or chunk when the union
                // does not fit (then the join reads the lists from global memory)
};

// Parts per row: n / 8192 (at least 1), fewer when the join's union of part lists (parts * k
// keys) would not fit in shared memory. Independent of the device.
TopkPlan topk_plan(int rows, int64_t n, int k) {
  (void)rows;
  int64_t p = (n + kPartLen - 1) / kPartLen;
  int64_t by_join = kCap / k;
  if (p > by_join) p = by_join;
  int64_t need = (n + kCap - 1) / kCap;
  if (p < need) p = need;
  if (p < 1) p = 1;
  int64_t chunk = (n + p - 1) / p;
  p = (n + chunk - 1) / chunk;
  int64_t uni = p * k;
  int64_t cap = uni <= kCap ? (uni > chunk ? uni : chunk) : chunk;
  return TopkPlan{(int)p, chunk, cap};
}

struct TopkWs {
  uint32_t* counters;  // [rows]
  int* counts;         // [rows][parts]  keys each part kept
  uint64_t* keys;      // [rows][parts][k], each part's list sorted descending
};

size_t topk_ws_layout(int rows, int parts, int k, char* base, TopkWs* out) {
  size_t c_bytes = tfd_host::round_up((size_t)rows * 4, 256);
  size_t n_bytes = tfd_host::round_up((size_t)rows * parts * 4, 256);
  size_t k_bytes = tfd_host::round_up((size_t)rows * parts * k * 8, 256);
  if (out) {
    out->counters = reinterpret_cast<uint32_t*>(base);
    out->counts = reinterpret_cast<int*>(base + c_bytes);
    out->keys = reinterpret_cast<uint64_t*>(base + c_bytes + n_bytes);
  }
  return c_bytes + n_bytes + k_bytes;
}

size_t topk_smem_fixed() { return sizeof(SelectSmem) + sizeof(FastSelectSmem) + 16; }
size_t topk_smem_bytes(const TopkPlan& pl) { return topk_smem_fixed() + (size_t)pl.cap * 8; }

__device__ __forceinline__ size_t topk_smem_fixed_dev() {
  return sizeof(SelectSmem) + sizeof(FastSelectSmem) + 16;
}

__global__ void __launch_bounds__(kSelectThreads)
topk_kernel(const float* __restrict__ logits, int64_t n, int64_t ld, int k,
            const int32_t* __restrict__ id_map, float* __restrict__ vals,
            int32_t* __restrict__ ids, int64_t ld_out, TopkWs ws, int parts, int64_t chunk,
            int64_t cap) {
  extern __shared__ __align__(16) unsigned char tk_smem[];
  SelectSmem& sel = *reinterpret_cast<SelectSmem*>(tk_smem);
  FastSelectSmem& fs = *reinterpret_cast<FastSelectSmem*>(tk_smem + sizeof(SelectSmem));
  int* is_last = reinterpret_cast<int*>(tk_smem + sizeof(SelectSmem) + sizeof(FastSelectSmem));
  uint64_t* keys = reinterpret_cast<uint64_t*>(tk_smem + topk_smem_fixed_dev());
  const int tid = threadIdx.x;
  const int p = blockIdx.x;
  const int r = blockIdx.y;
  const int64_t lo = (int64_t)p * chunk;
  const int64_t hi = lo + chunk < n ? lo + chunk : n;
  const int cnt = hi > lo ? (int)(hi - lo) : 0;  // <= cap by the plan
  const float* row = logits + (int64_t)r * ld;

  // ---- part: stage its keys in shared memory, select its top kk, publish the sorted list ----
  // 8 independent loads in flight per thread before any store
  for (int i0 = tid; i0 < cnt; i0 += 8 * kSelectThreads) {
    float v[8];
    int32_t id[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kSelectThreads;
      const int64_t j = lo + (i < cnt ? i : 0);
      v[u] = row[j];
      id[u] = id_map ? id_map[j] : (int32_t)j;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kSelectThreads;
      if (i < cnt) keys[i] = make_key(v[u], id[u]);
    }
  }
  const int kk = cnt < k ? cnt : k;
  block_topk_fast(cnt, k, keys, sel.out, fs, sel);
  uint64_t* dst = ws.keys + ((int64_t)r * parts + p) * k;
  for (int i = tid; i < kk; i += kSelectThreads) dst[i] = sel.out[i];
  if (tid == 0) ws.counts[r * parts + p] = kk;
  __threadfence();
  __syncthreads();
  if (tid == 0) *is_last = (atomicAdd(&ws.counters[r], 1u) == (uint32_t)(parts - 1));
  __syncthreads();
  if (!*is_last) return;
  __threadfence();

  // ---- join: the row's top k is the top k of the union of the parts' lists ----
  const uint64_t* rowkeys = ws.keys + (int64_t)r * parts * k;
  const int* rowcounts = ws.counts + r * parts;
  const int uni = parts * k;
  __syncthreads();
  if ((int64_t)uni <= cap) {
    for (int i0 = tid; i0 < uni; i0 += 8 * kSelectThreads) {
      uint64_t kv[8];
      int cq[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kSelectThreads;
        const int ii = i < uni ? i : 0;
        kv[u] = __ldcg(rowkeys + ii);
        cq[u] = __ldcg(rowcounts + ii / k);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kSelectThreads;
        if (i < uni) keys[i] = (i % k) < cq[u] ? kv[u] : 0ull;
      }
    }
    block_topk_fast(uni, k, keys, sel.out, fs, sel);
  } else {
    auto join_key = [&](int i) -> uint64_t {
      const int q = i / k;
      return (i - q * k) < __ldcg(rowcounts + q) ? __ldcg(rowkeys + i) : 0ull;
    };
    block_select_topk(uni, k, join_key, sel);
  }
  for (int i = tid; i < k; i += kSelectThreads) {
    vals[(int64_t)r * ld_out + i] = key_value(sel.out[i]);
    ids[(int64_t)r * ld_out + i] = key_id(sel.out[i]);
  }
  if (tid == 0) ws.counters[r] = 0u;  // leave the workspace counters at zero
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
  const size_t smem = topk_smem_bytes(pl);
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(topk_smem_fixed() + (size_t)kCap * 8)) != cudaSuccess)
    return TFD_ERR_CUDA;
  dim3 grid(pl.parts, rows);
  topk_kernel<<<grid, kSelectThreads, smem, stream>>>(logits, n, ld, k, id_map, vals, ids, ld_out,
                                                      w, pl.parts, pl.chunk, pl.cap);
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
