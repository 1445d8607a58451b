// topk.cu - split top-k over given fp32 logits: each (row, part) block keeps the exact top-k of a
// contiguous range, and the last block of a row to finish joins the parts' lists.
//
// Follows the TFE draft head page (#42): commit "... ocabulary head" (top cand_k of fp32 logits,
// 1..512, a tie at the k-th value going to the lower token id; the top-1 through an id map) and
// commit "pass kernels and FP8 linears" (a vocabulary row scanned in parts and joined).
#include "select.cuh"

namespace {

using namespace tfd;

constexpr int kStage = 4096;  // keys a block holds in shared memory (part length cap)

struct TopkPlan {
  int parts;
  int64_t chunk;
};

// Parts per row: at least n / 4096 (a part fits in shared memory), and about 320 blocks in all
// when the row is long enough for parts of max(4k, 1024). Independent of the device.
TopkPlan topk_plan(int rows, int64_t n, int k) {
  int64_t want = (320 + rows - 1) / rows;
  int64_t min_len = 4LL * k > 1024 ? 4LL * k : 1024;
  int64_t by_len = n / min_len;
  if (want > by_len) want = by_len;
  int64_t need = (n + kStage - 1) / kStage;
  int64_t p = want > need ? want : need;
  if (p < 1) p = 1;
  int64_t chunk = (n + p - 1) / p;
  p = (n + chunk - 1) / chunk;
  return TopkPlan{(int)p, chunk};
}

struct TopkWs {
  uint32_t* counters;  // [rows]
  int* counts;         // [rows][parts]  keys each part kept
  uint64_t* kth;       // [rows][parts]  the part's k-th key (0 when it kept fewer than k)
  uint64_t* keys;      // [rows][parts][k], each part's list sorted descending
};

size_t topk_ws_layout(int rows, int parts, int k, char* base, TopkWs* out) {
  size_t c_bytes = tfd_host::round_up((size_t)rows * 4, 256);
  size_t n_bytes = tfd_host::round_up((size_t)rows * parts * 4, 256);
  size_t t_bytes = tfd_host::round_up((size_t)rows * parts * 8, 256);
  size_t k_bytes = tfd_host::round_up((size_t)rows * parts * k * 8, 256);
  if (out) {
    out->counters = reinterpret_cast<uint32_t*>(base);
    out->counts = reinterpret_cast<int*>(base + c_bytes);
    out->kth = reinterpret_cast<uint64_t*>(base + c_bytes + n_bytes);
    out->keys = reinterpret_cast<uint64_t*>(base + c_bytes + n_bytes + t_bytes);
  }
  return c_bytes + n_bytes + t_bytes + k_bytes;
}

struct TopkSmem {
  SelectSmem sel;
  uint64_t keys[kStage];
  uint64_t red[kSelectThreads / 32];
  int scan[kSelectThreads / 32];
  int total;
  int is_last;
};

__global__ void __launch_bounds__(kSelectThreads)
topk_kernel(const float* __restrict__ logits, int64_t n, int64_t ld, int k,
            const int32_t* __restrict__ id_map, float* __restrict__ vals,
            int32_t* __restrict__ ids, int64_t ld_out, TopkWs ws, int parts, int64_t chunk) {
  __shared__ TopkSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int p = blockIdx.x;
  const int r = blockIdx.y;
  const int64_t lo = (int64_t)p * chunk;
  const int64_t hi = lo + chunk < n ? lo + chunk : n;
  const int cnt = hi > lo ? (int)(hi - lo) : 0;  // <= kStage by the plan
  const float* row = logits + (int64_t)r * ld;

  // ---- part: stage its keys in shared memory, select, publish the sorted list and its k-th ----
  for (int i = tid; i < cnt; i += kSelectThreads) {
    const int64_t j = lo + i;
    sm.keys[i] = make_key(row[j], id_map ? id_map[j] : (int32_t)j);
  }
  block_select_topk(cnt, k, [&](int i) { return sm.keys[i]; }, sm.sel);
  const int kk = cnt < k ? cnt : k;
  uint64_t* dst = ws.keys + ((int64_t)r * parts + p) * k;
  for (int i = tid; i < kk; i += kSelectThreads) dst[i] = sm.sel.out[i];
  if (tid == 0) {
    ws.counts[r * parts + p] = kk;
    ws.kth[r * parts + p] = kk == k ? sm.sel.out[k - 1] : 0ull;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) sm.is_last = (atomicAdd(&ws.counters[r], 1u) == (uint32_t)(parts - 1));
  __syncthreads();
  if (!sm.is_last) return;
  __threadfence();

  // ---- join: every key of the row's top-k is >= L = max over parts of the part's k-th key (the
  // part holding L has k keys >= L), so only each sorted list's prefix >= L takes part ----
  const uint64_t* rowkeys = ws.keys + (int64_t)r * parts * k;
  const int* rowcounts = ws.counts + r * parts;
  uint64_t L = 0ull;
  for (int q = tid; q < parts; q += kSelectThreads) L = umax64(L, __ldcg(ws.kth + r * parts + q));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L = umax64(L, shfl_xor_u64(L, o));
  if (lane == 0) sm.red[warp] = L;
  __syncthreads();
  L = 0ull;
  for (int w = 0; w < kSelectThreads / 32; ++w) L = umax64(L, sm.red[w]);
  // survivors of each part (binary search of its descending list); thread tid owns parts
  // tid, tid + 512, ... and their survivors are placed after an exclusive scan.
  int mine = 0;
  for (int q = tid; q < parts; q += kSelectThreads) {
    const uint64_t* lst = rowkeys + (int64_t)q * k;
    int a = 0, b = __ldcg(rowcounts + q);  // first index with key < L lies in [a, b]
    while (a < b) {
      int m = (a + b) >> 1;
      if (__ldcg(lst + m) >= L) a = m + 1; else b = m;
    }
    mine += a;
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sm.scan[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += sm.scan[w];
  if (tid == kSelectThreads - 1) sm.total = before + incl;
  __syncthreads();
  const int total = sm.total;
  if (total <= kStage) {
    int at = before + incl - mine;
    for (int q = tid; q < parts; q += kSelectThreads) {
      const uint64_t* lst = rowkeys + (int64_t)q * k;
      const int c = __ldcg(rowcounts + q);
      for (int i = 0; i < c; ++i) {
        const uint64_t key = __ldcg(lst + i);
        if (key < L) break;
        sm.keys[at++] = key;
      }
    }
    block_select_topk(total, k, [&](int i) { return sm.keys[i]; }, sm.sel);
  } else {
    // many near-equal keys at L: select from every list in global memory
    auto join_key = [&](int i) -> uint64_t {
      int q = i / k;
      int j = i - q * k;
      return j < __ldcg(rowcounts + q) ? __ldcg(rowkeys + i) : 0ull;
    };
    block_select_topk(parts * k, k, join_key, sm.sel);
  }
  for (int i = tid; i < k; i += kSelectThreads) {
    vals[(int64_t)r * ld_out + i] = key_value(sm.sel.out[i]);
    ids[(int64_t)r * ld_out + i] = key_id(sm.sel.out[i]);
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
