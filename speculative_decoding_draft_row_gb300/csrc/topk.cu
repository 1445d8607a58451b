// topk.cu - top-k of fp32 logits: a threshold filter run by one thread-block cluster per row.
//
// Follows the TFE draft head page (#42): commit "... ocabulary head" (top cand_k of fp32 logits,
// 1..512, a tie at the k-th value going to the lower token id; the top-1 through an id map) and
// commit "pass kernels and FP8 linears" (a vocabulary row scanned in parts and joined).
//
// Each row is cut into sub-groups of 16 consecutive logits. The k-th largest sub-group maximum m_k
// is at most the row's k-th largest logit: the k sub-groups holding the k largest maxima each hold
// a logit at least m_k. So every logit of the row's top k is >= m_k, and >= any T <= m_k.
//
// A cluster of 8 blocks takes one row, each block an eighth of it. Each block reads its part once
// and keeps its sub-group maxima in shared memory; a histogram of all the row's maxima, summed
// across the cluster through distributed shared memory, locates the bin holding m_k (fine bins
// measured down from the row's largest maximum; two 12-bit levels of the value key when m_k lies
// far below it), and T is the bin's lower edge. Only sub-groups whose maximum reaches T can hold
// a logit >= T: each block reads those again (about k / 8 sub-groups of 16 logits) and appends
// their logits >= T to a candidate list in block 0's shared memory, so the list holds little
// more than k keys. Block 0 selects the top k of the list (a rank count when it is short, else a
// sort). A list longer than its capacity (thousands of equal values at the k-th place) is
// abandoned for an exact radix select over the whole row.
#include <cooperative_groups.h>

#include "select.cuh"

namespace {

using namespace tfd;
namespace cg = cooperative_groups;

constexpr int kThreads = kSelectThreads;  // 512
constexpr int kCl = 8;                     // blocks per row: one cluster
constexpr int kUnroll = 4;                 // float4 loads in flight per thread in the maxima pass
constexpr int kSub = 16;                   // logits per sub-group
constexpr int kCandCap = 4096;             // keys of block 0's candidate list
constexpr int kSubCap = 4096;              // sub-group maxima a block keeps in shared memory
constexpr int kRankMax = 192;              // lists up to this length are ranked, else sorted
constexpr int kRange = kBins / kCl;        // histogram bins each block sums: 512
// Fused top-k after a GEMV that gives part maxima: threshold from them, one block per row (1), or
// the cluster's histogram of sub-group maxima (0).
#ifndef TFD_TOPK_PARTS
#define TFD_TOPK_PARTS 1
#endif

struct ClusterSmem {
  uint64_t cand[kCandCap];     // block 0: the row's candidate keys
  uint32_t hist[kBins];        // histogram of this block's maxima; later its qualifying sub-groups
  uint32_t maxima[kSubCap];    // this block's sub-group maxima (value keys)
  uint32_t red[kRange];        // cluster sums of the bins this block owns
  SelectSmem sel;
  uint32_t tot[kCl];           // cluster sum of each block's owned bins
  uint32_t warp_u[kThreads / 32];
  uint32_t bmax;               // this block's largest maximum
  uint32_t cand_count;         // block 0: candidates appended
  uint32_t n_qual;             // qualifying sub-groups found in the current window
  int res_bin, res_above;      // histogram boundary, written by the block that owns it
};

__device__ __forceinline__ uint32_t block_reduce_u32(uint32_t v, bool is_max, ClusterSmem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t x = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? max(v, x) : v + x;
  }
  __syncthreads();
  if (lane == 0) sm.warp_u[warp] = v;
  __syncthreads();
  uint32_t r = 0u;
  for (int w = 0; w < kThreads / 32; ++w) r = is_max ? max(r, sm.warp_u[w]) : r + sm.warp_u[w];
  return r;
}

// Loads 4 logits at e (NaN past hi, never read there); VEC: one 16-byte load when all 4 are in.
template <bool VEC>
__device__ __forceinline__ float4 load4(const float* __restrict__ row, int64_t e, int64_t hi) {
  const float nan = __uint_as_float(0x7FC00000u);
  if (VEC && e + 3 < hi) return __ldg(reinterpret_cast<const float4*>(row + e));
  float4 v;
  v.x = e < hi ? row[e] : nan;
  v.y = e + 1 < hi ? row[e + 1] : nan;
  v.z = e + 2 < hi ? row[e + 2] : nan;
  v.w = e + 3 < hi ? row[e + 3] : nan;
  return v;
}

// Value keys of 4 consecutive logits, reduced over the 4 lanes that hold one sub-group of 16.
__device__ __forceinline__ uint32_t sub_max4(const float4& v) {
  uint32_t m = max(max(value_key(v.x), value_key(v.y)), max(value_key(v.z), value_key(v.w)));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
  return max(m, __shfl_xor_sync(0xffffffffu, m, 2));
}

// Cluster-wide histogram boundary over every block's maxima[0..nsub). bin_of maps a value key to
// a bin in [0, kBins), or -1 to leave it out; bin 0 is counted per warp first, since it may
// collect most keys. Block q sums bins [512q, 512q + 512) over the cluster; the block owning the
// bin that holds the need-th largest entry writes that bin and the count of entries in higher
// bins into every block. Called by all threads of all blocks of the cluster.
template <class BinOf>
__device__ __noinline__ void cluster_boundary(const uint32_t* maxima, int nsub, BinOf bin_of,
                                              uint32_t need, ClusterSmem& sm, int& out_bin,
                                              uint32_t& out_above) {
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cluster.block_rank();
  for (int b = tid; b < kBins; b += kThreads) sm.hist[b] = 0u;
  __syncthreads();
  uint32_t zero_bin = 0u;
  for (int i = tid; i < nsub; i += kThreads) {
    const int b = bin_of(maxima[i]);
    if (b == 0) ++zero_bin;
    else if (b > 0) atomicAdd(&sm.hist[b], 1u);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) zero_bin += __shfl_xor_sync(0xffffffffu, zero_bin, o);
  if (lane == 0 && zero_bin != 0u) atomicAdd(&sm.hist[0], zero_bin);
  cluster.sync();  // every block's histogram is complete
  const int bin = rank * kRange + tid;  // kThreads == kRange: one owned bin per thread
  uint32_t c = 0u;
  for (int q = 0; q < kCl; ++q) c += cluster.map_shared_rank(sm.hist, q)[bin];
  sm.red[tid] = c;
  const uint32_t tot = block_reduce_u32(c, false, sm);
  if (tid < kCl) cluster.map_shared_rank(sm.tot, tid)[rank] = tot;
  cluster.sync();  // every block's range sum is everywhere
  uint32_t above = 0u;
  for (int q = rank + 1; q < kCl; ++q) above += sm.tot[q];
  if (above < need && above + sm.tot[rank] >= need) {  // block-uniform: this block owns it
    const uint32_t v = sm.red[tid];
    uint32_t incl = v;  // suffix sum over the warp's lanes (higher lanes own higher bins)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += x;
    }
    if (lane == 0) sm.warp_u[warp] = incl;
    __syncthreads();
    for (int w = warp + 1; w < kThreads / 32; ++w) incl += sm.warp_u[w];
    const uint32_t ab = above + incl - v;  // entries in bins above this one
    if (ab < need && ab + v >= need) {     // exactly one thread
      for (int q = 0; q < kCl; ++q) {
        *cluster.map_shared_rank(&sm.res_bin, q) = bin;
        *cluster.map_shared_rank(&sm.res_above, q) = (int)ab;
      }
    }
  }
  cluster.sync();  // the boundary is everywhere
  out_bin = sm.res_bin;
  out_above = (uint32_t)sm.res_above;
}

struct FineBin {  // bins of 4096 key units below the row's largest maximum K; bin 0 is the rest
  uint32_t K;
  __device__ int operator()(uint32_t key) const {
    const uint32_t fine = (K - key) >> 12;
    return fine < (uint32_t)(kBins - 1) ? kBins - 1 - (int)fine : 0;
  }
};
struct HighBits {  // bits 31..20 of the value key
  __device__ int operator()(uint32_t key) const { return (int)(key >> 20); }
};
struct MidBits {  // bits 19..8 of the value keys whose bits 31..20 are b1
  int b1;
  __device__ int operator()(uint32_t key) const {
    return (int)(key >> 20) == b1 ? (int)((key >> 8) & 0xFFFu) : -1;
  }
};

// T <= m_k for the row whose maxima the cluster holds (S >= k of them, largest K).
__device__ uint32_t cluster_threshold(const uint32_t* maxima, int nsub, uint32_t K, int k,
                                      ClusterSmem& sm) {
  int b;
  uint32_t above;
  cluster_boundary(maxima, nsub, FineBin{K}, (uint32_t)k, sm, b, above);
  if (b > 0) {
    const int64_t t = (int64_t)K - (int64_t)(kBins - 1 - b) * 4096 - 4095;
    return t > 0 ? (uint32_t)t : 0u;
  }
  // m_k lies far below the largest maximum: the value key's own bits, two levels
  int b1, b2;
  uint32_t a1, a2;
  cluster_boundary(maxima, nsub, HighBits{}, (uint32_t)k, sm, b1, a1);
  cluster_boundary(maxima, nsub, MidBits{b1}, (uint32_t)k - a1, sm, b2, a2);
  return ((uint32_t)b1 << 20) | ((uint32_t)b2 << 8);
}

template <bool VEC>
__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kThreads, 2)
topk_cluster_kernel(const float* __restrict__ logits, int64_t n, int64_t ld, int k,
                    const int32_t* __restrict__ id_map, float* __restrict__ vals,
                    int32_t* __restrict__ ids, int64_t ld_out,
                    const uint32_t* __restrict__ pre_max, uint32_t* __restrict__ gmaxima,
                    int64_t chunk, const uint32_t* __restrict__ part_max, int parts) {
  extern __shared__ __align__(16) unsigned char tk_smem[];
  ClusterSmem& sm = *reinterpret_cast<ClusterSmem*>(tk_smem);
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.y;
  const float* row = logits + (int64_t)r * ld;
  const int64_t lo = (int64_t)rank * chunk < n ? (int64_t)rank * chunk : n;
  const int64_t hi = lo + chunk < n ? lo + chunk : n;
  const int nsub = (int)((hi - lo + kSub - 1) / kSub);
  const int64_t sub_per_block = chunk / kSub;
  const int64_t S = (n + kSub - 1) / kSub;
  uint32_t* wmax = sub_per_block <= kSubCap
                       ? sm.maxima
                       : gmaxima + ((int64_t)r * kCl + rank) * sub_per_block;
  const uint32_t* maxima = wmax;
  if (tid == 0) sm.cand_count = 0u;

  uint32_t lmax = 0u;
  if (pre_max != nullptr) {  // maxima given (written by the producer of the logits)
    const uint32_t* src = pre_max + (int64_t)r * S + (int64_t)rank * sub_per_block;
    if (sub_per_block <= kSubCap) {
      for (int i = tid; i < nsub; i += kThreads) {
        const uint32_t m = __ldcg(src + i);
        wmax[i] = m;
        lmax = max(lmax, m);
      }
    } else {
      for (int i = tid; i < nsub; i += kThreads) lmax = max(lmax, __ldcg(src + i));
      maxima = src;
    }
  }
  // ---- pass 1: the part's sub-group maxima (the only full read of the logits) ----
  constexpr int kStep = 4 * kThreads * kUnroll;
  for (int64_t b0 = pre_max ? hi : lo; b0 < hi; b0 += kStep) {  // block-uniform bounds
    float4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      v[u] = load4<VEC>(row, b0 + 4 * (int64_t)(u * kThreads + tid), hi);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t m = sub_max4(v[u]);
      const int64_t sg = (b0 - lo + 4 * (int64_t)(u * kThreads + tid)) / kSub;
      if ((tid & 3) == 0 && sg < nsub) wmax[sg] = m;
      lmax = max(lmax, m);
    }
  }
  uint32_t T;
  if (part_max != nullptr) {
    // ---- the threshold from the producer's part maxima, in every block: T = the k-th largest
    // of them (k <= parts), the value v with (# > v) < k <= (# >= v) ----
    uint32_t* pm = sm.hist;
    for (int i = tid; i < parts; i += kThreads) pm[i] = __ldcg(part_max + (int64_t)i * gridDim.y + r);
    if (tid == 0) sm.res_bin = 0;
    __syncthreads();
    for (int i = tid; i < parts; i += kThreads) {
      const uint32_t v = pm[i];
      int gt = 0, ge = 0;
      for (int j = 0; j < parts; ++j) {
        const uint32_t x = pm[j];
        gt += x > v;
        ge += x >= v;
      }
      if (gt < k && ge >= k) sm.res_bin = (int)v;  // every writer writes the same value
    }
    cluster.sync();  // maxima, the threshold and block 0's zeroed count are visible
    T = (uint32_t)sm.res_bin;
  } else {
    const uint32_t bm = block_reduce_u32(lmax, true, sm);
    if (tid == 0) sm.bmax = bm;
    cluster.sync();  // maxima, block maxima and block 0's zeroed count are visible

    // ---- the threshold T <= m_k ----
    uint32_t K = 0u;
    for (int q = 0; q < kCl; ++q) K = max(K, *cluster.map_shared_rank(&sm.bmax, q));
    T = S >= k ? cluster_threshold(maxima, nsub, K, k, sm) : 0u;
  }

  // ---- pass 2: the logits >= T of the sub-groups whose maximum reaches T ----
  uint64_t* cand0 = cluster.map_shared_rank(sm.cand, 0);
  uint32_t* count0 = cluster.map_shared_rank(&sm.cand_count, 0);
  uint32_t* qual = sm.hist;  // free: no block reads another's histogram any more
  for (int w0 = 0; w0 < nsub; w0 += kBins) {  // windows of kBins maxima
    const int wn = nsub - w0 < kBins ? nsub - w0 : kBins;
    if (tid == 0) sm.n_qual = 0u;
    __syncthreads();
    for (int i0 = 0; i0 < wn; i0 += kThreads) {
      const int i = i0 + tid;
      const bool q = i < wn && maxima[w0 + i] >= T;
      const unsigned m = __ballot_sync(0xffffffffu, q);
      if (m != 0u) {
        const int leader = __ffs(m) - 1;
        uint32_t base = 0u;
        if (lane == leader) base = atomicAdd(&sm.n_qual, (uint32_t)__popc(m));
        base = __shfl_sync(0xffffffffu, base, leader);
        if (q) qual[base + __popc(m & ((1u << lane) - 1u))] = (uint32_t)(w0 + i);
      }
    }
    __syncthreads();
    const int nq = (int)sm.n_qual;
    for (int j0 = 0; j0 < nq; j0 += 2 * (kThreads / 32)) {  // a half-warp per sub-group
      const int j = j0 + 2 * warp + (lane >> 4);
      const bool valid = j < nq;
      const int64_t e = lo + (int64_t)(valid ? qual[j] : 0u) * kSub + (lane & 15);
      const float x = valid && e < hi ? row[e] : 0.0f;
      const bool take = valid && e < hi && value_key(x) >= T;
      const unsigned m = __ballot_sync(0xffffffffu, take);
      if (m != 0u) {
        const int leader = __ffs(m) - 1;
        uint32_t base = 0u;
        if (lane == leader) base = atomicAdd(count0, (uint32_t)__popc(m));
        base = __shfl_sync(0xffffffffu, base, leader);
        const uint32_t slot = base + (uint32_t)__popc(m & ((1u << lane) - 1u));
        if (take && slot < (uint32_t)kCandCap)
          cand0[slot] = make_key(x, id_map ? __ldg(id_map + e) : (int32_t)e);
      }
    }
    __syncthreads();  // the list of qualifying sub-groups is reused by the next window
  }
  cluster.sync();  // block 0's list is complete; no block touches another's memory after this
  if (rank != 0) return;

  // ---- block 0: the top k of the list (at least k keys) ----
  const uint32_t c = sm.cand_count;
  const uint64_t* top;
  if (c <= (uint32_t)kCandCap) {
    const int cn = (int)c;
    if (cn <= kRankMax) {
      rank_count_select(sm.cand, cn, k, sm.sel.out);
      top = sm.sel.out;
    } else if (cn <= 1024) {
      block_sort_desc_1024(sm.cand, cn);
      top = sm.cand;
    } else {
      int np = 1;
      while (np < cn) np <<= 1;
      for (int i = cn + tid; i < np; i += kThreads) sm.cand[i] = 0ull;
      block_sort_desc(sm.cand, np);
      top = sm.cand;
    }
  } else {
    block_select_topk((int)n, k, [&](int i) {
      return make_key(row[i], id_map ? id_map[i] : (int32_t)i);
    }, sm.sel);
    top = sm.sel.out;
  }
  for (int i = tid; i < k; i += kThreads) {
    vals[(int64_t)r * ld_out + i] = key_value(top[i]);
    ids[(int64_t)r * ld_out + i] = key_id(top[i]);
  }
}

int64_t part_len(int64_t n) {  // logits per block: an eighth of the row, whole sub-groups
  const int64_t c = (n + kCl - 1) / kCl;
  return (c + kSub - 1) / kSub * kSub;
}

size_t gmaxima_bytes(int rows, int64_t n) {
  const int64_t sub = part_len(n) / kSub;
  return sub <= kSubCap ? 0 : (size_t)rows * kCl * sub * 4;
}

}  // namespace

namespace tfd_internal {

size_t topk_workspace(int rows, int64_t n, int k) {
  if (rows < 1 || n < 1 || k < 1 || k > TFD_MAX_TOPK || k > n) return 0;
  return tfd_host::round_up(gmaxima_bytes(rows, n), 256) + 256;
}

tfd_status topk_launch(const float* logits, int rows, int64_t n, int64_t ld, int k,
                       const int32_t* id_map, float* vals, int32_t* ids, int64_t ld_out,
                       const uint32_t* pre_max, const uint32_t* part_max, int parts, void* ws,
                       size_t ws_bytes, cudaStream_t stream) {
  const size_t need = topk_workspace(rows, n, k);
  if (need == 0) return TFD_ERR_INVALID;
  if (ws == nullptr || ws_bytes < need) return TFD_ERR_WORKSPACE;
  const bool vec = tfd_host::aligned(logits, 16) && ld % 4 == 0;
  // the producer's part maxima give the threshold when there are at least k parts
  const bool use_parts = TFD_TOPK_PARTS && pre_max != nullptr && part_max != nullptr &&
                         k <= parts && parts <= kBins;
  const size_t smem = sizeof(ClusterSmem);
  auto kern = vec ? topk_cluster_kernel<true> : topk_cluster_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return TFD_ERR_CUDA;
  dim3 grid(kCl, (unsigned)rows);
  kern<<<grid, kThreads, smem, stream>>>(logits, n, ld, k, id_map, vals, ids, ld_out, pre_max,
                                         reinterpret_cast<uint32_t*>(ws), part_len(n),
                                         use_parts ? part_max : nullptr, use_parts ? parts : 0);
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
  return tfd_internal::topk_launch(logits, rows, n, ld, k, id_map, vals, ids, k, nullptr,
                                   nullptr, 0, ws, ws_bytes, tfd_host::as_stream(stream));
}
