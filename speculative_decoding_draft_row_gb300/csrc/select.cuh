// select.cuh - block-wide exact top-k selection by radix descent on 64-bit ordering keys.
#pragma once

#include "common.cuh"

namespace tfd {

constexpr int kSelectThreads = 512;
constexpr int kSelectMaxK = 512;

struct SelectSmem {
  uint64_t out[kSelectMaxK];     // selected keys (then sorted in place)
  uint32_t whist[kSelectThreads / 64][256];  // one histogram per pair of warps
  uint32_t hist[256];
  int found_digit;
  int found_above;
  int found_count;
  int out_count;
  int eq_count;
};

// Selects the min(k, cnt) largest of cnt keys (k <= kSelectMaxK) produced by key_at(i), i in
// [0, cnt), into sm.out[0..min(k, cnt)), sorted descending. Keys are unique except for exact duplicates,
// which are interchangeable. The radix descent histograms 8 bits of the key per pass among the
// keys that share the prefix found so far (shared-memory histograms per pair of warps, then summed),
// stopping as soon as the boundary bin is taken whole.
// Must be called by all kSelectThreads threads of the block.
template <class KeyAt>
__device__ void block_select_topk(int cnt, int k, KeyAt key_at, SelectSmem& sm, bool sort = true) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  __syncthreads();  // the previous use of sm is finished
  if (tid == 0) { sm.out_count = 0; sm.eq_count = 0; }
  __syncthreads();
  uint64_t prefix = 0;
  int shift = 64;
  int need = k;
  bool whole_bin = true;
  if (cnt > k) {
    whole_bin = false;
    for (int pass = 0; pass < 8; ++pass) {
      shift -= 8;
      for (int b = tid; b < (kSelectThreads / 64) * 256; b += kSelectThreads)
        (&sm.whist[0][0])[b] = 0;
      __syncthreads();
      for (int i = tid; i < cnt; i += kSelectThreads) {
        const uint64_t key = key_at(i);
        if (shift == 56 || (key >> (shift + 8)) == prefix)
          atomicAdd(&sm.whist[warp >> 1][(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      for (int b = tid; b < 256; b += kSelectThreads) {
        uint32_t c = 0;
#pragma unroll
        for (int w = 0; w < kSelectThreads / 64; ++w) c += sm.whist[w][b];
        sm.hist[b] = c;
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins [248 - 8l, 255 - 8l]; lane 0 the highest.
        uint32_t local[8];
        uint32_t sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) { local[j] = sm.hist[255 - 8 * lane - j]; sum += local[j]; }
        uint32_t incl = sum;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
          uint32_t o = __shfl_up_sync(0xffffffffu, incl, m);
          if (lane >= m) incl += o;
        }
        uint32_t excl = incl - sum;
        unsigned hit = __ballot_sync(0xffffffffu, incl >= (uint32_t)need);
        int first = __ffs(hit) - 1;
        if (lane == first) {
          uint32_t above = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (above + local[j] >= (uint32_t)need) {
              sm.found_digit = 255 - 8 * lane - j;
              sm.found_above = (int)above;
              sm.found_count = (int)local[j];
              break;
            }
            above += local[j];
          }
        }
      }
      __syncthreads();
      int d = sm.found_digit;
      need -= sm.found_above;
      prefix = (prefix << 8) | (uint64_t)d;
      bool done = (sm.found_count == need);
      __syncthreads();
      if (done) { whole_bin = true; break; }
    }
  }
  // Gather: keys above the prefix, and keys equal to it (all of them when the bin is taken whole,
  // else `need` of the identical keys left after 8 passes).
  for (int i = tid; i < cnt; i += kSelectThreads) {
    uint64_t key = key_at(i);
    bool take;
    if (cnt <= k) {
      take = true;
    } else {
      uint64_t top = shift >= 64 ? 0ull : (key >> shift);
      take = top > prefix;
      if (!take && top == prefix) take = whole_bin || atomicAdd(&sm.eq_count, 1) < need;
    }
    if (take) {
      int slot = atomicAdd(&sm.out_count, 1);
      if (slot < kSelectMaxK) sm.out[slot] = key;
    }
  }
  __syncthreads();
  if (!sort) return;
  // Bitonic sort of the min(k, cnt) selected keys, descending (padded with zero keys).
  const int kk = cnt < k ? cnt : k;
  int kpad = 1;
  while (kpad < kk) kpad <<= 1;
  for (int i = kk + tid; i < kpad; i += kSelectThreads) sm.out[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= kpad; size <<= 1) {
    for (int j = size >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < kpad; i += kSelectThreads) {
        int ixj = i ^ j;
        if (ixj > i) {
          uint64_t a = sm.out[i], b = sm.out[ixj];
          bool first_half_desc = (i & size) == 0;
          if (first_half_desc ? (a < b) : (a > b)) { sm.out[i] = b; sm.out[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
}

// One warp sorts a[0..n) descending in shared memory (n a power of two, <= 1024).
__device__ inline void warp_sort_desc(uint64_t* a, int n) {
  const int lane = threadIdx.x & 31;
  for (int size = 2; size <= n; size <<= 1) {
    for (int j = size >> 1; j > 0; j >>= 1) {
      for (int t = lane; t < (n >> 1); t += 32) {
        const int i = 2 * t - (t & (j - 1));
        const uint64_t x = a[i], y = a[i + j];
        if (((i & size) == 0) ? (x < y) : (x > y)) { a[i] = y; a[i + j] = x; }
      }
      __syncwarp();
    }
  }
}

constexpr int kDigitBits = 12;
constexpr int kBins = 1 << kDigitBits;
constexpr int kCandCap = 2048;     // keys at or above the boundary bin that are ranked directly
constexpr int kRankDirect = 1024;  // at most this many keys are ranked without a histogram

struct FastSelectSmem {
  uint32_t hist[kBins];
  uint64_t cand[kCandCap];
  int warp_sum[kSelectThreads / 32];
  int bstar, n_cand;
};

// out[rank] = key for the keys of c[0..n) whose rank (number of keys that beat it; equal keys are
// ordered by position) is below k: the top min(k, n) in descending order. One broadcast read of
// each candidate per thread; no sorting network.
__device__ inline void rank_count_select(const uint64_t* c, int n, int k, uint64_t* out) {
  const int tid = threadIdx.x;
  for (int i0 = tid; i0 < n; i0 += 2 * kSelectThreads) {
    const int i1 = i0 + kSelectThreads;
    const uint64_t a = c[i0];
    const uint64_t b = i1 < n ? c[i1] : 0ull;
    int ra = 0, rb = 0;
    int j = 0;
    for (; j + 8 <= n; j += 8) {  // 8 independent broadcast loads in flight
      uint64_t x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = c[j + u];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        ra += (x[u] > a) | ((x[u] == a) & (j + u < i0));
        rb += (x[u] > b) | ((x[u] == b) & (j + u < i1));
      }
    }
    for (; j < n; ++j) {
      const uint64_t x = c[j];
      ra += (x > a) | ((x == a) & (j < i0));
      rb += (x > b) | ((x == b) & (j < i1));
    }
    if (ra < k) out[ra] = a;
    if (i1 < n && rb < k) out[rb] = b;
  }
  __syncthreads();
}

// Top min(k, cnt) of keys[0..cnt) (shared memory), descending, written to out[0..min(k, cnt)).
// Small inputs are ranked directly. Otherwise one histogram of the top 12 key bits finds the bin
// holding the k-th key, every key in that bin or above is gathered (warp-aggregated appends) and
// ranked. Degenerate inputs (more than kCandCap keys at or above that bin) use the radix descent.
// Called by all kSelectThreads threads of the block.
__device__ inline void block_topk_fast(int cnt, int k, const uint64_t* keys, uint64_t* out,
                                       FastSelectSmem& fs, SelectSmem& sel) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __syncthreads();
  if (cnt <= kRankDirect || cnt <= k) {
    rank_count_select(keys, cnt, k, out);
    return;
  }
  for (int b = tid; b < kBins; b += kSelectThreads) fs.hist[b] = 0u;
  if (tid == 0) fs.n_cand = 0;
  __syncthreads();
  for (int i = tid; i < cnt; i += kSelectThreads)
    atomicAdd(&fs.hist[keys[i] >> (64 - kDigitBits)], 1u);
  __syncthreads();
  constexpr int per = kBins / kSelectThreads;  // bins [per * tid, per * tid + per) per thread
  uint32_t c[per];
  int mine = 0;
#pragma unroll
  for (int j = 0; j < per; ++j) { c[j] = fs.hist[per * tid + j]; mine += (int)c[j]; }
  int incl = mine;  // suffix sum over the warp's lanes (higher lanes own higher bins)
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += v;
  }
  if (lane == 0) fs.warp_sum[warp] = incl;
  __syncthreads();
  int above = incl - mine;
  for (int w = warp + 1; w < kSelectThreads / 32; ++w) above += fs.warp_sum[w];
  if (above < k && above + mine >= k) {
#pragma unroll
    for (int j = per - 1; j >= 0; --j) {
      if (above + (int)c[j] >= k) { fs.bstar = per * tid + j; break; }
      above += (int)c[j];
    }
  }
  __syncthreads();
  const uint64_t bstar = (uint64_t)fs.bstar;
  // gather the keys at or above the boundary bin: each warp counts its takers with ballots,
  // reserves its slots with one atomic, then writes them in order
  const int rounds = (cnt + kSelectThreads - 1) / kSelectThreads;
  int wcount = 0;
  for (int r = 0; r < rounds; ++r) {
    const int i = r * kSelectThreads + tid;
    const bool take = i < cnt && (keys[i] >> (64 - kDigitBits)) >= bstar;
    wcount += __popc(__ballot_sync(0xffffffffu, take));
  }
  int base = 0;
  if (lane == 0) base = atomicAdd(&fs.n_cand, wcount);
  base = __shfl_sync(0xffffffffu, base, 0);
  for (int r = 0; r < rounds; ++r) {
    const int i = r * kSelectThreads + tid;
    const uint64_t key = i < cnt ? keys[i] : 0ull;
    const bool take = i < cnt && (key >> (64 - kDigitBits)) >= bstar;
    const unsigned m = __ballot_sync(0xffffffffu, take);
    const int at = base + __popc(m & ((1u << lane) - 1u));
    if (take && at < kCandCap) fs.cand[at] = key;
    base += __popc(m);
  }
  __syncthreads();
  const int ncand = fs.n_cand;
  if (ncand > kCandCap) {
    block_select_topk(cnt, k, [&](int i) { return keys[i]; }, sel, true);
    for (int i = tid; i < k; i += kSelectThreads) out[i] = sel.out[i];
    __syncthreads();
    return;
  }
  rank_count_select(fs.cand, ncand, k, out);
}

// Sorts a[0..np) descending in shared memory by a bitonic network (np a power of two). Called by
// all kSelectThreads threads of the block; returns after a barrier.
__device__ inline void block_sort_desc(uint64_t* a, int np) {
  const int tid = threadIdx.x;
  __syncthreads();
  for (int size = 2; size <= np; size <<= 1) {
    for (int j = size >> 1; j > 0; j >>= 1) {
      for (int t = tid; t < (np >> 1); t += kSelectThreads) {
        const int i = 2 * t - (t & (j - 1));
        const uint64_t x = a[i], y = a[i + j];
        if (((i & size) == 0) ? (x < y) : (x > y)) { a[i] = y; a[i + j] = x; }
      }
      __syncthreads();
    }
  }
}

// Sorts keys[0..c) descending for c <= 1024 (room for 1024; slots past c count as zero keys),
// by a bitonic network over 1024 slots. Each warp holds 64 consecutive slots, two per lane, so the
// 45 stages whose partners are at most 32 slots apart run in registers with warp shuffles; only
// the 10 stages with partners 64 or more apart go through shared memory and block barriers.
// Called by all kSelectThreads threads of the block; returns after a barrier.
__device__ inline void block_sort_desc_1024(uint64_t* keys, int c) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = 64 * warp + 2 * lane, i1 = i0 + 1;  // this thread's two slots
  __syncthreads();
  uint64_t a0 = i0 < c ? keys[i0] : 0ull;
  uint64_t a1 = i1 < c ? keys[i1] : 0ull;
  for (int size = 2; size <= 1024; size <<= 1) {
    for (int j = size >> 1; j > 0; j >>= 1) {
      uint64_t y0, y1;
      if (j >= 64) {  // partner in another warp
        __syncthreads();
        keys[i0] = a0;
        keys[i1] = a1;
        __syncthreads();
        y0 = keys[i0 ^ j];
        y1 = keys[i1 ^ j];
      } else if (j >= 2) {  // partner lane ^ (j / 2), same register
        y0 = shfl_xor_u64(a0, j >> 1);
        y1 = shfl_xor_u64(a1, j >> 1);
      } else {  // partners in the same lane
        y0 = a1;
        y1 = a0;
      }
      // keep the larger where the slot's block of `size` runs descending and it is the lower
      // slot of the pair, or where its block runs ascending and it is the upper one
      const bool km0 = ((i0 & size) == 0) == ((i0 & j) == 0);
      const bool km1 = ((i1 & size) == 0) == ((i1 & j) == 0);
      a0 = km0 ? umax64(a0, y0) : (a0 < y0 ? a0 : y0);
      a1 = km1 ? umax64(a1, y1) : (a1 < y1 ? a1 : y1);
    }
  }
  __syncthreads();
  keys[i0] = a0;
  keys[i1] = a1;
  __syncthreads();
}

}  // namespace tfd
