// select.cuh - block-wide exact top-k selection by radix descent on 64-bit ordering keys.
#pragma once

#include "common.cuh"

namespace tfd {

constexpr int kSelectThreads = 512;
constexpr int kSelectMaxK = 512;

struct SelectSmem {
  uint64_t out[kSelectMaxK];     // selected keys (then sorted in place)
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
// keys that share the prefix found so far, stopping as soon as the boundary bin is taken whole.
// Must be called by all kSelectThreads threads of the block.
template <class KeyAt>
__device__ void block_select_topk(int cnt, int k, KeyAt key_at, SelectSmem& sm) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int cnt_round = (cnt + 31) & ~31;

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
      for (int b = tid; b < 256; b += kSelectThreads) sm.hist[b] = 0;
      __syncthreads();
      for (int i = tid; i < cnt_round; i += kSelectThreads) {
        bool valid = i < cnt;
        uint64_t key = valid ? key_at(i) : 0ull;
        bool match = valid && (shift == 56 || (key >> (shift + 8)) == prefix);
        int bin = match ? (int)((key >> shift) & 255u) : 256;
        unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (bin < 256 && (__ffs(peers) - 1) == lane) atomicAdd(&sm.hist[bin], __popc(peers));
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

}  // namespace tfd
