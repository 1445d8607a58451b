// common.cuh - device and host helpers shared by the libtfd kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tfd.h"

namespace tfd {

// ---- ordering keys ------------------------------------------------------------------------------
// Every top-k here ranks by (value desc, id asc), with -0 == +0 and NaN below -inf. A 64-bit key
// whose unsigned order is that ranking: high word = order-preserving image of the value (NaN -> 0),
// low word = complement of the biased id (lower id -> larger word).

__device__ __forceinline__ uint32_t value_key(float v) {
  if (v != v) return 0u;
  uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint64_t key) {
  uint32_t k = (uint32_t)(key >> 32);
  if (k == 0u) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint32_t id_key(int32_t id) { return ~((uint32_t)id ^ 0x80000000u); }

__device__ __forceinline__ int32_t key_id(uint64_t key) {
  return (int32_t)(~(uint32_t)key ^ 0x80000000u);
}

__device__ __forceinline__ uint64_t make_key(float v, int32_t id) {
  return ((uint64_t)value_key(v) << 32) | id_key(id);
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((uint64_t)hi << 32) | lo;
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

// ---- device status ------------------------------------------------------------------------------
__device__ __forceinline__ void set_dev_status(int32_t* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

// ---- bf16 ---------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

// ---- streaming loads ----------------------------------------------------------------------------
// Weights are read once per call: bypass L1, ask L2 for 256-byte fetches (TFD_L2_PREFETCH=1, the
// default) and mark the lines first to be evicted (the policy from l2_stream_policy), so that what
// a call writes and reads again (logits, sub-group maxima, part keys) stays in L2 meanwhile.
#ifndef TFD_L2_PREFETCH
#define TFD_L2_PREFETCH 1
#endif
#ifndef TFD_L2_EVICT_FIRST
#define TFD_L2_EVICT_FIRST 1
#endif
#if TFD_L2_PREFETCH
#define TFD_LD_STREAM "ld.global.nc.L1::no_allocate.L2::cache_hint.L2::256B"
#else
#define TFD_LD_STREAM "ld.global.nc.L1::no_allocate.L2::cache_hint"
#endif
__device__ __forceinline__ uint64_t l2_stream_policy() {
  uint64_t pol;
#if TFD_L2_EVICT_FIRST
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
#else
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
#endif
  return pol;
}
__device__ __forceinline__ uint4 ldg_stream16(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile(TFD_LD_STREAM ".v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream8(const void* p, uint64_t pol) {
  uint2 v;
  asm volatile(TFD_LD_STREAM ".v2.u32 {%0,%1}, [%2], %3;" : "=r"(v.x), "=r"(v.y) : "l"(p), "l"(pol));
  return v;
}

// ---- a planted failure for the bounded waits (TFD_TEST_STALL_EXCHANGE builds only) --------------
// A build with -DTFD_TEST_STALL_EXCHANGE=1 has the second block of every two-block cluster split
// drop its partial sums instead of sending them, so the leader's bounded waits run out and report
// TFD_ERR_TIMEOUT in the device status (tests of the failure path); the default build sends them.
#ifndef TFD_TEST_STALL_EXCHANGE
#define TFD_TEST_STALL_EXCHANGE 0
#endif

// ---- phase timestamps (TFD_TRACE builds only) -----------------------------------------------------
// A build with -DTFD_TRACE=1 records the global nanosecond timer at fixed points of a kernel, one
// row of kTraceSlots stamps per block, into a caller-given device buffer (tfd_trace_set); the
// default build compiles none of it.
#ifndef TFD_TRACE
#define TFD_TRACE 0
#endif
constexpr int kTraceSlots = 64;
#if TFD_TRACE
__device__ __forceinline__ void trace_stamp(uint64_t* buf, int slot) {
  if (buf != nullptr && threadIdx.x == 0 && slot < kTraceSlots) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    buf[(int64_t)blockIdx.x * kTraceSlots + slot] = t;
  }
}
#define TFD_STAMP(buf, slot) trace_stamp((buf), (slot))
#else
#define TFD_STAMP(buf, slot) \
  do {                       \
  } while (0)
#endif

// ---- warp reductions ----------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

}  // namespace tfd

// ---- host helpers (shared by the C entry points) -----------------------------------------------
namespace tfd_host {

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }
inline cudaStream_t as_stream(void* s) { return (cudaStream_t)s; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch status: the CUDA error of the launch just made, as a tfd_status.
inline tfd_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TFD_OK : TFD_ERR_CUDA;
}

// Number of SMs of the current device (0 when no device answers).
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace tfd_host

// Internal launchers shared across translation units.
namespace tfd_internal {
// Top-k over fp32 logits by a threshold filter, one thread-block cluster per row (topk.cu). The
// workspace is tfd_topk_workspace() bytes. pre_max, when not null, already holds the value key of
// the maximum of every 16-logit sub-group of each row, [rows][ceil(n / 16)], so the logits are
// read only where a sub-group can reach the threshold. part_max, when not null, holds the value
// key of the largest logit of each of `parts` contiguous parts of each row, [parts][rows]; with
// k <= parts the threshold is then the k-th largest of those (one block per row).
tfd_status topk_launch(const float* logits, int rows, int64_t n, int64_t ld, int k,
                       const int32_t* id_map, float* vals, int32_t* ids, int64_t ld_out,
                       const uint32_t* pre_max, const uint32_t* part_max, int parts, void* ws,
                       size_t ws_bytes, cudaStream_t stream);
size_t topk_workspace(int rows, int64_t n, int k);
}  // namespace tfd_internal
