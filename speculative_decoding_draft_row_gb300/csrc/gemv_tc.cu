// gemv_tc.cu - the 17-32-row bf16 head GEMV on the fifth-generation tensor cores: weights staged
// into shared memory by TMA, tcgen05 MMAs (128 weight rows x 32 activation rows x 16 k) issued by
// one thread, fp32 accumulators in tensor memory, and warp-specialised roles.
//
// Follows the subset page (#1011): decode windows of 17 to 32 rows on the vocabulary head; the
// arithmetic (fp32 logits of bf16 weights and rows, top-1 by value then lower id) is the one of
// the TFE draft head page (#42), commit "pass kernels and FP8 linears".
//
// Design. A 32-row activation tile of a 4096-wide head (256 KB) does not fit one block's shared
// memory, so each 128-row group's k range is split over a cluster of two blocks (k halves), like
// the register-ring kernel; the difference is how the weights travel. Here the weight stream is
// TMA boxes of 128 rows x 64 k (16 KB, 128-byte swizzle) into a ring of shared-memory stages,
// five deep: the bytes in flight are held by shared memory, not registers, and one thread issues
// each box. Roles per block (192 threads): warp 0 lane 0 issues the TMA loads; warp 1 allocates
// the tensor memory and lane 0 issues the MMAs (four per stage, the accumulator of a group in one
// of two tensor-memory column buffers, each stage released by a tcgen05 commit); warps 2-5 read a
// finished accumulator (one row of 32 outputs a thread), and the second block of the pair sends
// its half into the leader's shared memory with asynchronous stores, where the leader adds it in
// rank order and runs the epilogue (fp32 logits, the running top-1 of each activation row and the
// online softmax state of its confidence, or for a fused top-k > 1 each 16-row sub-group's maximum
// and the part's maximum per row). At the end each leader writes its part's keys (and softmax
// states) and the last one to finish joins the parts.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cooperative_groups.h>
#include <mutex>

#include "gemv_kernel.cuh"

namespace tfd_gemv_tc {

using namespace tfd;

constexpr int kM = 128;                      // weight rows per group (tensor-memory lanes)
constexpr int kN = 32;                       // activation rows, zero-padded
constexpr int kKB = 64;                      // k per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 5;
constexpr int kStageBytes = kM * kKB * 2;    // 16 KB
constexpr int kXBlockBytes = kN * kKB * 2;   // 4 KB: 32 rows x 64 k of the activation tile
constexpr int kMaxKHalf = 2048;              // a block's k range: 32 rows x 2048 k = 128 KB
constexpr int kXBytes = kMaxKHalf / kKB * kXBlockBytes;
constexpr int kInboxBytes = kM * kN * 4;     // the second block's partials of one group
constexpr int kThreads = 192;
constexpr int kTmemCols = 64;                // two accumulator buffers of 32 columns

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr int kOffX = 0;
constexpr int kOffStage = kOffX + kXBytes;
constexpr int kOffInbox = kOffStage + kStages * kStageBytes;
constexpr int kOffBar = kOffInbox + kInboxBytes;  // mbarriers (8 bytes each)
constexpr int kNumBars = 2 * kStages + 1 + 2 + 2 + 2;
constexpr int kOffBest = kOffBar + kNumBars * 8 + 8;  // (+ the tensor-memory address)
constexpr int kOffJoin = kOffBest + 4 * kN * 8;
constexpr int kOffPmax = kOffJoin + kN * 8;
constexpr int kSmemUsed = kOffPmax + kN * 4 + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // room to align the base

struct TcArgs {
  int64_t n, k;
  int rows;
  int parts;  // clusters
  int64_t ngroups;
  float* y;  // fp32 logits [rows][ldy] (the top-k's logits when topk > 1), or null
  int64_t ldy;
  int topk;
  const int32_t* id_map;
  uint32_t* submax;    // topk > 1: [rows][ceil(n / 16)]
  uint32_t* part_max;  // topk > 1: [parts][rows]
  float* top1_conf;    // topk == 1: [rows] softmax probability of the top-1, or null
  float2* part_ms;     // with the confidence: [parts][rows] (max, sum of exp(l - max))
  uint64_t* part_keys;  // [parts][rows]
  uint32_t* counter;
  float* top_vals;
  int32_t* top_ids;
  int64_t ldt;
  int32_t* status;
};

__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}
// Bounded wait for the phase of parity `par` (about a second of global time); false on timeout.
// A thread that has timed out once waits no more, so a stuck pipeline ends within seconds.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t par) {
  uint64_t t0 = 0;
  for (int it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(par)
        : "memory");
    if (ok) return true;
    uint64_t now;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
    if (it == 0) t0 = now;
    else if (now - t0 > 1000000000ull) return false;
  }
}
__device__ __forceinline__ uint32_t to_cluster(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// TMA: box at coordinates (c0 = k element, c1 = row) of the 2D map into shared memory, counted by
// the mbarrier's transaction bytes.
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                           // leading byte offset (unused here): 16 B
  d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset
  d |= (uint64_t)1 << 46;                           // descriptor version
  d |= (uint64_t)2 << 61;                           // 128-byte swizzle
  return d;
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major, M x N.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) |
                            ((uint32_t)(kM >> 4) << 24);

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
// 32 consecutive accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st_async4(uint32_t dst, float a, float b, float c, float d,
                                          uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(dst),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
      : "memory");
}

template <bool CONF>  // the top-1 confidence (a second instantiation: its state costs registers)
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
gemv_tc_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
               const TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  namespace cg = cooperative_groups;
  const uint32_t crank = cg::this_cluster().block_rank();
  const int cid = blockIdx.x >> 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t g_begin = (int64_t)cid * a.ngroups / a.parts;
  const int64_t g_end = (int64_t)(cid + 1) * a.ngroups / a.parts;
  const int ng = (int)(g_end - g_begin);
  const int nkb = (int)(a.k / 2 / kKB);  // k blocks of this block's half
  const int kb0 = (int)crank * nkb;

  const uint32_t s_x = sa(smem + kOffX), s_stage = sa(smem + kOffStage);
  float* inbox = reinterpret_cast<float*>(smem + kOffInbox);
  const uint32_t b0 = sa(smem + kOffBar);
  auto full = [&](int s) { return b0 + 8u * s; };
  auto empty = [&](int s) { return b0 + 8u * (kStages + s); };
  const uint32_t xfull = b0 + 8u * (2 * kStages);
  auto tfull = [&](int b) { return b0 + 8u * (2 * kStages + 1 + b); };
  auto tempty = [&](int b) { return b0 + 8u * (2 * kStages + 3 + b); };
  const uint32_t ifull = b0 + 8u * (2 * kStages + 5);   // leader: the second block's partials
  const uint32_t iempty = b0 + 8u * (2 * kStages + 6);  // second block: the leader has read them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
  uint64_t* sbest = reinterpret_cast<uint64_t*>(smem + kOffBest);
  uint64_t* sjoin = reinterpret_cast<uint64_t*>(smem + kOffJoin);
  uint32_t* spmax = reinterpret_cast<uint32_t*>(smem + kOffPmax);

  if (tid < kN) spmax[tid] = 0u;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      bar_init(full(s), 1);
      bar_init(empty(s), 1);
    }
    bar_init(xfull, 1);
    for (int b = 0; b < 2; ++b) {
      bar_init(tfull(b), 1);
      bar_init(tempty(b), 4);
    }
    bar_init(ifull, 1);
    bar_init(iempty, 4);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     sa(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncwarp();
  // barriers initialised and tensor memory allocated in both blocks of the pair
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
  fence_after();
  const uint32_t tmem = *tmem_slot;
  bool timed_out = false;

  if (warp == 0) {
    if (lane == 0 && ng > 0) {
      // the activation tile of this block's k half, then the weight boxes group by group
      bar_expect_tx(xfull, (uint32_t)(nkb * kXBlockBytes));
      for (int kb = 0; kb < nkb; ++kb)
        tma_2d(s_x + (uint32_t)(kb * kXBlockBytes), &tx, (kb0 + kb) * kKB, 0, xfull);
      int it = 0;
      for (int64_t g = g_begin; g < g_end; ++g)
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !timed_out && !bar_wait(empty(s), (uint32_t)((it / kStages) - 1) & 1u))
            timed_out = true;
          bar_expect_tx(full(s), kStageBytes);
          tma_2d(s_stage + (uint32_t)(s * kStageBytes), &tw, (kb0 + kb) * kKB, (int)(g * kM), full(s));
        }
    }
  } else if (warp == 1) {
    if (lane == 0 && ng > 0) {
      if (!bar_wait(xfull, 0)) timed_out = true;  // (the first wait of this thread)
      fence_after();
      int it = 0;
      for (int j = 0; j < ng; ++j) {
        const int buf = j & 1;
        if (j >= 2 && !timed_out && !bar_wait(tempty(buf), (uint32_t)((j >> 1) - 1) & 1u)) timed_out = true;
        fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * kN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kStages;
          if (!timed_out && !bar_wait(full(s), (uint32_t)(it / kStages) & 1u)) timed_out = true;
          fence_after();
          const uint64_t da = sdesc(s_stage + (uint32_t)(s * kStageBytes));
          const uint64_t db = sdesc(s_x + (uint32_t)(kb * kXBlockBytes));
#pragma unroll
          for (int kk = 0; kk < kKB / 16; ++kk)  // 16 k (32 bytes, 2 address units) per MMA
            mma(d, da + 2u * kk, db + 2u * kk, (kb | kk) != 0);
          mma_commit(empty(s));  // the stage is free once these MMAs have read it
        }
        mma_commit(tfull(buf));  // the group's accumulator is complete
      }
    }
  } else {
    // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31, one weight row a thread
    const int q = warp & 3;
    const int rl = 32 * q + lane;
    uint64_t best[kN];
    float2 ms[CONF ? kN : 1];  // online softmax state of this thread's outputs (the confidence)
    constexpr bool want_conf = CONF;
#pragma unroll
    for (int c = 0; c < kN; ++c) {
      best[c] = 0ull;
      if (CONF) ms[CONF ? c : 0] = make_float2(-INFINITY, 0.0f);
    }
    for (int j = 0; j < ng; ++j) {
      const int buf = j & 1;
      const int64_t g = g_begin + j;
      if (!timed_out && !bar_wait(tfull(buf), (uint32_t)(j >> 1) & 1u)) timed_out = true;
      fence_after();
      float v[kN];
      tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * kN), v);
      fence_before();
      __syncwarp();
      if (lane == 0) bar_arrive(tempty(buf));
      if (crank != 0) {
        // the second block: its half of the group into the leader's inbox, once the leader has
        // read the previous group's
        if (j >= 1 && !timed_out && !bar_wait(iempty, (uint32_t)(j - 1) & 1u)) timed_out = true;
        const uint32_t dst = to_cluster(sa(inbox + rl * kN), 0);
        const uint32_t rb = to_cluster(ifull, 0);
#pragma unroll
        for (int c = 0; c < kN; c += 4)
          if (!TFD_TEST_STALL_EXCHANGE) st_async4(dst + 4u * c, v[c], v[c + 1], v[c + 2], v[c + 3], rb);
        continue;
      }
      if (warp == 2 && lane == 0) bar_expect_tx(ifull, kInboxBytes);
      if (!timed_out && !bar_wait(ifull, (uint32_t)j & 1u)) timed_out = true;
      float u[kN];
#pragma unroll
      for (int c = 0; c < kN; c += 4) {
        const float4 t = *reinterpret_cast<const float4*>(inbox + rl * kN + c);
        u[c] = t.x; u[c + 1] = t.y; u[c + 2] = t.z; u[c + 3] = t.w;
      }
#pragma unroll
      for (int c = 0; c < kN; ++c) v[c] += u[c];  // rank order: the leader's half, then the other
      __syncwarp();  // every lane has consumed its row
      if (lane == 0) bar_arrive_remote(to_cluster(iempty, 1));
      const int64_t row = g * kM + rl;
      const bool in = row < a.n;
      const int32_t id = in ? (a.id_map ? __ldg(a.id_map + row) : (int32_t)row) : 0;
      const int64_t S = (a.n + 15) / 16;
#pragma unroll
      for (int c = 0; c < kN; ++c) {
        if (c < a.rows) {  // warp-uniform
          if (in && a.y) a.y[(int64_t)c * a.ldy + row] = v[c];
          if (a.topk == 1 && in) best[c] = umax64(best[c], make_key(v[c], id));
          if (CONF && in && v[c] > -INFINITY) {  // NaN and -inf add nothing
            float2& m = ms[CONF ? c : 0];
            if (v[c] > m.x) {
              m.y = m.y * expf(m.x - v[c]) + 1.0f;
              m.x = v[c];
            } else {
              m.y += expf(v[c] - m.x);
            }
          }
          if (a.topk > 1) {  // the 16 rows of a sub-group are 16 lanes of this warp
            uint32_t m = in ? value_key(v[c]) : 0u;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            const int64_t sg = row / 16;
            if ((lane & 15) == 0 && sg < S) {
              a.submax[(int64_t)c * S + sg] = m;
              atomicMax(&spmax[c], m);
            }
          }
        }
      }
    }
    if (crank == 0 && a.topk == 1) {
      // the part's best of each activation row: lanes, then the four warps in a fixed order
      float2* sms = reinterpret_cast<float2*>(inbox);  // (the inbox is no longer written)
      // every epilogue warp has read its rows of the last group from the inbox
      asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
      for (int c = 0; c < kN; ++c) {
        uint64_t kk = best[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kk = umax64(kk, shfl_xor_u64(kk, o));
        if (lane == 0) sbest[q * kN + c] = kk;
        if (CONF) {
          float2 m = ms[CONF ? c : 0];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
            m = tfd_gemv::ms_merge(m, make_float2(__shfl_xor_sync(0xffffffffu, m.x, o),
                                                  __shfl_xor_sync(0xffffffffu, m.y, o)));
          if (lane == 0) sms[q * kN + c] = m;
        }
      }
    }
  }
  if (timed_out) set_dev_status(a.status, TFD_ERR_TIMEOUT);
  __syncthreads();
  // the pair's last remote operations are done before either block leaves
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
  if (crank != 0) return;
  if (a.topk > 1) {
    if (tid < a.rows) a.part_max[(int64_t)cid * a.rows + tid] = spmax[tid];
    return;
  }
  if (a.topk != 1) return;
  __shared__ int is_last;
  constexpr bool want_conf = CONF;
  float2* sms = reinterpret_cast<float2*>(inbox);
  float2* sjms = sms + 4 * kN;  // [warps][rows] of the join
  if (tid < a.rows) {
    uint64_t m = sbest[tid];
    for (int w = 1; w < 4; ++w) m = umax64(m, sbest[w * kN + tid]);
    a.part_keys[(int64_t)cid * a.rows + tid] = m;
    if (want_conf) {
      float2 qm = sms[tid];
      for (int w = 1; w < 4; ++w) qm = tfd_gemv::ms_merge(qm, sms[w * kN + tid]);
      a.part_ms[(int64_t)cid * a.rows + tid] = qm;
    }
  }
  if (tid < kN) sjoin[tid] = 0ull;
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(a.counter, 1u) == (uint32_t)(a.parts - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int tot = a.parts * a.rows;
  for (int i = tid; i < tot; i += kThreads)
    atomicMax(reinterpret_cast<unsigned long long*>(&sjoin[i % a.rows]),
              (unsigned long long)__ldcg(a.part_keys + i));
  if (want_conf) {
    // parts merged in a fixed order: p = tid, tid + 192, ..., then lanes, then warps
    for (int r = 0; r < a.rows; ++r) {
      float2 qm = make_float2(-INFINITY, 0.0f);
      for (int p = tid; p < a.parts; p += kThreads)
        qm = tfd_gemv::ms_merge(qm, __ldcg(a.part_ms + (int64_t)p * a.rows + r));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        qm = tfd_gemv::ms_merge(qm, make_float2(__shfl_xor_sync(0xffffffffu, qm.x, o),
                                                __shfl_xor_sync(0xffffffffu, qm.y, o)));
      if (lane == 0) sjms[warp * kN + r] = qm;
    }
  }
  __syncthreads();
  if (tid < a.rows) {
    const uint64_t key = sjoin[tid];
    a.top_vals[tid * a.ldt] = key_value(key);
    a.top_ids[tid * a.ldt] = key_id(key);
    if (want_conf) {
      float2 qm = make_float2(-INFINITY, 0.0f);
      for (int w = 0; w < kThreads / 32; ++w) qm = tfd_gemv::ms_merge(qm, sjms[w * kN + tid]);
      a.top1_conf[tid] = qm.y > 0.0f ? 1.0f / qm.y : __uint_as_float(0x7FC00000u);
    }
  }
  if (tid == 0) *a.counter = 0u;  // leave the workspace zeroed
}

// ---- host ----
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      (void)cudaGetLastError();
  });
  return fn;
}

bool map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
            uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tfd_gemv_tc

// Takes the call when it is this kernel's (bf16 weights and rows, 17-32 rows, a k range of at
// most 2048 per block of the pair in whole 64-wide blocks, fp32 logits or none, any top-k, the
// confidence); *taken = false leaves it to the register-ring kernel.
tfd_status gemv_tc_launch(const tfd_gemv::GemvArgs& g, int wfmt, int xfmt, int parts_req,
                          cudaStream_t stream, bool* taken) {
  using namespace tfd_gemv_tc;
  *taken = false;
#ifdef TFD_GEMV_TC
  if (!TFD_GEMV_TC) return TFD_OK;
#endif
  if (wfmt != TFD_W_BF16 || xfmt != TFD_X_BF16 || g.rows < 17 || g.rows > 32) return TFD_OK;
  if (g.k % (2 * kKB) != 0 || g.k / 2 > kMaxKHalf) return TFD_OK;
  if (g.topk > 1 && (g.submax == nullptr || g.part_max == nullptr || g.logits == nullptr))
    return TFD_OK;
  if (g.out_mode != TFD_OUT_NONE && g.out_mode != TFD_OUT_F32) return TFD_OK;
  if ((g.ldx * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(g.x) & 15) != 0) return TFD_OK;
  CUtensorMap tw, tx;
  if (!map_2d(&tw, g.w, (uint64_t)g.k, (uint64_t)g.n, (uint64_t)g.k * 2, kKB, kM) ||
      !map_2d(&tx, g.x, (uint64_t)g.k, (uint64_t)g.rows, (uint64_t)g.ldx * 2, kKB, kN))
    return TFD_OK;
  const bool conf = g.topk == 1 && g.top1_conf != nullptr;
  auto kern = conf ? gemv_tc_kernel<true> : gemv_tc_kernel<false>;
  static bool attr_set[2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TFD_ERR_CUDA;
  if (dev < 64 && !attr_set[conf][dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return TFD_ERR_CUDA;
    attr_set[conf][dev] = true;
  }
  TcArgs a{};
  a.n = g.n;
  a.k = g.k;
  a.rows = g.rows;
  a.ngroups = (g.n + kM - 1) / kM;
  int64_t p = parts_req > 0 ? parts_req : tfd_host::sm_count() / 2;
  if (p > a.ngroups) p = a.ngroups;
  if (p > tfd_gemv::kMaxParts) p = tfd_gemv::kMaxParts;
  a.parts = (int)p;
  // a top-k > 1 ranks the fp32 logits (in y, or in the workspace when there is no output)
  a.y = g.topk > 1 ? g.logits : g.out_mode == TFD_OUT_F32 ? reinterpret_cast<float*>(g.y) : nullptr;
  a.ldy = g.topk > 1 ? g.ld_logits : g.ldy;
  a.topk = g.topk;
  a.id_map = g.id_map;
  a.submax = g.submax;
  a.part_max = g.part_max;
  a.top1_conf = g.top1_conf;
  a.part_ms = g.part_ms;
  a.part_keys = g.part_keys;
  a.counter = g.counter;
  a.top_vals = g.top_vals;
  a.top_ids = g.top_ids;
  a.ldt = g.ldt;
  a.status = g.status;
  if (g.parts_used != nullptr) *g.parts_used = a.parts;
  *taken = true;
  kern<<<2 * a.parts, kThreads, kSmemBytes, stream>>>(tw, tx, a);
  return tfd_host::launch_status();
}
