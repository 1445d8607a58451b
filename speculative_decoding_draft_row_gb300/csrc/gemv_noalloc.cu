// gemv_noalloc.cu - tfd_head_gemv for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: serving loops that forbid allocator calls on
// the hot path (cudaMalloc can block, or synchronise the whole device, in the middle of a decode
// round), and plugins whose host framework owns all device memory and offers them no allocator.
// This entry point runs the same head GEMV as tfd_head_gemv, but its scratch is a fixed
// file-scope device array, so the caller only passes inputs and outputs.
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kMaxDevices = 64;

// The fixed scratch. Every GPU that loads this library holds it until the process exits. In host
// code this name is only a host-side stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TFD_NOALLOC_SCRATCH_BYTES];

std::mutex g_lock[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];  // set only after a successful lookup

// Device address of the scratch on the current device, looked up once per device (with that
// device current, as it is during the call that does the lookup). A failed lookup is not cached:
// its error is cleared from the runtime's last-error slot and the next call tries again.
tfd_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TFD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TFD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_lock[dev]);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return TFD_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return TFD_OK;
}

}  // namespace

extern "C" tfd_status tfd_head_gemv_noalloc(const void* w, int wfmt, const void* w_scales,
                                            int64_t n, int64_t k, const void* x, int xfmt,
                                            int rows, int64_t ldx, int out_mode, void* y,
                                            int64_t ldy, int topk, int parts,
                                            const int32_t* id_map, float* top_vals,
                                            int32_t* top_ids, int64_t ldt, float* top1_conf,
                                            int32_t* dev_status, void* stream) {
  const size_t need = tfd_head_gemv_workspace(rows, n, topk, parts);
  if (need > (size_t)TFD_NOALLOC_SCRATCH_BYTES) return TFD_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    tfd_status st = scratch_for_current_device(&ws);
    if (st != TFD_OK) return st;
    // The array keeps the previous call's contents; its arrival counters must start at zero.
    if (cudaMemsetAsync(ws, 0, need, tfd_host::as_stream(stream)) != cudaSuccess)
      return TFD_ERR_CUDA;
  }
  return tfd_head_gemv(w, wfmt, w_scales, n, k, x, xfmt, rows, ldx, out_mode, y, ldy, topk, parts,
                       id_map, top_vals, top_ids, ldt, top1_conf, ws, need, dev_status, stream);
}
