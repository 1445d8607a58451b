// accept.cu - accept-prefix count of a verify round, with per-position asked/kept histograms.
//
// Follows the TFE draft head page (#42), commit "... rnel test TF_DS_ACCEPT_LOG=N": a draft is kept
// when it and every earlier draft equal the round's draws; the log reports the drafts asked and
// kept at each window position. Only drafts are counted (not the verifier's bonus token).
#include "common.cuh"

namespace {

using namespace tfd;

__global__ void __launch_bounds__(256)
accept_kernel(const int32_t* __restrict__ drafts, const int32_t* __restrict__ n_asked,
              const int32_t* __restrict__ draws, int streams, int win, int32_t* __restrict__ n_kept,
              unsigned long long* asked_hist, unsigned long long* kept_hist, int32_t* dev_status) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= streams) return;
  const int na = n_asked[s];
  if (na < 0 || na > win) {
    n_kept[s] = 0;
    set_dev_status(dev_status, TFD_ERR_DEVICE_DATA);
    return;
  }
  const int32_t* d = drafts + (int64_t)s * win;
  const int32_t* w = draws + (int64_t)s * win;
  int kept = 0;
  while (kept < na && d[kept] == w[kept]) ++kept;
  n_kept[s] = kept;
  if (asked_hist) {
    for (int i = 0; i < na; ++i) atomicAdd(asked_hist + i, 1ull);
    for (int i = 0; i < kept; ++i) atomicAdd(kept_hist + i, 1ull);
  }
}

}  // namespace

extern "C" tfd_status tfd_accept(const int32_t* drafts, const int32_t* n_asked,
                                 const int32_t* draws, int streams, int win, int32_t* n_kept,
                                 int64_t* asked_hist, int64_t* kept_hist, int32_t* dev_status,
                                 void* stream) {
  using tfd_host::aligned;
  if (!drafts || !n_asked || !draws || !n_kept) return TFD_ERR_INVALID;
  if (streams < 1 || win < 1 || win > TFD_MAX_TOPK) return TFD_ERR_INVALID;
  if ((asked_hist == nullptr) != (kept_hist == nullptr)) return TFD_ERR_INVALID;
  if (!aligned(drafts, 4) || !aligned(n_asked, 4) || !aligned(draws, 4) || !aligned(n_kept, 4))
    return TFD_ERR_INVALID;
  if (asked_hist && (!aligned(asked_hist, 8) || !aligned(kept_hist, 8))) return TFD_ERR_INVALID;
  const int threads = 256;
  const int blocks = (streams + threads - 1) / threads;
  accept_kernel<<<blocks, threads, 0, tfd_host::as_stream(stream)>>>(
      drafts, n_asked, draws, streams, win, n_kept,
      reinterpret_cast<unsigned long long*>(asked_hist),
      reinterpret_cast<unsigned long long*>(kept_hist), dev_status);
  return tfd_host::launch_status();
}
