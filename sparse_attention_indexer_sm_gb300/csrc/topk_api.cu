// C ABI of the exact top-k transform: argument checks, the choice of how many
// CTAs share a row, per-device set-up, and the launch. See
// include/topk_transform.h for the contract of every entry point.

#include <atomic>
#include <climits>
#include <cstdlib>
#include <mutex>

#include "topk_select.cuh"
#include "topk_transform.h"

namespace {

using topk_gb300::Form;
using topk_gb300::Params;

constexpr int kMaxDevices = 64;
constexpr int kRowSplitUnset = INT_MIN;

std::atomic<int> g_row_split{kRowSplitUnset};
std::atomic<int> g_tie_cap{topk_gb300::kTieCapMax};
std::atomic<int> g_fast_tier{1};
thread_local int t_last_cuda_error = 0;

struct DeviceState {
  std::once_flag once;
  int sm_count = 0;
  cudaError_t err = cudaSuccess;
};
DeviceState g_devices[kMaxDevices];

int row_split_setting() {
  int v = g_row_split.load(std::memory_order_relaxed);
  if (v == kRowSplitUnset) {
    const char* e = std::getenv("TOPK_ROW_SPLIT");
    const int from_env = (e != nullptr && *e != '\0') ? std::atoi(e) : 0;
    int expected = kRowSplitUnset;
    g_row_split.compare_exchange_strong(expected, from_env);
    v = g_row_split.load(std::memory_order_relaxed);
  }
  return v;
}

// How many CTAs (one cluster) share a row. The exact kernel of the sglang
// PR #37591 page splits a row over several blocks only for small batches of long
// rows (section "关键源码片段", row_split: no split under 65536 elements, at most
// 32 blocks, none when fewer than 4). Here a split costs no extra launch (the CTAs
// of a cluster merge histograms in distributed shared memory); the rule below is
// the measured one. row_len <= 0 means unknown: treated as long.
int choose_split(int32_t batch, int64_t row_len, int sm_count) {
  const int forced = row_split_setting();
  if (forced >= 1) {
    int g = 1;
    while (g * 2 <= forced && g * 2 <= topk_gb300::kMaxCluster) g *= 2;
    return g;
  }
  // Rows up to 32768 elements run fastest on one CTA each: a cluster adds
  // barriers and distributed-shared-memory traffic that a slice this short does
  // not pay back. Longer rows get about 8192 elements per CTA, as long as the
  // grid still fits two CTAs per SM; two-CTA clusters measured slower than one
  // CTA, so a split is at least four.
  if (row_len > 0 && row_len <= 32768) return 1;
  const int64_t len = row_len > 0 ? row_len : INT64_C(1) << 30;
  const int64_t slots = static_cast<int64_t>(sm_count) * 2;
  int g = 1;
  while (g < topk_gb300::kMaxCluster && len / (g * 2) >= 8192) g *= 2;
  while (g > 1 && static_cast<int64_t>(batch) * g > slots) g /= 2;
  return g >= 4 ? g : 1;
}

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return TOPK_ERR_CUDA;
}

int run(Form form, Params p, int64_t row_len_hint, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return fail_cuda(cudaErrorInvalidDevice);
  DeviceState& ds = g_devices[dev];
  std::call_once(ds.once, [&ds, dev]() {
    ds.err = cudaDeviceGetAttribute(&ds.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (ds.err == cudaSuccess) ds.err = topk_gb300::prepare_device();
  });
  if (ds.err != cudaSuccess) return fail_cuda(ds.err);
  const int g = choose_split(p.batch, row_len_hint, ds.sm_count);
  if (static_cast<int64_t>(p.batch) * g > INT_MAX) return TOPK_ERR_INVALID_ARGUMENT;
  p.tie_cap = g_tie_cap.load(std::memory_order_relaxed);
  p.use_filter = g_fast_tier.load(std::memory_order_relaxed);
  e = topk_gb300::launch(form, p, g, stream);
  if (e != cudaSuccess) return fail_cuda(e);
  return TOPK_OK;
}

int check_common(const float* scores, const int32_t* seq_lens, int32_t batch, int32_t k,
                 const int32_t* out) {
  if (batch < 0) return TOPK_ERR_INVALID_ARGUMENT;
  if (k < 1 || k > TOPK_MAX_K) return TOPK_ERR_UNSUPPORTED_K;
  if (batch == 0) return TOPK_OK;
  if (scores == nullptr || seq_lens == nullptr || out == nullptr) return TOPK_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(scores) & 3u) != 0) return TOPK_ERR_INVALID_ARGUMENT;
  return TOPK_OK;
}

Params base_params(const float* scores, const int32_t* seq_lens, int32_t batch, int32_t k,
                   int32_t* out) {
  Params p = {};
  p.scores = scores;
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.k = k;
  p.out = out;
  p.page_size = 1;
  p.page_shift = 0;
  return p;
}

}  // namespace

extern "C" {

size_t topk_workspace_bytes(int32_t /*batch*/, int64_t /*max_row_len*/, int32_t /*k*/) {
  return 0;
}

int topk_transform_raw(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                       int32_t batch, int32_t k, int32_t* out, void* /*workspace*/,
                       size_t /*workspace_bytes*/, cudaStream_t stream) {
  const int st = check_common(scores, seq_lens, batch, k, out);
  if (st != TOPK_OK || batch == 0) return st;
  if (row_stride < 1) return TOPK_ERR_INVALID_ARGUMENT;
  Params p = base_params(scores, seq_lens, batch, k, out);
  p.row_stride = row_stride;
  return run(topk_gb300::kRaw, p, row_stride, stream);
}

int topk_transform_paged(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                         const int32_t* page_table, int64_t page_table_stride,
                         int32_t page_size, int32_t batch, int32_t k, int32_t* out,
                         void* /*workspace*/, size_t /*workspace_bytes*/, cudaStream_t stream) {
  const int st = check_common(scores, seq_lens, batch, k, out);
  if (st != TOPK_OK || batch == 0) return st;
  if (row_stride < 1 || page_table == nullptr || page_table_stride < 1 || page_size < 1)
    return TOPK_ERR_INVALID_ARGUMENT;
  Params p = base_params(scores, seq_lens, batch, k, out);
  p.row_stride = row_stride;
  p.page_table = page_table;
  p.pt_stride = page_table_stride;
  p.page_size = page_size;
  p.page_shift = (page_size & (page_size - 1)) == 0 ? __builtin_ctz(page_size) : -1;
  return run(topk_gb300::kPaged, p, row_stride, stream);
}

int topk_transform_ragged(const float* scores, const int32_t* row_starts,
                          const int32_t* seq_lens, int64_t max_row_len_hint, int32_t batch,
                          int32_t k, int32_t* out, void* /*workspace*/,
                          size_t /*workspace_bytes*/, cudaStream_t stream) {
  const int st = check_common(scores, seq_lens, batch, k, out);
  if (st != TOPK_OK || batch == 0) return st;
  if (row_starts == nullptr || max_row_len_hint < 0) return TOPK_ERR_INVALID_ARGUMENT;
  Params p = base_params(scores, seq_lens, batch, k, out);
  p.row_starts = row_starts;
  return run(topk_gb300::kRagged, p, max_row_len_hint, stream);
}

int topk_transform_window(const float* scores, int64_t row_stride, const int32_t* starts,
                          const int32_t* seq_lens, int32_t batch, int32_t k, int32_t* out,
                          void* /*workspace*/, size_t /*workspace_bytes*/, cudaStream_t stream) {
  const int st = check_common(scores, seq_lens, batch, k, out);
  if (st != TOPK_OK || batch == 0) return st;
  if (row_stride < 1 || starts == nullptr) return TOPK_ERR_INVALID_ARGUMENT;
  Params p = base_params(scores, seq_lens, batch, k, out);
  p.row_stride = row_stride;
  p.row_starts = starts;
  return run(topk_gb300::kWindow, p, row_stride, stream);
}

const char* topk_status_string(int status) {
  switch (status) {
    case TOPK_OK: return "ok";
    case TOPK_ERR_INVALID_ARGUMENT: return "invalid argument";
    case TOPK_ERR_UNSUPPORTED_K: return "unsupported k (must be in [1, TOPK_MAX_K])";
    case TOPK_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case TOPK_ERR_CUDA: return "CUDA error (see topk_last_cuda_error)";
    default: return "unknown status";
  }
}

int topk_last_cuda_error(void) { return t_last_cuda_error; }

int topk_set_row_split(int g) {
  const int prev = row_split_setting();
  g_row_split.store(g < 1 ? 0 : g, std::memory_order_relaxed);
  return prev < 1 ? 0 : prev;
}

int topk_set_fast_tier(int enable) {
  return g_fast_tier.exchange(enable != 0 ? 1 : 0, std::memory_order_relaxed);
}

int topk_set_tie_capacity(int cap) {
  if (cap < 0) cap = 0;
  if (cap > TOPK_TIE_CAPACITY_MAX) cap = TOPK_TIE_CAPACITY_MAX;
  return g_tie_cap.exchange(cap, std::memory_order_relaxed);
}

}  // extern "C"
