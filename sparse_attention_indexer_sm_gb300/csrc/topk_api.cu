// C ABI of the exact top-k transform: argument checks, the choice of how many
// CTAs share a row, per-device set-up, and the launch. See
// include/topk_transform.h for the contract of every entry point.

#include <algorithm>
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
std::atomic<int> g_cta_threads{0};  // 0: automatic; 512 or 256: that build
std::atomic<int> g_staged{1};       // staged tier: 0 off, 1 automatic, 2 whole row, 3 half
std::atomic<int> g_chip_split{1};   // chip-wide split: 0 off, 1 automatic, 2 wherever it can run

// The scratch of topk_transform_grouped_static: part of the module, one per device.
// Host code must not hand this name to a kernel: on the host it is only a stand-in
// for the symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_stage[TOPK_STATIC_WORKSPACE_BYTES];
thread_local int t_last_cuda_error = 0;

struct DeviceState {
  std::once_flag once;
  int sm_count = 0;
  cudaError_t err = cudaSuccess;
  // The static scratch's device address, stored once a lookup has succeeded (a
  // failed lookup is not remembered: the next call tries again).
  std::mutex stage_mu;
  std::atomic<void*> stage{nullptr};
  // clusters of 4, 8 and 16 CTAs the device holds at once (0: not known)
  int clusters4 = 0, clusters8 = 0, clusters16 = 0;
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
int choose_split(int64_t batch, int64_t row_len, const DeviceState& ds) {
  const int sm_count = ds.sm_count;
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
  while (g > 1 && batch * g > slots) g /= 2;
  // and the rows' clusters resident at once: the hardware places a cluster within one
  // GPC, so fewer clusters of 16 fit than SMs alone allow (C4, 16 rows of 65536-262144
  // elements: a second wave of clusters at G = 16)
  auto fits = [&](int gg) {
    const int n = gg == 16 ? ds.clusters16 : gg == 8 ? ds.clusters8 : gg == 4 ? ds.clusters4 : 0;
    return n <= 0 || batch <= n;
  };
  while (g > 4 && !fits(g)) g /= 2;
  return g >= 4 ? g : 1;
}

// Launches of more rows than two 512-thread CTAs per SM hold take the 256-thread
// build (four CTAs per SM, so each SM overlaps more rows) when one CTA owns a row,
// every problem's candidates fit that build's smaller buffer (k <= 1024), and
// either the rows are at most 8192 elements or there are at least 16 rows per SM
// (four waves of it). Measured: with shorter rows or enough waves the extra rows
// in flight win; 1024 rows of 32768 (under two waves) run faster on the 512-thread
// build, whose shorter per-row chain leaves a shorter last wave. row_len <= 0
// means unknown.
bool use_cta256(int64_t rows, int64_t row_len, int g, int32_t k_max, int sm_count) {
  const int forced = g_cta_threads.load(std::memory_order_relaxed);
  if (forced != 0) return forced == 256;
  const int64_t sms = sm_count;
  return g == 1 && rows > 2 * sms && k_max <= 1024 &&
         ((row_len > 0 && row_len <= 8192) || rows >= 16 * sms);
}

// Single-CTA rows of a known length of at most 32768 elements may run on the staged
// tier of the 512-thread build (the row copied to shared memory from kernel start).
// Returns 1 for the whole row staged (one CTA per SM), 2 for half a row (two CTAs per
// SM), 0 for the streaming tiers. Automatically, launches of 64 rows up to one per
// SM whose rows may hold 16384 elements or more take the whole-row variant (measured:
// faster there; fewer or shorter rows, and launches of more rows, are faster on the
// streaming tier).
int use_staged(int g, int64_t rows, int64_t row_len, int use_filter, int sm_count) {
  const int mode = g_staged.load(std::memory_order_relaxed);
  if (g != 1 || use_filter == 0 || mode == 0 || !topk_gb300::cta512::staged_fits(row_len)) return 0;
  if (mode == 2) return 1;
  if (mode == 3) return 2;
  return rows >= 64 && rows <= sm_count && row_len >= 16384 ? 1 : 0;
}

// The chip-wide split of a call's rows: CTAs per row (0: the split is not used) and
// the candidate capacities, from the tie capacity (so that small capacities also
// exercise its fallback). Automatically, batches of 4 rows up to one row per 16 SMs,
// rows of at least 65536 elements: there one cluster of 16 CTAs per row leaves most
// of the chip idle. Measured on 262144-element rows (k = 2048): 4 rows 13.9 against
// 16.7 us on clusters; 2 rows 13.8 against 13.7 us and one row 14.1 against 13.7 us,
// where the clusters keep the rows. The CTAs per row are the largest power of two
// that keeps the filter launch within two CTAs per SM and each CTA's slice at 2048
// elements or more (forced: any batch and length, at least one CTA per row).
struct SplitPlan {
  int parts = 0, cap = 0, gather_cap = 0;
};
SplitPlan split_plan(int64_t batch, int64_t row_len, int sm_count, int tie_cap) {
  SplitPlan plan;
  const int mode = g_chip_split.load(std::memory_order_relaxed);
  if (mode == 0 || batch < 1) return plan;
  const int64_t len = row_len > 0 ? row_len : INT64_C(1) << 30;
  if (mode == 1 && (len < 65536 || batch < 4 || batch * 16 > sm_count)) return plan;
  int s = 1;
  while (s * 2 <= topk_gb300::kMaxSplit && batch * s * 2 <= 2 * static_cast<int64_t>(sm_count) &&
         len / (s * 2) >= 2048)
    s *= 2;
  if (mode == 1 && s < 8) return plan;
  plan.parts = s;
  plan.cap = std::min(topk_gb300::kSplitCapMax, std::max(tie_cap, 0));
  plan.gather_cap = std::min(topk_gb300::kGatherCapMax, 4 * std::max(tie_cap, 0));
  return plan;
}

int fail_cuda(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return TOPK_ERR_CUDA;
}

// The current device's state, set up on first use (SM count, kernel attributes).
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return fail_cuda(cudaErrorInvalidDevice);
  DeviceState& ds = g_devices[dev];
  std::call_once(ds.once, [&ds, dev]() {
    ds.err = cudaDeviceGetAttribute(&ds.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (ds.err == cudaSuccess) ds.err = topk_gb300::cta512::prepare_device();
    if (ds.err == cudaSuccess) ds.err = topk_gb300::cta256::prepare_device();
    // a failed query leaves the count unknown (the split then ignores it)
    if (ds.err == cudaSuccess) {
      if (topk_gb300::cta512::max_active_clusters(4, &ds.clusters4) != cudaSuccess) ds.clusters4 = 0;
      if (topk_gb300::cta512::max_active_clusters(8, &ds.clusters8) != cudaSuccess) ds.clusters8 = 0;
      if (topk_gb300::cta512::max_active_clusters(16, &ds.clusters16) != cudaSuccess) ds.clusters16 = 0;
      (void)cudaGetLastError();  // a failed query leaves no sticky error
    }
  });
  if (ds.err != cudaSuccess) return fail_cuda(ds.err);
  *out = &ds;
  return TOPK_OK;
}

// Checks one problem on the host and fills its kernel parameters; *len_hint gets
// the longest row it can have (for the row split). Nothing in device memory is
// read.
int build_params(const topk_problem_t& q, Params* p, int64_t* len_hint) {
  if (q.batch < 0) return TOPK_ERR_INVALID_ARGUMENT;
  if (q.k < 1 || q.k > TOPK_MAX_K) return TOPK_ERR_UNSUPPORTED_K;
  if (q.form < TOPK_FORM_RAW || q.form > TOPK_FORM_WINDOW) return TOPK_ERR_INVALID_ARGUMENT;
  if ((q.flags & ~TOPK_FLAG_SORTED) != 0u || q.reserved != 0u) return TOPK_ERR_INVALID_ARGUMENT;
  *p = Params{};
  p->batch = q.batch;
  p->k = q.k;
  p->page_size = 1;
  p->page_shift = 0;
  if (q.batch == 0) return TOPK_OK;
  if (q.scores == nullptr || q.seq_lens == nullptr || q.out == nullptr)
    return TOPK_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(q.scores) & 3u) != 0) return TOPK_ERR_INVALID_ARGUMENT;
  p->scores = q.scores;
  p->seq_lens = q.seq_lens;
  p->out = q.out;
  p->values = q.values;
  if (q.form == TOPK_FORM_RAGGED) {
    if (q.row_starts == nullptr || q.max_row_len_hint < 0) return TOPK_ERR_INVALID_ARGUMENT;
    p->row_starts = q.row_starts;
    *len_hint = q.max_row_len_hint;
    return TOPK_OK;
  }
  if (q.row_stride < 1) return TOPK_ERR_INVALID_ARGUMENT;
  p->row_stride = q.row_stride;
  *len_hint = q.row_stride;
  if (q.form == TOPK_FORM_PAGED) {
    if (q.page_table == nullptr || q.page_table_stride < 1 || q.page_size < 1)
      return TOPK_ERR_INVALID_ARGUMENT;
    p->page_table = q.page_table;
    p->pt_stride = q.page_table_stride;
    p->page_size = q.page_size;
    p->page_shift = (q.page_size & (q.page_size - 1)) == 0 ? __builtin_ctz(q.page_size) : -1;
  } else if (q.form == TOPK_FORM_WINDOW) {
    if (q.row_starts == nullptr || q.max_row_len_hint < 0) return TOPK_ERR_INVALID_ARGUMENT;
    p->row_starts = q.row_starts;
    if (q.max_row_len_hint > 0 && q.max_row_len_hint < q.row_stride)
      *len_hint = q.max_row_len_hint;
  }
  return TOPK_OK;
}

// The process-wide knobs, read once per call (every problem of a launch must see
// the same tie capacity: it sizes the launch's shared memory).
struct Settings {
  int tie_cap, use_filter;
};
Settings settings() {
  return Settings{g_tie_cap.load(std::memory_order_relaxed),
                  g_fast_tier.load(std::memory_order_relaxed)};
}
void apply_settings(const Settings& s, Params* p) {
  p->tie_cap = s.tie_cap;
  p->use_filter = s.use_filter;
}

int run_one(const topk_problem_t& q, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Params p;
  int64_t hint = 0;
  int st = build_params(q, &p, &hint);
  if (st != TOPK_OK || q.batch == 0) return st;
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != TOPK_OK) return st;
  const int g = choose_split(p.batch, hint, *ds);
  if (static_cast<int64_t>(p.batch) * g > INT_MAX) return TOPK_ERR_INVALID_ARGUMENT;
  apply_settings(settings(), &p);
  cudaError_t e;
  // the chip-wide split, when planned and the caller's workspace holds it
  const SplitPlan plan = split_plan(p.batch, hint, ds->sm_count, p.tie_cap);
  if (plan.parts > 0 && p.use_filter != 0 && workspace != nullptr &&
      (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0 &&
      workspace_bytes >= topk_gb300::split_workspace_bytes(p.batch, plan.parts, plan.cap) &&
      static_cast<int64_t>(p.batch) * plan.parts <= INT_MAX) {
    p.split_ws = workspace;
    p.split_s = plan.parts;
    p.split_cap = plan.cap;
    p.gather_cap = plan.gather_cap;
    // the select kernel's cluster: the row split the clusters would take (its exact tier
    // runs there when a row's candidates do not fit)
    p.split_g = std::max(g, 1);
    e = topk_gb300::cta512::launch_split(static_cast<Form>(q.form), p, stream);
    return e == cudaSuccess ? TOPK_OK : fail_cuda(e);
  }
  if (use_cta256(p.batch, hint, g, p.k, ds->sm_count)) {
    p.tie_cap = std::min(p.tie_cap, topk_gb300::kTieCap256);
    e = topk_gb300::cta256::launch(static_cast<Form>(q.form), p, g, p.batch > ds->sm_count, 0,
                                   stream);
  } else {
    // more rows than SMs: SMs hold two CTAs and the candidates' L2 read-back
    // contends, so the filter reads them back from L1 instead (measured); rows that
    // fit in shared memory take the staged tier
    e = topk_gb300::cta512::launch(static_cast<Form>(q.form), p, g, p.batch > ds->sm_count,
                                   use_staged(g, p.batch, hint, p.use_filter, ds->sm_count), stream);
  }
  return e == cudaSuccess ? TOPK_OK : fail_cuda(e);
}

// Bytes of the sorted problems' staging areas (each batch * k pairs of 8 bytes,
// rounded up to 256); offsets[i] (if given) gets problem i's offset.
size_t staging_bytes(const topk_problem_t* problems, int32_t n, size_t* offsets) {
  size_t total = 0;
  for (int i = 0; i < n; ++i) {
    if (offsets != nullptr) offsets[i] = total;
    const topk_problem_t& q = problems[i];
    if ((q.flags & TOPK_FLAG_SORTED) == 0u || q.batch <= 0 || q.k <= 0) continue;
    const size_t bytes = static_cast<size_t>(q.batch) * static_cast<size_t>(q.k) * 8u;
    total += (bytes + 255u) / 256u * 256u;
  }
  return total;
}

// The checks of a grouped call, in order: the array, then each problem. Fills the
// problems' kernel parameters, row-length hints and the rows of each form.
int check_group(const topk_problem_t* problems, int32_t n_problems, Params* params,
                int64_t* hints, int64_t* rows_of_form) {
  static_assert(TOPK_MAX_GROUP <= topk_gb300::kMaxGroup, "group limit");
  static_assert(TOPK_MAX_K == topk_gb300::kMaxK, "largest k");
  if (n_problems < 0 || n_problems > TOPK_MAX_GROUP) return TOPK_ERR_INVALID_ARGUMENT;
  if (n_problems > 0 && problems == nullptr) return TOPK_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < n_problems; ++i) {
    hints[i] = 0;
    const int st = build_params(problems[i], &params[i], &hints[i]);
    if (st != TOPK_OK) return st;
    rows_of_form[problems[i].form] += problems[i].batch;
  }
  return TOPK_OK;
}

topk_problem_t problem(int32_t form, const float* scores, int64_t row_stride,
                       const int32_t* seq_lens, int32_t batch, int32_t k, int32_t* out) {
  topk_problem_t q = {};
  q.form = form;
  q.scores = scores;
  q.row_stride = row_stride;
  q.seq_lens = seq_lens;
  q.batch = batch;
  q.k = k;
  q.out = out;
  return q;
}

}  // namespace

extern "C" {

size_t topk_workspace_bytes(int32_t batch, int64_t max_row_len, int32_t /*k*/) {
  if (batch < 1) return 0;
  DeviceState* ds = nullptr;
  if (device_state(&ds) != TOPK_OK) return 0;
  const SplitPlan plan =
      split_plan(batch, max_row_len, ds->sm_count, g_tie_cap.load(std::memory_order_relaxed));
  if (plan.parts == 0 || g_fast_tier.load(std::memory_order_relaxed) == 0) return 0;
  return topk_gb300::split_workspace_bytes(batch, plan.parts, plan.cap);
}

size_t topk_problem_bytes(void) { return sizeof(topk_problem_t); }

size_t topk_problem_workspace_bytes(const topk_problem_t* problems, int32_t n_problems) {
  if (problems == nullptr || n_problems < 0 || n_problems > TOPK_MAX_GROUP) return 0;
  return staging_bytes(problems, n_problems, nullptr);
}

int topk_transform_raw(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                       int32_t batch, int32_t k, int32_t* out, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
  return run_one(problem(TOPK_FORM_RAW, scores, row_stride, seq_lens, batch, k, out), workspace,
                 workspace_bytes, stream);
}

int topk_transform_paged(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                         const int32_t* page_table, int64_t page_table_stride,
                         int32_t page_size, int32_t batch, int32_t k, int32_t* out,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  topk_problem_t q = problem(TOPK_FORM_PAGED, scores, row_stride, seq_lens, batch, k, out);
  q.page_table = page_table;
  q.page_table_stride = page_table_stride;
  q.page_size = page_size;
  return run_one(q, workspace, workspace_bytes, stream);
}

int topk_transform_ragged(const float* scores, const int32_t* row_starts,
                          const int32_t* seq_lens, int64_t max_row_len_hint, int32_t batch,
                          int32_t k, int32_t* out, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  topk_problem_t q = problem(TOPK_FORM_RAGGED, scores, 0, seq_lens, batch, k, out);
  q.row_starts = row_starts;
  q.max_row_len_hint = max_row_len_hint;
  return run_one(q, workspace, workspace_bytes, stream);
}

int topk_transform_window(const float* scores, int64_t row_stride, const int32_t* starts,
                          const int32_t* seq_lens, int64_t max_row_len_hint, int32_t batch,
                          int32_t k, int32_t* out, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  topk_problem_t q = problem(TOPK_FORM_WINDOW, scores, row_stride, seq_lens, batch, k, out);
  q.row_starts = starts;
  q.max_row_len_hint = max_row_len_hint;
  return run_one(q, workspace, workspace_bytes, stream);
}

int topk_transform_grouped(const topk_problem_t* problems, int32_t n_problems,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  // every problem is checked before anything is launched
  Params params[TOPK_MAX_GROUP];
  int64_t hints[TOPK_MAX_GROUP];
  int64_t rows_of_form[4] = {0, 0, 0, 0};
  const int checked = check_group(problems, n_problems, params, hints, rows_of_form);
  if (checked != TOPK_OK) return checked;
  // sorted problems stage (key, position) pairs in the workspace
  size_t offsets[TOPK_MAX_GROUP];
  const size_t need = staging_bytes(problems, n_problems, offsets);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return workspace_bytes < need ? TOPK_ERR_WORKSPACE_TOO_SMALL : TOPK_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < n_problems; ++i)
      if ((problems[i].flags & TOPK_FLAG_SORTED) != 0u && problems[i].batch > 0)
        params[i].staged = reinterpret_cast<uint2*>(static_cast<char*>(workspace) + offsets[i]);
  }
  DeviceState* ds = nullptr;
  bool any = false;
  for (int f = 0; f < 4; ++f) any = any || rows_of_form[f] > 0;
  if (!any) return TOPK_OK;
  int st = device_state(&ds);
  if (st != TOPK_OK) return st;
  const Settings knobs = settings();
  for (int f = 0; f < 4; ++f) {
    if (rows_of_form[f] == 0) continue;
    topk_gb300::GroupParams gp;
    gp.n = 0;
    int64_t rows = 0, hint = 0;
    for (int i = 0; i < n_problems; ++i) {
      if (problems[i].form != f || problems[i].batch == 0) continue;
      apply_settings(knobs, &params[i]);
      gp.probs[gp.n] = params[i];
      gp.row_begin[gp.n] = static_cast<int32_t>(rows);
      rows += problems[i].batch;
      // the longest row decides the split; ragged rows of unknown length count as long
      hint = (hint < 0 || hints[i] <= 0) ? -1 : (hints[i] > hint ? hints[i] : hint);
      ++gp.n;
    }
    const int g = choose_split(rows, hint < 0 ? 0 : hint, *ds);
    if (rows * g > INT_MAX) return TOPK_ERR_INVALID_ARGUMENT;
    gp.row_begin[gp.n] = static_cast<int32_t>(rows);
    int32_t k_max = 0;
    bool opts = false;  // the values output or the sorted option
    for (int i = 0; i < gp.n; ++i) {
      k_max = std::max(k_max, gp.probs[i].k);
      opts = opts || gp.probs[i].values != nullptr || gp.probs[i].staged != nullptr;
    }
    cudaError_t e;
    if (use_cta256(rows, hint, g, k_max, ds->sm_count)) {
      for (int i = 0; i < gp.n; ++i)
        gp.probs[i].tie_cap = std::min(gp.probs[i].tie_cap, topk_gb300::kTieCap256);
      e = topk_gb300::cta256::launch_group(static_cast<Form>(f), gp, g, opts,
                                           rows > ds->sm_count, 0, stream);
    } else {
      e = topk_gb300::cta512::launch_group(static_cast<Form>(f), gp, g, opts,
                                           rows > ds->sm_count,
                                           use_staged(g, rows, hint, knobs.use_filter, ds->sm_count),
                                           stream);
    }
    if (e != cudaSuccess) return fail_cuda(e);
  }
  for (int i = 0; i < n_problems; ++i) {  // the sort pass of each sorted problem
    if (params[i].staged == nullptr) continue;
    apply_settings(knobs, &params[i]);
    const cudaError_t e =
        topk_gb300::cta512::sort_rows(static_cast<Form>(problems[i].form), params[i], stream);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return TOPK_OK;
}

int topk_transform_grouped_static(const topk_problem_t* problems, int32_t n_problems,
                                  cudaStream_t stream) {
  {  // every problem first, as the workspace call does, then the array's limit
    Params params[TOPK_MAX_GROUP];
    int64_t hints[TOPK_MAX_GROUP];
    int64_t rows_of_form[4] = {0, 0, 0, 0};
    const int checked = check_group(problems, n_problems, params, hints, rows_of_form);
    if (checked != TOPK_OK) return checked;
  }
  const size_t need = staging_bytes(problems, n_problems, nullptr);
  if (need > TOPK_STATIC_WORKSPACE_BYTES) return TOPK_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (need > 0) {
    DeviceState* ds = nullptr;  // loads the module on this device first
    const int st = device_state(&ds);
    if (st != TOPK_OK) return st;
    // The array's device address, looked up with its device current (device_state
    // keyed the state by the current device) and kept only once the lookup worked.
    scratch = ds->stage.load(std::memory_order_acquire);
    if (scratch == nullptr) {
      std::lock_guard<std::mutex> lock(ds->stage_mu);
      scratch = ds->stage.load(std::memory_order_acquire);
      if (scratch == nullptr) {
        const cudaError_t e = cudaGetSymbolAddress(&scratch, g_static_stage);
        if (e != cudaSuccess) return fail_cuda(e);
        ds->stage.store(scratch, std::memory_order_release);
      }
    }
  }
  return topk_transform_grouped(problems, n_problems, scratch, need > 0 ? need : 0, stream);
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

int topk_guard_hits(uint64_t* hits) {
  if (hits == nullptr) return TOPK_ERR_INVALID_ARGUMENT;
  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != TOPK_OK) return st;
  unsigned int a = 0, b = 0;
  cudaError_t e = topk_gb300::cta512::guard_hits(&a);
  if (e == cudaSuccess) e = topk_gb300::cta256::guard_hits(&b);
  if (e != cudaSuccess) return fail_cuda(e);
  *hits = static_cast<uint64_t>(a) + b;
  return TOPK_OK;
}

int topk_reset_guard_hits(void) {
  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != TOPK_OK) return st;
  cudaError_t e = topk_gb300::cta512::reset_guard_hits();
  if (e == cudaSuccess) e = topk_gb300::cta256::reset_guard_hits();
  return e == cudaSuccess ? TOPK_OK : fail_cuda(e);
}

int topk_set_row_split(int g) {
  const int prev = row_split_setting();
  g_row_split.store(g < 1 ? 0 : g, std::memory_order_relaxed);
  return prev < 1 ? 0 : prev;
}

int topk_set_fast_tier(int enable) {
  return g_fast_tier.exchange(enable != 0 ? 1 : 0, std::memory_order_relaxed);
}

int topk_set_staged_tier(int mode) {
  return g_staged.exchange(mode >= 0 && mode <= 3 ? mode : 1, std::memory_order_relaxed);
}

int topk_set_chip_split(int mode) {
  return g_chip_split.exchange(mode >= 0 && mode <= 2 ? mode : 1, std::memory_order_relaxed);
}

int topk_set_cta_threads(int threads) {
  return g_cta_threads.exchange(threads == 512 || threads == 256 ? threads : 0,
                                std::memory_order_relaxed);
}

int topk_set_tie_capacity(int cap) {
  if (cap < 0) cap = 0;
  if (cap > TOPK_TIE_CAPACITY_MAX) cap = TOPK_TIE_CAPACITY_MAX;
  return g_tie_cap.exchange(cap, std::memory_order_relaxed);
}

}  // extern "C"
