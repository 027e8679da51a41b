// Internal interface between the C ABI (topk_api.cu) and the kernels
// (topk_select.cu). Not installed; the public interface is include/topk_transform.h.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace topk_gb300 {

enum Form : int { kRaw = 0, kPaged = 1, kRagged = 2, kWindow = 3 };

constexpr int kMaxBins = 4096;         // widest histogram (12 key bits)
constexpr int kMaxK = 2048;            // largest k (TOPK_MAX_K of the public header)
constexpr int kTieCapMax = 4096;       // shared tie buffer entries, 8 bytes each
constexpr int kMaxCluster = 16;        // CTAs per row (non-portable cluster size)

struct Params {
  const float* scores;
  int64_t row_stride;          // raw, paged, window: elements between row starts
  const int32_t* seq_lens;     // [batch]
  const int32_t* row_starts;   // ragged: row offsets [batch]; window: window starts [batch]
  const int32_t* page_table;   // paged: [batch, pt_stride]
  int64_t pt_stride;
  int32_t page_size;
  int32_t page_shift;          // log2(page_size) when it is a power of two, else -1
  int32_t* out;                // [batch, k]
  float* values;               // [batch, k] or null: each slot's score, -inf in padding slots
  uint2* staged;               // [batch, k] or null: (key, position) per slot instead of out
                               // and values, for the sort pass (sort_rows) to order and write
  int32_t k;
  int32_t tie_cap;             // <= kTieCapMax
  int32_t batch;
  int32_t use_filter;          // 1: try the sampled-threshold filter pass first
  // chip-wide split (split_s > 0): split_s CTAs per row filter their slices into the
  // workspace split_ws (split_workspace_bytes), a second kernel selects per row
  void* split_ws;
  int32_t split_s;             // CTAs per row: a power of two, at most kMaxSplit
  int32_t split_cap;           // candidates one filter CTA may store
  int32_t gather_cap;          // candidates the select CTA may gather
  int32_t split_g;             // CTAs of the select cluster (its exact tier's row split)
};

// The chip-wide split's workspace for `rows` rows of `s` CTAs storing up to `cap`
// candidates each: per row the threshold and bin width (uint2), per CTA its
// candidate count (int32), per CTA `cap` (key, position) pairs; each part 256-byte
// aligned.
constexpr int kMaxSplit = 256;
constexpr int kSplitCapMax = 256;     // candidates one filter CTA may store, at most
constexpr int kGatherCapMax = 16384;  // candidates the select CTA may gather, at most
__host__ __device__ constexpr size_t split_align(size_t b) { return (b + 255u) / 256u * 256u; }
__host__ __device__ constexpr size_t split_counts_offset(int64_t rows) { return split_align(8u * static_cast<size_t>(rows)); }
__host__ __device__ constexpr size_t split_entries_offset(int64_t rows, int s) {
  return split_counts_offset(rows) + split_align(4u * static_cast<size_t>(rows) * static_cast<size_t>(s));
}
__host__ __device__ constexpr size_t split_workspace_bytes(int64_t rows, int s, int cap) {
  return split_entries_offset(rows, s) +
         split_align(8u * static_cast<size_t>(rows) * static_cast<size_t>(s) * static_cast<size_t>(cap));
}

// Problems of one form sharing a launch (kMaxGroup at most; row_begin holds the
// prefix sums of their batches, row_begin[n] = all rows). Passed by value as a
// kernel parameter.
constexpr int kMaxGroup = 32;
struct GroupParams {
  int32_t n;
  int32_t row_begin[kMaxGroup + 1];
  Params probs[kMaxGroup];
};

// The kernels are built for two CTA sizes (topk_select.cu): cta512 has 512-thread
// CTAs, two per SM; cta256 has 256-thread CTAs, four per SM, and takes tie
// capacities up to kTieCap256 only. Each build exports the same functions.
constexpr int kTieCap256 = 3072;

#define TOPK_CTA_INTERFACE                                                              \
  /* Dynamic shared memory one CTA needs for a cluster of `g` CTAs. */                  \
  size_t smem_bytes(int g, int tie_cap);                                                \
  /* One-time per-device function attributes (max dynamic smem, cluster size 16). */    \
  cudaError_t prepare_device();                                                         \
  /* Enqueue the kernel: grid = batch * g CTAs in clusters of g along x. With g = 1, */  \
  /* staged = 1 (whole row staged, one CTA per SM) or 2 (half a row, two per SM) */     \
  /* picks the staged tier (rows for which staged_fits holds; p.use_filter set), */     \
  /* else keys_in_filter the variant that reads candidates back from L1 in the */       \
  /* filter (faster once SMs hold two CTAs each). */                                    \
  cudaError_t launch(Form form, const Params& p, int g, bool keys_in_filter, int staged, \
                     cudaStream_t stream);                                              \
  /* Whether rows of at most row_len elements (0: unknown) can run on this build's */  \
  /* staged tier (whole row copied to shared memory; the 512-thread build only). */    \
  bool staged_fits(int64_t row_len);                                                   \
  /* Enqueue one launch over every row of the group's problems (all of `form`, with */  \
  /* one tie capacity): grid = row_begin[n] * g CTAs in clusters of g. opts: some */    \
  /* problem has the values output or the sorted option (staged). */                    \
  cudaError_t launch_group(Form form, const GroupParams& gp, int g, bool opts,          \
                           bool keys_in_filter, int staged, cudaStream_t stream);       \
  /* The sort pass of the sorted output: p.staged (filled by a launch with p) is */     \
  /* ordered per row and written to p.out and p.values; one CTA per row. */             \
  cudaError_t sort_rows(Form form, const Params& p, cudaStream_t stream);                \
  /* Enqueue the chip-wide split (p.split_*: set; no values or sorted output): */        \
  /* batch * split_s filter CTAs, then one select CTA per row. */                       \
  cudaError_t launch_split(Form form, const Params& p, cudaStream_t stream);             \
  /* Clusters of g CTAs (at the largest tie capacity) the device holds at once. */       \
  cudaError_t max_active_clusters(int g, int* n);                                       \
  /* The count of failed internal consistency checks on the current device (a */       \
  /* synchronous read), and its reset. */                                               \
  cudaError_t guard_hits(unsigned int* hits);                                           \
  cudaError_t reset_guard_hits();

// The same calls for one form, each in an object of its own (the calls above
// dispatch to these).
#define TOPK_FORM_INTERFACE                                                             \
  cudaError_t prepare_device();                                                         \
  cudaError_t launch(const Params& p, int g, bool keys_in_filter, int staged,           \
                     cudaStream_t stream);                                              \
  cudaError_t launch_group(const GroupParams& gp, int g, bool opts, bool keys_in_filter, \
                           int staged, cudaStream_t stream);                            \
  cudaError_t sort_rows(const Params& p, cudaStream_t stream);                          \
  cudaError_t launch_split(const Params& p, cudaStream_t stream);                       \
  cudaError_t max_active_clusters(int g, int* n);                                       \
  cudaError_t guard_hits(unsigned int* hits);                                           \
  cudaError_t reset_guard_hits();

namespace cta512 {
TOPK_CTA_INTERFACE
namespace raw { TOPK_FORM_INTERFACE }
namespace paged { TOPK_FORM_INTERFACE }
namespace ragged { TOPK_FORM_INTERFACE }
namespace window { TOPK_FORM_INTERFACE }
}
namespace cta256 {
TOPK_CTA_INTERFACE
namespace raw { TOPK_FORM_INTERFACE }
namespace paged { TOPK_FORM_INTERFACE }
namespace ragged { TOPK_FORM_INTERFACE }
namespace window { TOPK_FORM_INTERFACE }
}
#undef TOPK_CTA_INTERFACE
#undef TOPK_FORM_INTERFACE

}  // namespace topk_gb300
