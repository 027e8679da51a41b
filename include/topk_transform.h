/*
 * topk_transform.h - exact per-row top-k transform of sparse-attention indexer
 * scores, for NVIDIA GB300 (sm_103a).
 *
 * What the operation computes (per row b of a batch):
 *   L = clamp(seq_lens[b], 0, row_stride)   (raw, paged)
 *     = max(seq_lens[b], 0)                 (ragged)
 *     = max(hi - lo, 0)                     (window: lo = clamp(starts[b], 0, row_stride),
 *                                            hi = clamp(seq_lens[b], 0, row_stride))
 *   Select the m = min(k, L) positions j < L whose fp32 scores are largest,
 *   exactly: scores are ranked by the order-preserving 32-bit key of their bit
 *   pattern (negative values bit-inverted, the others with the sign bit set),
 *   which is float order with -0.0 just below +0.0 (sglang PR #37591 summary
 *   page, section "关键源码片段" (code excerpts), order_key32). Among equal keys at
 *   the threshold the smaller position wins, so the selected set is unique. No
 *   element is ever dropped, whatever the distribution (PR #37591 page, sections
 *   "执行摘要" (summary) and "实现拆解" (implementation breakdown) item 1).
 *   Each selected j is written mapped:
 *     raw     j
 *     paged   page_table[b * page_table_stride + j / page_size] * page_size + j % page_size
 *     ragged  row_starts[b] + j
 *     window  lo + j (the column in row b; position j of the window is column lo + j)
 *   and the slots m .. k-1 of the row are written with -1 (sglang PR #36004
 *   summary page, section "关键源码片段": test_deepseek_v4_topk_transform
 *   pre-fills the output with -1 and uses an identity page table, under which the
 *   paged slot equals the token position). The first three entry points mirror
 *   the three API forms named on the PR #37591 page, "实现拆解" item 2. The window
 *   form is the "variable windows" its tests cover (same page, item 3), read as
 *   one [start, end) window per row of a strided matrix (prefill-shaped batches:
 *   query b attends to keys start .. end-1).
 *
 * Output order: the order of the m positions inside out[b, 0:k) is unspecified;
 * compare rows as sets. The SET is deterministic.
 *
 * Memory and ownership: every pointer argument is device memory owned by the
 * caller (for example torch tensors passed as data_ptr()). The library never
 * allocates, frees or synchronises; each call enqueues one kernel on `stream`
 * (NULL = the legacy default stream; two kernels for a call that takes the
 * chip-wide split, see topk_workspace_bytes) and returns. All inputs must stay
 * valid and unmodified until the call's kernels have finished. `out` is fully written, including
 * the -1 padding, so it need not be pre-filled. The first call on a device sets
 * kernel attributes on that device; make it before capturing a CUDA graph.
 *
 * Stream order: every launch allows programmatic dependent launch, so it may be
 * scheduled while the previous kernel of the stream is still running, and it lets
 * the next kernel of the stream do the same. Before it reads or writes any buffer
 * it waits until the previous kernel has completed and its memory is visible
 * (griddepcontrol.wait), so the usual stream ordering of data holds. A kernel
 * that follows in the stream and was itself launched with programmatic
 * serialization must wait the same way before it reads `out`.
 *
 * Layouts (all row-major, int32 unless stated):
 *   scores      fp32, 4-byte aligned. raw/paged: row b starts at
 *               scores + b * row_stride (elements); ragged: row b starts at
 *               scores + row_starts[b]; window: row b's window starts at
 *               scores + b * row_stride + lo. Any alignment of a row start is
 *               accepted.
 *   seq_lens    [batch]
 *   page_table  [batch, page_table_stride]; entries are trusted. Each row must
 *               hold the entries of pages 0 .. ceil(L/page_size)-1, so
 *               page_table_stride >= ceil(L/page_size) for every row. A row that
 *               needs more pages than page_table_stride never reads past its own
 *               entries: the kernel counts it once in topk_guard_hits and writes
 *               -1 for each selected position whose page is missing.
 *   row_starts  [batch], element offsets into `scores`; row_starts[b] + j must
 *               fit in int32.
 *   starts      [batch] (window form), any int32 value: it is clamped as above.
 *   out         [batch, k]
 *
 * Errors: host-checkable problems return a status and launch nothing. Values
 * that live in device memory (seq_lens, page_table, row_starts, starts) are not
 * validated: seq_lens and starts are clamped as above, the others are trusted. A launch
 * failure returns TOPK_ERR_CUDA; topk_last_cuda_error() gives the cudaError_t.
 */
#ifndef TOPK_TRANSFORM_H_
#define TOPK_TRANSFORM_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TOPK_OK = 0,
  TOPK_ERR_INVALID_ARGUMENT = 1, /* null pointer, negative batch, bad stride or page size */
  TOPK_ERR_UNSUPPORTED_K = 2,    /* k outside [1, TOPK_MAX_K] */
  TOPK_ERR_WORKSPACE_TOO_SMALL = 3,
  TOPK_ERR_CUDA = 4              /* a CUDA runtime call or the launch failed */
} topk_status_t;

/* Largest supported k. The pages' kernels fix k at 1024 (the legacy
 * deepseek_v4_topk_transform, PR #36004 page, "关键源码片段", kMaxTopK) and at
 * 2048 (the exact kernel, PR #37591 page, "实现拆解" item 2, kTopK). Any k in
 * [1, TOPK_MAX_K] is accepted. */
#define TOPK_MAX_K 2048

/* Device workspace (bytes) that lets a single-form call of these sizes on the
 * current device take the chip-wide split: small batches of long rows (by default
 * 4 rows up to one row per 16 SMs, rows of at least 65536 elements; see
 * topk_set_chip_split) are each split over many CTAs anywhere on the chip, which
 * store their candidates in the workspace for a second kernel that selects per
 * row. This restates the row split of the exact kernel on the PR #37591 page
 * ("关键源码片段", row_split and the per-split histograms merged in global memory)
 * with one sampled threshold instead of merged histograms. 0 when the split does
 * not apply (then every per-row state stays in shared memory). The size depends on
 * the SM count and the tie capacity (topk_set_tie_capacity) at the time of the
 * query. A call given a workspace of at least this size (device memory, 256-byte
 * aligned, owned by the caller; not read before the call writes it, so it needs no
 * initialisation; calls that may overlap in time need separate workspaces) takes
 * the split; a call given less (or NULL) runs the same rows on one cluster of CTAs
 * per row. The result is the same either way. Returns 0 when no CUDA device is
 * usable. */
size_t topk_workspace_bytes(int32_t batch, int64_t max_row_len, int32_t k);

/* Raw form. scores [batch, row_stride] fp32 (row_stride >= 1 elements),
 * seq_lens [batch], out [batch, k]. `workspace` may be NULL when
 * `workspace_bytes` is 0. Returns a topk_status_t. */
int topk_transform_raw(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                       int32_t batch, int32_t k, int32_t* out,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Paged form: as raw, each position mapped through the row's page table
 * (page_size >= 1; page_table_stride >= 1, and at least ceil(L/page_size) for
 * every row, see page_table above). */
int topk_transform_paged(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                         const int32_t* page_table, int64_t page_table_stride,
                         int32_t page_size, int32_t batch, int32_t k, int32_t* out,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Ragged form: row b is scores[row_starts[b] .. row_starts[b] + seq_lens[b]) of a
 * packed buffer; each selected position is written as row_starts[b] + j.
 * max_row_len_hint (>= 0) is an upper bound of the row lengths, used only to
 * choose how many CTAs share a row; 0 means "unknown, assume long". */
int topk_transform_ragged(const float* scores, const int32_t* row_starts,
                          const int32_t* seq_lens, int64_t max_row_len_hint, int32_t batch,
                          int32_t k, int32_t* out, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/* Window form: row b of scores [batch, row_stride] selects among its columns
 * [starts[b], seq_lens[b]) (both clamped to [0, row_stride]; an empty window if
 * the end is not after the start) and writes the selected columns. With every
 * start 0 it is the raw form. row_stride >= 1; starts, seq_lens [batch].
 * max_row_len_hint (>= 0) is an upper bound of the window lengths, used only to
 * choose the kernel configuration; 0 means row_stride. */
int topk_transform_window(const float* scores, int64_t row_stride, const int32_t* starts,
                          const int32_t* seq_lens, int64_t max_row_len_hint, int32_t batch,
                          int32_t k, int32_t* out, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/* ------------------------------------------------------------------ grouped calls
 *
 * Several independent transforms in as few launches as possible: one launch per
 * form present, in which the rows of every problem of that form run
 * concurrently (the per-decode-step batching of the PR #37591 page's serving
 * context: the many small top-k calls of one step no longer run one after the
 * other). The result of each problem is exactly what the entry point of its form
 * writes. */
typedef enum {
  TOPK_FORM_RAW = 0,
  TOPK_FORM_PAGED = 1,
  TOPK_FORM_RAGGED = 2,
  TOPK_FORM_WINDOW = 3
} topk_form_t;

/* Options of a problem (topk_problem_t.flags). TOPK_FLAG_SORTED: the m selected
 * slots of each row in rank order (largest score first, equal scores by smaller
 * position first; the -1 padding after them). Needs a device workspace of
 * topk_problem_workspace_bytes bytes; the ordering runs as a second kernel per
 * sorted problem. (The "extra outputs" of the next steps after the pages' design:
 * the pages fix the set, not an order.) */
#define TOPK_FLAG_SORTED 1u

/* One problem: the arguments of its form's entry point. Fields a form does not
 * use are ignored (row_stride: raw, paged, window; page_table, page_table_stride,
 * page_size: paged; row_starts: ragged row offsets or window starts;
 * max_row_len_hint: ragged and window, as for their entry points).
 * values (optional, [batch, k] fp32, device): each slot's score (its fp32 bits
 * unchanged), -inf in the padding slots; NULL: not written. */
typedef struct {
  int32_t form;               /* topk_form_t */
  int32_t batch;              /* rows, >= 0 (0: nothing to do) */
  int32_t k;                  /* [1, TOPK_MAX_K] */
  int32_t page_size;
  int64_t row_stride;
  int64_t page_table_stride;
  int64_t max_row_len_hint;
  const float* scores;
  const int32_t* seq_lens;
  const int32_t* row_starts;
  const int32_t* page_table;
  int32_t* out;               /* [batch, k] */
  float* values;              /* [batch, k] or NULL */
  uint32_t flags;             /* TOPK_FLAG_* */
  uint32_t reserved;          /* 0 */
} topk_problem_t;

/* Most problems one grouped call takes. */
#define TOPK_MAX_GROUP 32

/* sizeof(topk_problem_t) as this library was built (for bindings to check their
 * copy of the layout). */
size_t topk_problem_bytes(void);

/* Device workspace bytes a grouped call with these problems needs: for each
 * problem with TOPK_FLAG_SORTED, 8 bytes per output slot (batch * k), rounded up
 * to 256 bytes; 0 when no problem asks for sorted output. problems: host array of
 * n_problems (invalid arguments give 0). */
size_t topk_problem_workspace_bytes(const topk_problem_t* problems, int32_t n_problems);

/* problems: HOST array of n_problems (0 .. TOPK_MAX_GROUP) descriptors, read
 * during the call only; the pointers inside are device memory, as for the single
 * entry points. Every problem is checked first, in order: on the first problem
 * that fails its check nothing is launched and its status is returned; a
 * workspace smaller than topk_problem_workspace_bytes returns
 * TOPK_ERR_WORKSPACE_TOO_SMALL, also before any launch (workspace: device memory,
 * 256-byte aligned, owned by the caller, used until the launches finish).
 * Problems of one form share a launch; distinct output buffers are required. */
int topk_transform_grouped(const topk_problem_t* problems, int32_t n_problems,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* As topk_transform_grouped, with no workspace argument, for callers that cannot
 * allocate device memory: a plug-in inside a host runtime that hands it only fixed
 * input and output buffers and no allocator; a serving engine whose caching
 * allocator has reserved the device's memory up front, so a cudaMalloc of its own
 * would fail or stall every stream on an implicit synchronisation in the middle of
 * a decode step.
 *
 * Sorted problems stage their (key, position) pairs in a scratch array the library
 * keeps in device memory instead: a static __device__ array of
 * TOPK_STATIC_WORKSPACE_BYTES (16 MiB), part of the loaded module, so every device
 * that loads the library holds it until the process exits. The call itself
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 *
 * Limit: problems needing more than TOPK_STATIC_WORKSPACE_BYTES of staging
 * (topk_problem_workspace_bytes: 8 bytes per output slot of each sorted problem,
 * so more than 1024 rows at k = 2048) get TOPK_ERR_WORKSPACE_TOO_SMALL before any
 * launch.
 * Problems without TOPK_FLAG_SORTED never touch the array.
 *
 * Set-up: the first call on a device that has a sorted problem looks up the
 * array's device address (cudaGetSymbolAddress, once per device, on the current
 * device); make that first call before any stream capture.
 *
 * Sharing: every call on a device uses the same array, which keeps the last call's
 * contents. Nothing in it needs to start at zero (the selection kernel writes every
 * slot the sort pass reads, padding included). Calls whose launches overlap on the
 * GPU race on the array and give wrong results: issue them on one stream, or order
 * their streams. */
#define TOPK_STATIC_WORKSPACE_BYTES (16u << 20)
int topk_transform_grouped_static(const topk_problem_t* problems, int32_t n_problems,
                                  cudaStream_t stream);

/* A static English description of a status code. */
const char* topk_status_string(int status);

/* The cudaError_t of the last TOPK_ERR_CUDA returned on this host thread. */
int topk_last_cuda_error(void);

/* Diagnostics. Every write the kernels make into a row's output, the tie list or
 * the tie buffer is guarded by a check that consistent inputs never fail (it can
 * fail only if inputs change while a kernel runs, or through a bug); a failed check
 * skips the write and is counted on the device instead of trapping.
 * topk_guard_hits(&n) reads the count on the current device (synchronously: it
 * waits for the device's pending work); topk_reset_guard_hits() sets it to 0. */
int topk_guard_hits(uint64_t* hits);
int topk_reset_guard_hits(void);

/* Tuning and test controls (process-wide; each returns the previous value).
 *
 * topk_set_row_split(g): number of CTAs (a thread-block cluster) that share one
 * row: 1, 2, 4, 8 or 16 (other values round down to a power of two); any value
 * < 1 restores the built-in choice, which depends on batch, row length and SM
 * count (the row-split heuristic of the PR #37591 page, "关键源码片段",
 * row_split, restated for a cluster). The environment variable TOPK_ROW_SPLIT
 * sets the initial value.
 *
 * topk_set_tie_capacity(cap): entries of the shared candidate/tie buffer,
 * clamped to [0, TOPK_TIE_CAPACITY_MAX]. Smaller values send more rows through
 * the exact tier's extra radix rounds and its position-ordered rescan (used by
 * tests); the result never changes.
 *
 * topk_set_fast_tier(enable): 1 (default) first tries the one-pass filter whose
 * threshold comes from a sample of the row and is verified afterwards; 0 always
 * runs the exact histogram tier. The result is the same either way.
 *
 * topk_set_staged_tier(mode): where rows owned by one CTA whose length is known
 * to be at most 32768 elements (row_stride for raw and paged, the length hints for
 * ragged and window) run on the staged tier, which copies the row into shared
 * memory from kernel start: 1 (default) automatically (launches of 64 rows up to
 * one row per SM, rows that may hold 16384 elements or more); 2 always, with the
 * whole row staged (one CTA per SM); 3 always, with half a row staged (two CTAs per
 * SM); 0 never (the streaming fast tier). Other values mean 1. The result is the
 * same either way.
 *
 * topk_set_chip_split(mode): when single-form calls with enough workspace take the
 * chip-wide split (topk_workspace_bytes): 1 (default) automatically; 2 for every
 * batch and row length (used by tests); 0 never. Other values mean 1. The result is
 * the same either way.
 *
 * topk_set_cta_threads(t): which build of the kernels runs: 512-thread CTAs (two
 * per SM) or 256-thread CTAs (four per SM, at most 3072 tie-buffer entries); any
 * other value restores the built-in choice, which takes the 256-thread build for
 * launches of more rows than two CTAs per SM hold, with one CTA per row, k <= 1024,
 * and rows of at most 8192 elements (by row_stride, or the ragged and window hints)
 * or at least 16 rows per SM.
 * The result is the same either way. */
#define TOPK_TIE_CAPACITY_MAX 4096
int topk_set_row_split(int g);
int topk_set_tie_capacity(int cap);
int topk_set_fast_tier(int enable);
int topk_set_cta_threads(int threads);
int topk_set_staged_tier(int mode);
int topk_set_chip_split(int mode);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* TOPK_TRANSFORM_H_ */
