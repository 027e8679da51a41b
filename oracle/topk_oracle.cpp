// CPU oracle for the exact per-row top-k transform of a sparse-attention indexer.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product library loads, links or calls
// this file. Only the tests, the smoke check and the benchmark's CPU-baseline leg
// use it. It shares no code, header, table or helper with the CUDA library: it is
// the plain definition of the operation, written out, so that a reader can check
// it against the source pages by eye.
//
// Sources: the prhub.com.cn summary pages of two sglang pull requests,
//   [36004] sglang PR #36004 (ROCm: DSv4 top-k with 1024-thread blocks, first unit test)
//   [37591] sglang PR #37591 (ROCm: exact DSA-indexer top-k, the "coop" kernel)
//
// What one row b computes:
//   1. L = clamp(seq_len[b], 0, row_stride) for the raw and paged forms; for the
//      ragged form L = max(seq_len[b], 0) and the row is scores[row_starts[b] ...].
//      (The pages do not say what happens outside [0, row_stride]; clamping is the
//      plainest reading.)
//   2. Every position j < L gets the order-preserving key of its fp32 bit pattern:
//      negative values have all bits inverted, the rest get the sign bit set, so
//      that an unsigned compare of keys is the float order ([37591], section
//      "关键源码片段" (code excerpts), order_key32).
//   3. The pairs (key, j) are sorted by key, largest first, with a STABLE sort, so
//      pairs with equal keys stay in position order: at the threshold the smaller
//      position wins. The pages do not fix the tie rule ([36004]'s unit test
//      compares against torch.topk, whose tie choice is unspecified); smaller
//      position wins is the reading adopted, and it makes the selected set unique.
//      The selection is exact: no element is ever dropped ([37591], section
//      "执行摘要" (summary) and "实现拆解" (implementation breakdown) item 1).
//   4. The first m = min(k, L) positions are emitted, each mapped:
//        raw:    j
//        paged:  page_table[b][j / page_size] * page_size + j % page_size
//                (with an identity table this is j again, which is what the unit
//                test on [36004], section "关键源码片段", relies on)
//        ragged: row_starts[b] + j   (the position inside the packed buffer;
//                [37591] "关键源码片段", CoopParams, names row_starts as the
//                row offsets of the ragged API but not the emitted value)
//        window: lo + j, the column of the selected element in its row
//   The window form ([37591] "实现拆解" item 3: the tests cover variable
//   windows) selects among one window [lo, hi) of each row of a strided matrix:
//   lo = starts[b] and hi = seq_lens[b], both clamped to [0, row_stride], and
//   L = max(hi - lo, 0). With lo = 0 it is the raw form. (The pages name
//   variable windows without defining them; a per-row [start, end) inside the
//   row, emitting row columns, is the reading adopted.)
//   5. Slots m .. k-1 get -1 ([36004] "关键源码片段": the test pre-fills the
//      output with -1, so short rows leave -1 behind).
//   The m positions are written in rank order: largest key first, equal keys by
//   smaller position first (the order of the stable sort). This is the order of the
//   optional sorted output; the plain output may hold the same set in any order.
//   Optionally, values[b][i] gets the fp32 score of the element in slot i (its bit
//   pattern unchanged) and -inf in the padding slots (the extra outputs of the
//   "runtime k generalisation" item of the next steps; the pages name returned
//   values without fixing the padding, -inf is the reading adopted).
//
// Build: g++ -O2 -std=c++17 -shared -fPIC -pthread topk_oracle.cpp

#include <sched.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// Step 2: the order-preserving key of an fp32 bit pattern.
uint32_t order_key(float x) {
  uint32_t bits;
  std::memcpy(&bits, &x, sizeof bits);
  if (bits & 0x80000000u) return ~bits;
  return bits | 0x80000000u;
}

struct Pair {
  uint32_t key;
  int32_t pos;
};

// Steps 2-3: positions of the m = min(k, L) largest keys, in (key desc, pos asc)
// order.
void select_row(const float* row, int64_t L, int64_t k, std::vector<int32_t>& chosen) {
  std::vector<Pair> pairs(static_cast<size_t>(L));
  for (int64_t j = 0; j < L; ++j) pairs[j] = Pair{order_key(row[j]), static_cast<int32_t>(j)};
  std::stable_sort(pairs.begin(), pairs.end(),
                   [](const Pair& a, const Pair& b) { return a.key > b.key; });
  const int64_t m = std::min(k, L);
  chosen.resize(static_cast<size_t>(m));
  for (int64_t i = 0; i < m; ++i) chosen[i] = pairs[i].pos;
}

enum Form { kRaw = 0, kPaged = 1, kRagged = 2, kWindow = 3 };

struct Job {
  Form form;
  const float* scores;
  int64_t row_stride;          // raw, paged
  const int32_t* row_starts;   // ragged: row offsets; window: window starts
  const int32_t* seq_lens;
  const int32_t* page_table;   // paged
  int64_t page_table_stride;   // paged
  int32_t page_size;           // paged
  int32_t k;
  int32_t* out;                // [batch, k]
  float* values;               // [batch, k] or null
};

void run_row(const Job& job, int64_t b, std::vector<int32_t>& chosen) {
  const int64_t s = job.seq_lens[b];
  int64_t L;
  const float* row;
  int64_t lo = 0;  // window: first column of the window
  if (job.form == kRagged) {
    L = std::max<int64_t>(s, 0);
    row = job.scores + job.row_starts[b];
  } else if (job.form == kWindow) {
    lo = std::clamp<int64_t>(job.row_starts[b], 0, job.row_stride);
    const int64_t hi = std::clamp<int64_t>(s, 0, job.row_stride);
    L = hi > lo ? hi - lo : 0;
    row = job.scores + b * job.row_stride + lo;
  } else {
    L = std::min<int64_t>(std::max<int64_t>(s, 0), job.row_stride);
    row = job.scores + b * job.row_stride;
  }
  select_row(row, L, job.k, chosen);
  int32_t* out = job.out + b * static_cast<int64_t>(job.k);
  const int64_t m = static_cast<int64_t>(chosen.size());
  for (int64_t i = 0; i < m; ++i) {
    const int32_t j = chosen[i];
    int32_t v = j;
    if (job.form == kPaged) {
      const int32_t* pt = job.page_table + b * job.page_table_stride;
      v = pt[j / job.page_size] * job.page_size + j % job.page_size;
    } else if (job.form == kRagged) {
      v = job.row_starts[b] + j;
    } else if (job.form == kWindow) {
      v = static_cast<int32_t>(lo + j);
    }
    out[i] = v;
  }
  for (int64_t i = m; i < job.k; ++i) out[i] = -1;
  if (job.values != nullptr) {
    float* v = job.values + b * static_cast<int64_t>(job.k);
    for (int64_t i = 0; i < m; ++i) v[i] = row[chosen[i]];
    for (int64_t i = m; i < job.k; ++i) v[i] = -INFINITY;
  }
}

int usable_cores() {
  cpu_set_t set;
  CPU_ZERO(&set);
  if (sched_getaffinity(0, sizeof set, &set) == 0) {
    const int n = CPU_COUNT(&set);
    if (n > 0) return n;
  }
  const unsigned n = std::thread::hardware_concurrency();
  return n > 0 ? static_cast<int>(n) : 1;
}

// Rows are independent; threads take interleaved rows.
int run(const Job& job, int32_t batch, int threads) {
  if (batch < 0 || job.k < 1 || job.scores == nullptr || job.seq_lens == nullptr ||
      job.out == nullptr)
    return 1;
  if (job.form != kRagged && job.row_stride < 1) return 1;
  if (job.form == kPaged && (job.page_table == nullptr || job.page_size < 1)) return 1;
  if ((job.form == kRagged || job.form == kWindow) && job.row_starts == nullptr) return 1;
  if (batch == 0) return 0;
  if (threads < 1) threads = usable_cores();
  threads = std::min<int>(threads, batch);
  if (threads == 1) {
    std::vector<int32_t> chosen;
    for (int64_t b = 0; b < batch; ++b) run_row(job, b, chosen);
    return 0;
  }
  std::vector<std::thread> pool;
  pool.reserve(threads);
  for (int t = 0; t < threads; ++t) {
    pool.emplace_back([&job, batch, threads, t]() {
      std::vector<int32_t> chosen;
      for (int64_t b = t; b < batch; b += threads) run_row(job, b, chosen);
    });
  }
  for (auto& th : pool) th.join();
  return 0;
}

}  // namespace

extern "C" {

// The key of step 2, exposed so that tests can pin it on its own.
uint32_t oracle_order_key(float x) { return order_key(x); }

// Number of host cores this process may run on (sched_getaffinity).
int oracle_usable_cores(void) { return usable_cores(); }

// scores [batch, row_stride] fp32, seq_lens [batch] int32, out [batch, k] int32.
// threads < 1 means every usable core. Returns 0, or 1 on invalid arguments.
int oracle_topk_raw(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                    int32_t batch, int32_t k, int32_t* out, int threads) {
  Job job{kRaw, scores, row_stride, nullptr, seq_lens, nullptr, 0, 0, k, out, nullptr};
  return run(job, batch, threads);
}

// As oracle_topk_raw, plus page_table [batch, page_table_stride] int32.
int oracle_topk_paged(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                      const int32_t* page_table, int64_t page_table_stride,
                      int32_t page_size, int32_t batch, int32_t k, int32_t* out,
                      int threads) {
  Job job{kPaged, scores, row_stride, nullptr, seq_lens, page_table, page_table_stride,
          page_size, k, out, nullptr};
  return run(job, batch, threads);
}

// scores: the packed rows; row b is scores[row_starts[b] .. row_starts[b] + seq_lens[b]).
int oracle_topk_ragged(const float* scores, const int32_t* row_starts,
                       const int32_t* seq_lens, int32_t batch, int32_t k, int32_t* out,
                       int threads) {
  Job job{kRagged, scores, 0, row_starts, seq_lens, nullptr, 0, 0, k, out, nullptr};
  return run(job, batch, threads);
}

// The window form: row b selects among scores[b, lo .. hi) with lo = starts[b]
// and hi = seq_lens[b] (both clamped to [0, row_stride]) and emits columns lo + j.
int oracle_topk_window(const float* scores, int64_t row_stride, const int32_t* starts,
                       const int32_t* seq_lens, int32_t batch, int32_t k, int32_t* out,
                       int threads) {
  Job job{kWindow, scores, row_stride, starts, seq_lens, nullptr, 0, 0, k, out, nullptr};
  return run(job, batch, threads);
}

// Any form (0 raw, 1 paged, 2 ragged, 3 window; the arguments a form does not use
// are ignored) with the optional values output (null: not written). Positions are
// in rank order.
int oracle_topk_values(int32_t form, const float* scores, int64_t row_stride,
                       const int32_t* row_starts, const int32_t* seq_lens,
                       const int32_t* page_table, int64_t page_table_stride, int32_t page_size,
                       int32_t batch, int32_t k, int32_t* out, float* values, int threads) {
  if (form < kRaw || form > kWindow) return 1;
  Job job{static_cast<Form>(form), scores, row_stride, row_starts, seq_lens, page_table,
          page_table_stride, page_size, k, out, values};
  return run(job, batch, threads);
}

}  // extern "C"
