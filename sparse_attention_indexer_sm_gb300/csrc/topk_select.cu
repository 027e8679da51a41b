// Exact per-row top-k selection of fp32 indexer scores on GB300 (sm_103a).
//
// One thread-block cluster of G CTAs (G = 1, 2, 4, 8 or 16) owns one row; each
// CTA owns a contiguous slice of it. The method is the exact "coop" top-k of the
// sglang PR #37591 summary page (section "实现拆解" (implementation breakdown)
// item 1 and the coop_topk_kernel excerpt under "关键源码片段"): an
// order-preserving 32-bit key, radix histograms over the high key bits to find
// the threshold bucket, a scatter of winners and threshold-bucket ties, an exact
// refinement of the ties on the full key, and a rescan when the tie buffer
// overflows. On this machine it runs in two tiers:
//
// Fast tier (one pass over the row, normally the only one):
//  F1. sample    each CTA loads a sample of its slice (one 16-byte quad per thread,
//                in runs of 512 bytes) before anything else. Two sample ranks are
//                wanted: r_s, four standard deviations below the expected sample rank
//                of the row's k-th key, and r_lo three above it. A 1024-bin histogram
//                of the top 10 key bits (summed over the cluster through distributed
//                shared memory) finds the coarse bins of both; a second 1024-bin
//                histogram spanning just those coarse bins resolves them: lambda is the
//                lower edge of r_s's fine bin, lambda_hi the upper edge of r_lo's. Every
//                thread takes part in each threshold search. Rows that fit the candidate
//                buffer skip the sample (lambda = 0); cluster rows whose sample predicts
//                far more candidates than the buffer holds go to the exact tier at once.
//  F2. filter    one streaming pass with 128-bit loads compares every raw fp32 bit
//                pattern with lambda (a single integer compare: for lambda in the
//                non-negative range a signed compare, otherwise an unsigned one,
//                both equal to "key >= lambda"). Candidates go to CTA 0's shared
//                buffer as (key, position) and are counted in a 2048-bin candidate
//                histogram whose bins of width 2^s2 start at lambda (s2 chosen so that
//                fewer than 1024 bins span [lambda, lambda_hi]; the last bin takes
//                every larger key; rows that skip the sample use the top 11 key bits).
//                A row owned by one CTA keeps only positions in the pass (so the
//                loads of several iterations stay in flight) and reads the candidates'
//                values back from L2 afterwards; the CTAs of a cluster write keys and
//                their own histograms directly, summed into CTA 0's afterwards.
//  F3. select    if the cluster found between k and capacity candidates, every
//                element of the exact top-k is among them (they hold k elements with
//                key >= lambda, so the k-th key is >= lambda). CTA 0 finds the
//                threshold bin of the candidate histogram, writes the candidates above
//                it (through output slots in shared memory, written out at the end),
//                and orders the candidates of that bin on the 64-bit composite
//                (key, ~position), so equal keys go to the smaller position: by a rank
//                count spread over the CTA up to 256 of them, by radix rounds beyond.
//                Otherwise the exact tier runs.
//
// Exact tier (any distribution; the page's design, re-planned):
//  E1. rounds    4096-bin shared histograms of the top 12 key bits over the slice
//                (merged over the cluster), then of the next 12 and 8 bits inside
//                the threshold bin while that bin holds more elements than the tie
//                buffer (the page's round0/round1 coarse histograms).
//  E2. scatter   elements above the threshold bin go straight to the output;
//                elements in it go to CTA 0's tie buffer (the page's scatter pass).
//  E3. refine    as F3, on the ties (the page's radix sort of the ties on the full
//                fp32 key).
//  E4. rescan    when more elements than the buffer holds equal the exact 32-bit
//                threshold key, every CTA re-reads its slice in position order and
//                takes its quota of equal elements by a block-wide prefix count (the
//                page's overflow rescan): nothing is ever dropped.
//
// Two more paths share these steps (each described at its code): the staged tier
// (single-CTA rows of 16384 to 32768 elements, 64 rows up to one per SM: the row is
// copied into shared memory from kernel start and lambda comes from one sample round
// in value space) and the chip-wide split (batches of 4 rows up to one per 16 SMs of
// rows of 65536 elements or more: many CTAs per row filter into a caller workspace,
// one cluster per row then selects).
//
// No step waits on another CTA except through the hardware cluster barrier or the
// grid dependency between launches: no spin loop. One launch per call (two for the
// chip-wide split, whose workspace the caller provides).

#include <cstdint>

#include "topk_select.cuh"

// This file is compiled for two CTA sizes: TOPK_CTA_THREADS = 512 (namespace cta512:
// two CTAs per SM, every launch that fits one wave) and 256 (cta256: four CTAs per
// SM, for launches of more rows than that, so that each SM overlaps four rows'
// latency chains instead of two). For each size it is compiled once per form
// (TOPK_FORM = 0 .. 3: that form's kernels and launches) and once without
// TOPK_FORM (the dispatch by form), so that the objects build in parallel.
#ifndef TOPK_CTA_THREADS
#define TOPK_CTA_THREADS 512
#endif
#if TOPK_CTA_THREADS == 512
#define TOPK_CTA_NS cta512
#elif TOPK_CTA_THREADS == 256
#define TOPK_CTA_NS cta256
#else
#error "TOPK_CTA_THREADS must be 512 or 256"
#endif

namespace topk_gb300 {
namespace TOPK_CTA_NS {
namespace {

constexpr int kThreads = TOPK_CTA_THREADS;  // threads per CTA
constexpr int kCtasPerSm = 1024 / kThreads;  // at 64 registers per thread
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;            // 128-bit loads in flight per thread per step (exact tier)
constexpr int kFilterUnroll = 8;      // 128-bit loads in flight per thread in the filter
constexpr int kMaskIters = 2;         // filter iterations whose masks are decoded together
constexpr int kRowRoundBits = 12;     // histogram width of the rounds over the row
constexpr int kBufRoundBits = 12;     // histogram width of the rounds over a buffer
constexpr int kSampleQuads = 512 / kThreads;  // sampled 16-byte quads per thread (2048 keys per CTA)
constexpr uint32_t kPrefetchBytes = 16384;  // one bulk L2 prefetch
// page-table entries staged in shared memory (rows with more pages read the table
// from global memory); the 256-thread build keeps its shared memory within a
// quarter of the SM's
constexpr int kPtCap = kThreads == 512 ? 4096 : 1024;
constexpr int kRankDirect = 256;      // threshold bins this small are ordered by rank count
constexpr unsigned kFull = 0xFFFFFFFFu;

// Histograms are stored padded, one spare word after every 32 bins, so that the
// threshold scan (each thread reads a run of consecutive bins) is free of shared
// memory bank conflicts.
__host__ __device__ constexpr int hist_index(int b) { return b + (b >> 5); }
constexpr int kHistWords = hist_index(kMaxBins);
// (key, position) entries of the list region (the candidates of the threshold bin;
// a bin holding more is refined in the candidate buffer instead). The 256-thread
// build keeps a short list to give its candidate buffer room.
constexpr int kListCap = kThreads == 512 ? kHistWords / 2 : 512;
constexpr int kListWords = 2 * kListCap;

// The fast tier's histograms have 1024 bins, small enough for one warp to find a
// threshold in (no block-wide scan). Each has its own region of `hist` (and, in
// CTA 0 of a cluster, of `mhist`), all cleared once at the start: the sample's
// coarse and fine rounds and the candidate histogram.
constexpr int kFastBits = 10;
constexpr int kFastBins = 1 << kFastBits;
constexpr int kFastWords = hist_index(kFastBins);
constexpr int kH1 = 0;                // sample, coarse round
constexpr int kH2 = kFastWords;       // sample, fine round
constexpr int kHC = 2 * kFastWords;   // candidates
// The candidate histogram has 2048 bins (its region runs to the end of `hist`): the
// finer its bins, the fewer candidates share the threshold bin.
constexpr int kCandBits = 11;
constexpr int kCandBins = 1 << kCandBits;
constexpr int kCandWords = hist_index(kCandBins);
static_assert(kHC + kCandWords <= kHistWords, "fast-tier histograms must fit the histogram region");
static_assert(kHC >= kMaxK, "a row's output slots fit below the candidate histogram");

struct Ctl {
  uint32_t scan[kWarps];              // per-warp partials of block scans
  uint32_t sel_t, sel_above, sel_count;  // threshold bin of the current round
  uint32_t win_cnt, tie_cnt, out_cnt;    // slot counters
  uint32_t cand_cnt;                  // candidates found by the filter (CTA 0)
  uint32_t n_cand;                    // cand_cnt of CTA 0, broadcast
  uint32_t sel2_t, sel2_above, sel2_count;  // second threshold of find_threshold2
  uint32_t ns;                        // valid sample size (CTA 0)
  uint32_t win_lo, win_shift, win_above;  // fine sample window (broadcast)
  uint32_t lambda, lambda_shift;      // filter threshold key and bin width, broadcast
  uint32_t skip_fast;                 // the sample predicts an overflowing filter, broadcast
  uint32_t ex_shift;                  // with skip_fast: the exact tier's first window, broadcast
  uint32_t sup[32];                   // super-bin sums of the histogram being searched
  uint32_t xa[kMaxCluster];           // per-CTA winners (cluster exchange)
  uint32_t xt[kMaxCluster];           // per-CTA threshold-bin elements
  // staged tier
  uint32_t wmax[kWarps], wmin[kWarps], wcnt[kWarps];  // per-warp sample extremes and sizes
};

struct Sel {
  uint32_t t, above, count;
};

// ------------------------------------------------------------------ primitives

__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  // negative: all bits inverted; otherwise: sign bit set
  const uint32_t flip = static_cast<uint32_t>(static_cast<int32_t>(bits) >> 31) | 0x80000000u;
  return bits ^ flip;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t r;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
  return r;
}

// Internal consistency checks that consistent inputs never fail (a failure means
// the scores changed while a kernel ran, or a bug) skip the access they guard and
// are counted here, instead of trapping, so that the host can read the count
// (guard_hits) and the context stays usable.
__device__ unsigned int g_guard_hits;
__device__ __forceinline__ void guard_hit() { atomicAdd(&g_guard_hits, 1u); }

// Programmatic dependent launch: every launch lets the next kernel of the stream be
// scheduled before it ends. allow_next_grid signals that (early, from every
// thread); wait_prior_grids returns once the previous kernel of the stream has
// completed and its memory is visible. Each kernel calls it before it reads or
// writes any buffer, so only shared-memory set-up overlaps the previous kernel.
__device__ __forceinline__ void allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_prior_grids() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Full cluster barrier; release/acquire orders shared-memory traffic across CTAs.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void dsmem_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t dsmem_fetch_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" :: "r"(addr), "r"(a), "r"(b)
               : "memory");
}

// 128-bit read-only load that does not allocate in L1.
// 128-bit read-only load that keeps its line in L1 (so that a candidate's value can
// be read again from L1 right after).
__device__ __forceinline__ uint4 ld_keep(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::evict_last.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Asynchronous 4-byte copy global -> shared (no register holds the value).
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_addr(smem_dst)), "l"(gsrc)
               : "memory");
}

// Waits until this thread's asynchronous copies have landed in shared memory.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Ask the memory system to bring [p, p + bytes) into L2 (16-byte aligned, bytes a
// multiple of 16). Nothing waits for it; later loads simply hit L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// Inclusive warp prefix sum of n; *total gets the warp sum. All 32 lanes.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t n, uint32_t* total) {
  const int lane = threadIdx.x & 31;
  uint32_t x = n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
  *total = __shfl_sync(kFull, x, 31);
  return x;
}

// Reserve n consecutive slots of a shared counter for this lane, one atomic per
// warp. `remote` selects a distributed-shared-memory counter (cluster address).
__device__ __forceinline__ uint32_t warp_reserve(uint32_t* counter, uint32_t counter_remote,
                                                 bool remote, uint32_t n) {
  uint32_t total;
  const uint32_t x = warp_incl_scan(n, &total);
  uint32_t base = 0;
  if (total != 0) {
    if ((threadIdx.x & 31) == 31)
      base = remote ? dsmem_fetch_add(counter_remote, total) : atomicAdd(counter, total);
    base = __shfl_sync(kFull, base, 31);
  }
  return base + x - n;
}

// One slot of a local shared counter for each lane whose `pred` holds. All lanes.
__device__ __forceinline__ uint32_t warp_reserve_bit(uint32_t* counter, bool pred) {
  const uint32_t b = __ballot_sync(kFull, pred);
  uint32_t base = 0;
  if (b != 0) {
    const int leader = __ffs(b) - 1;
    if ((threadIdx.x & 31) == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(b)));
    base = __shfl_sync(kFull, base, leader);
  }
  return base + static_cast<uint32_t>(__popc(b & lanemask_lt()));
}

// Sum over the block; every thread gets the total.
__device__ __forceinline__ uint32_t block_sum(uint32_t v, Ctl& ctl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  if (lane == 0) ctl.scan[warp] = v;
  __syncthreads();
  uint32_t total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) total += ctl.scan[w];
  __syncthreads();
  return total;
}

// Exclusive prefix sum in thread order; *total gets the block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, Ctl& ctl, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t wsum;
  const uint32_t x = warp_incl_scan(v, &wsum);
  if (lane == 31) ctl.scan[warp] = x;
  __syncthreads();
  uint32_t below = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t s = ctl.scan[w];
    below += w < warp ? s : 0u;
    all += s;
  }
  __syncthreads();
  *total = all;
  return below + x - v;
}

// Threshold bin of the (padded) histogram h of nbins bins: the bin t where the
// count from the top reaches `need` (need <= sum of h). Writes t, the count
// strictly above t and h[t] into ctl.sel_*; all threads see them on return.
__device__ __forceinline__ void find_threshold(const uint32_t* h, int nbins, uint32_t need,
                                               Ctl& ctl) {
  constexpr int kMaxPer = kMaxBins / kThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nbins >= kThreads ? nbins / kThreads : 1;
  const int b0 = tid * per;
  uint32_t c[kMaxPer];
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    c[i] = (i < per && b0 + i < nbins) ? h[hist_index(b0 + i)] : 0u;
    s += c[i];
  }
  // suffix scan: thread t gets the count held by threads > t (higher bins)
  uint32_t x = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_down_sync(kFull, x, off);
    if (lane + off < 32) x += y;
  }
  if (lane == 0) ctl.scan[warp] = x;
  __syncthreads();
  uint32_t higher = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) higher += w > warp ? ctl.scan[w] : 0u;
  const uint32_t excl = higher + x - s;
  if (s != 0 && excl < need && need <= excl + s) {
    uint32_t acc = excl;
    bool found = false;
#pragma unroll
    for (int i = kMaxPer - 1; i >= 0; --i) {
      if (!found && i < per && acc + c[i] >= need) {
        ctl.sel_t = static_cast<uint32_t>(b0 + i);
        ctl.sel_above = acc;
        ctl.sel_count = c[i];
        found = true;
      }
      acc += found ? 0u : c[i];
    }
  }
  __syncthreads();
}

// Every thread of the CTA: in the padded histogram h of kThreads * P bins, the bin
// where the count from the top reaches need1 (-> ctl.sel_*) and, if `two`, need2
// (-> ctl.sel2_*); a need outside [1, sum of h] finds nothing. Thread t holds bins
// [P t, P t + P): a suffix scan over the warp's lanes, one barrier for the warps'
// totals, and each thread checks its own bins. The results are visible after the
// caller's next barrier; ctl.scan is written. (A lone warp searching the whole
// histogram measured several times slower: its dependent shared loads, shuffles
// and branches do not overlap with any other warp's.)
template <int P>
__device__ __forceinline__ void block_find2(const uint32_t* h, uint32_t need1, uint32_t need2,
                                            bool two, Ctl& ctl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t c[P];
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < P; ++i) {
    c[i] = h[hist_index(tid * P + i)];
    s += c[i];
  }
  uint32_t x = s;  // count in the bins of lanes >= lane
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_down_sync(kFull, x, off);
    if (lane + off < 32) x += y;
  }
  if (lane == 0) ctl.scan[warp] = x;
  __syncthreads();
  // the count in higher warps' bins: lane w < kWarps reads warp w's total
  uint32_t a = __reduce_add_sync(kFull, lane < kWarps && lane > warp ? ctl.scan[lane] : 0u) + x - s;
  const uint32_t n2 = two ? need2 : 0u;
#pragma unroll
  for (int i = P - 1; i >= 0; --i) {
    const uint32_t b = static_cast<uint32_t>(tid * P + i);
    if (a < need1 && need1 <= a + c[i]) {
      ctl.sel_t = b;
      ctl.sel_above = a;
      ctl.sel_count = c[i];
    }
    if (a < n2 && n2 <= a + c[i]) {
      ctl.sel2_t = b;
      ctl.sel2_above = a;
      ctl.sel2_count = c[i];
    }
    a += c[i];
  }
}

// Cluster-wide threshold bin of the CTAs' histograms `hist` (complete and
// visible to the whole CTA on entry). With G > 1 the histograms are summed into
// CTA 0's `mhist` through distributed shared memory; CTA 0 finds the bin, sends
// it to every CTA and clears `mhist` for the next round.
__device__ __forceinline__ Sel threshold_of(const uint32_t* hist, uint32_t* mhist, int nbins,
                                            uint32_t need, int G, int rank, Ctl& ctl) {
  const int tid = threadIdx.x;
  if (G == 1) {
    find_threshold(hist, nbins, need, ctl);
    return Sel{ctl.sel_t, ctl.sel_above, ctl.sel_count};
  }
  const uint32_t m0 = map_rank(smem_addr(mhist), 0);
  for (int i = tid; i < hist_index(nbins); i += kThreads) {
    const uint32_t v = hist[i];
    if (v != 0) dsmem_add(m0 + 4u * static_cast<uint32_t>(i), v);
  }
  cluster_sync();
  if (rank == 0) {
    find_threshold(mhist, nbins, need, ctl);
    if (tid > 0 && tid < G) {
      dsmem_st(map_rank(smem_addr(&ctl.sel_t), tid), ctl.sel_t);
      dsmem_st(map_rank(smem_addr(&ctl.sel_above), tid), ctl.sel_above);
      dsmem_st(map_rank(smem_addr(&ctl.sel_count), tid), ctl.sel_count);
    }
    for (int i = tid; i < hist_index(nbins); i += kThreads) mhist[i] = 0;
  }
  cluster_sync();
  return Sel{ctl.sel_t, ctl.sel_above, ctl.sel_count};
}

// ------------------------------------------------------------------ row slices

// This CTA's part of a row: a 16-byte-aligned body of 4-element quads split
// evenly over the cluster, plus the unaligned head (CTA 0) and tail (last CTA).
struct Slice {
  const float* row;
  const uint4* vec;       // this CTA's first quad
  int32_t nq;             // this CTA's quads
  int32_t j0;             // row position of this CTA's first quad
  int32_t nvec;           // quads of the whole aligned body
  int32_t n_head;         // positions [0, n_head) belong to this CTA
  int32_t tail0, n_tail;  // positions [tail0, tail0 + n_tail) belong to this CTA
  int32_t lo, hi;         // the CTA's positions as one range [lo, hi)
};

// Quads [q0, q1) of CTA `rank` of G (a power of two) in an aligned body of nvec.
__device__ __forceinline__ void quad_range(int32_t nvec, int rank, int G, int32_t* q0,
                                           int32_t* q1) {
  const int lg = __ffs(G) - 1;
  *q0 = static_cast<int32_t>((static_cast<uint64_t>(nvec) * static_cast<uint32_t>(rank)) >> lg);
  *q1 = static_cast<int32_t>((static_cast<uint64_t>(nvec) * static_cast<uint32_t>(rank + 1)) >> lg);
}

__device__ __forceinline__ Slice make_slice(const float* row, int32_t L, int rank, int G) {
  Slice s;
  s.row = row;
  const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row) >> 2) & 3u;
  int32_t head = static_cast<int32_t>((4u - mis) & 3u);
  if (head > L) head = L;
  s.nvec = (L - head) >> 2;
  int32_t q0, q1;
  quad_range(s.nvec, rank, G, &q0, &q1);
  s.vec = reinterpret_cast<const uint4*>(row + head) + q0;
  s.nq = q1 - q0;
  s.j0 = head + 4 * q0;
  const int32_t tail0 = head + 4 * s.nvec;
  s.n_head = rank == 0 ? head : 0;
  s.tail0 = tail0;
  s.n_tail = rank == G - 1 ? L - tail0 : 0;
  s.lo = rank == 0 ? 0 : s.j0;
  s.hi = rank == G - 1 ? L : head + 4 * q1;
  return s;
}

// The unaligned head/tail position of this thread, if any (at most one).
__device__ __forceinline__ bool edge_position(const Slice& s, int32_t* j) {
  const int tid = threadIdx.x;
  if (tid < s.n_head) {
    *j = tid;
    return true;
  }
  if (tid >= 4 && tid - 4 < s.n_tail) {
    *j = s.tail0 + (tid - 4);
    return true;
  }
  *j = 0;
  return false;
}

// Calls f(valid, key, position) for every position of the slice. Control flow is
// block-uniform; `valid` is false for padding lanes.
template <class F>
__device__ __forceinline__ void visit_keys(const Slice& s, F&& f) {
  const int tid = threadIdx.x;
  {
    int32_t j;
    const bool ok = edge_position(s, &j);
    const uint32_t key = ok ? order_key(__float_as_uint(s.row[j])) : 0u;
    f(ok, key, j);
  }
  for (int32_t base = 0; base < s.nq; base += kUnroll * kThreads) {
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t q = base + u * kThreads + tid;
      x[u] = q < s.nq ? ld_stream(s.vec + q) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t q = base + u * kThreads + tid;
      const bool ok = q < s.nq;
      const int32_t j = s.j0 + 4 * q;
      f(ok, order_key(x[u].x), j);
      f(ok, order_key(x[u].y), j + 1);
      f(ok, order_key(x[u].z), j + 2);
      f(ok, order_key(x[u].w), j + 3);
    }
  }
}

// Bulk L2 prefetch of a slice's aligned body, in 16 KB pieces over the threads
// from `first` on (the issuing threads wait while the copy engine's queue is full,
// so the caller picks threads that are not on the critical path).
__device__ __forceinline__ void prefetch_slice(const Slice& s, int first = 0) {
  const uint64_t bytes = 16ull * static_cast<uint64_t>(s.nq);
  const uint64_t pieces = (bytes + kPrefetchBytes - 1) / kPrefetchBytes;
  const int t = static_cast<int>(threadIdx.x) - first;
  if (t < 0) return;
  for (uint64_t i = static_cast<uint64_t>(t); i < pieces; i += static_cast<uint64_t>(kThreads - first))
    prefetch_l2(reinterpret_cast<const char*>(s.vec) + i * kPrefetchBytes,
                static_cast<uint32_t>(min(static_cast<uint64_t>(kPrefetchBytes),
                                          bytes - i * kPrefetchBytes)));
}

// ------------------------------------------------------------------ output map

struct OutMap {
  const int32_t* pt_row;  // paged: this row's page table (global memory)
  const int32_t* pt_smem; // paged: the same entries staged in shared memory, or null
  int32_t pt_n;           // paged: entries of the row that may be read (the row's pages,
                          // at most the table's row stride)
  int32_t ps;             // page size
  int32_t ps_shift;       // log2(ps) or -1
  int32_t rstart;         // ragged: row start in the packed buffer; window: its first column
  float* values;          // this row's values output, or null
  uint2* staged;          // this row's (key, position) staging for the sort pass, or null
};

// The kernels' template argument F is a Form, plus kOpts when the launch has the
// values output or the sorted option (so that launches without them carry neither).
constexpr int kOpts = 4;
// ... and kSingle for launches of one CTA per row (no cluster code at all), and
// kKeysInFilter for single-CTA rows whose filter reads each candidate's value back
// from L1 at once (instead of from L2 in a pass after the filter)
constexpr int kSingle = 8;
constexpr int kKeysInFilter = 16;
// ... and kStaged for single-CTA rows on the staged tier (the whole row copied to
// shared memory at kernel start; 512-thread build only)
constexpr int kStaged = 32;
// ... and kHalfStage with kStaged for the staged tier with half a row of staging
// (two CTAs per SM)
constexpr int kHalfStage = 64;
__host__ __device__ constexpr int form_of(int F) { return F & 3; }
__host__ __device__ constexpr bool opts_of(int F) { return (F & kOpts) != 0; }

// The fp32 bit pattern of an order-preserving key (the inverse of order_key).
__device__ __forceinline__ uint32_t key_bits(uint32_t key) {
  return (key & 0x80000000u) != 0u ? key ^ 0x80000000u : ~key;
}

template <int F>
__device__ __forceinline__ int32_t map_pos(const OutMap& m, int32_t j) {
  if constexpr (form_of(F) == kPaged) {
    int32_t page, off;
    if (m.ps_shift >= 0) {
      page = j >> m.ps_shift;
      off = j & (m.ps - 1);
    } else {
      page = j / m.ps;
      off = j - page * m.ps;
    }
    // a page past the row's entries (a table narrower than the row; counted once per
    // row where pt_n is set) is not read
    if (page >= m.pt_n) return -1;
    const int32_t phys = m.pt_smem != nullptr ? m.pt_smem[page] : __ldg(m.pt_row + page);
    return phys * m.ps + off;
  } else if constexpr (form_of(F) == kRagged || form_of(F) == kWindow) {
    return m.rstart + j;
  } else {
    return j;
  }
}

// Every write of a row's output goes through here: position j with key `key` in
// slot `slot`, mapped, and its value when asked for; or, for the sorted output,
// the pair (key, j) to the staging buffer the sort pass orders. Slots at or beyond
// k are dropped. By construction no slot is ever >= k; the check keeps a miscount
// (say, scores modified while the kernel runs) from writing outside the row.
template <int F>
__device__ __forceinline__ void emit(int32_t* out, int32_t k, uint32_t slot, const OutMap& m,
                                     int32_t j, uint32_t key) {
  if (slot >= static_cast<uint32_t>(k)) return;  // the callers' checks count misses
  if constexpr (opts_of(F)) {
    if (m.staged != nullptr) {
      m.staged[slot] = make_uint2(key, static_cast<uint32_t>(j));
      return;
    }
    if (m.values != nullptr) m.values[slot] = __uint_as_float(key_bits(key));
  }
  out[slot] = map_pos<F>(m, j);
}

// An empty slot: -1 (and -inf for the value), or the padding pair of the staging.
template <int F>
__device__ __forceinline__ void emit_pad(int32_t* out, uint32_t slot, const OutMap& m) {
  if constexpr (opts_of(F)) {
    if (m.staged != nullptr) {
      m.staged[slot] = make_uint2(0u, 0xFFFFFFFFu);
      return;
    }
    if (m.values != nullptr) m.values[slot] = __uint_as_float(0xFF800000u);  // -inf
  }
  out[slot] = -1;
}

// ------------------------------------------------------------------ fast tier

// F1a: the sample of a CTA's part of the row: keys of the sampled 16-byte
// quads and the row position of each quad's first element (INT32_MAX when the
// thread has no quad). An element counts only if its position is below the row's
// length, which for the raw and paged forms is read while the sample is in flight.
template <int Q = kSampleQuads>
struct SampleT {
  static constexpr int kQuads = Q;  // sampled quads per thread
  uint32_t key[4 * Q];
  int32_t j[Q];
};
using Sample = SampleT<>;

// The sample is taken in runs of 32 consecutive quads (512 bytes, one per warp and
// round) spread evenly over the slice: whole DRAM bursts instead of one 16-byte
// piece of every few lines, so the sample arrives sooner; the later stream finds
// these lines in L2.
template <class Smp>
__device__ __forceinline__ void load_sample(const Slice& s, Smp& sm) {
  constexpr int kSampleQuads = Smp::kQuads;
  constexpr int32_t kRuns = kWarps * kSampleQuads;
  const int32_t spacing = max(32, s.nq / kRuns);  // quads from one run to the next
#pragma unroll
  for (int r = 0; r < kSampleQuads; ++r) {
    const int32_t run = static_cast<int32_t>(threadIdx.x >> 5) + r * kWarps;
    const int32_t q = run * spacing + static_cast<int32_t>(threadIdx.x & 31);
    const bool ok = q < s.nq;
    const uint4 x = ok ? ld_stream(s.vec + q) : make_uint4(0, 0, 0, 0);
    sm.key[4 * r + 0] = order_key(x.x);
    sm.key[4 * r + 1] = order_key(x.y);
    sm.key[4 * r + 2] = order_key(x.z);
    sm.key[4 * r + 3] = order_key(x.w);
    sm.j[r] = ok ? s.j0 + 4 * q : INT32_MAX;
  }
}

template <class Smp>
__device__ __forceinline__ bool sample_valid(const Smp& sm, int i, int32_t L) {
  return sm.j[i / 4] < L - (i & 3);
}

// Sums the `words` words of this CTA's histogram region h into the same region of
// CTA 0 (mh, G > 1), then a cluster barrier.
__device__ __forceinline__ void merge_into_cta0(const uint32_t* h, uint32_t* mh, int words) {
  const uint32_t m0 = map_rank(smem_addr(mh), 0);
  for (int i = threadIdx.x; i < words; i += kThreads) {
    const uint32_t v = h[i];
    if (v != 0) dsmem_add(m0 + 4u * static_cast<uint32_t>(i), v);
  }
  cluster_sync();
}

// F1b: lambda and the candidate-histogram bin width from the cluster's sample (see
// the header comment). The kH1 and kH2 regions of `hist` and of CTA 0's `mhist`
// are zero on entry, and so is CTA 0's ctl.ns. Returns lambda; *shift2 gets the
// candidate-histogram bin width exponent.
template <class Smp>
__device__ __forceinline__ uint32_t sample_lambda(const Smp& sm, const Slice& s, bool prefetched,
                                                  int32_t L, uint32_t k, int G, int rank,
                                                  uint32_t* hist, uint32_t* mhist, Ctl& ctl,
                                                  uint32_t* shift2, uint32_t cap = 0xFFFFFFFFu,
                                                  bool predict = false) {
  constexpr int kSampleQuads = Smp::kQuads;
  const int tid = threadIdx.x;
  const bool finder = rank == 0 && tid < 32;  // the warp that finds the thresholds
  // first sample round: coarse bins (top 10 key bits), one shared atomic per sample key (this
  // measured faster than first aggregating a warp's equal bins with a match). The
  // valid sample size goes to CTA 0.
  uint32_t mine = 0;
#pragma unroll
  for (int i = 0; i < 4 * kSampleQuads; ++i) {
    const bool v = sample_valid(sm, i, L);
    const uint32_t bin = sm.key[i] >> (32 - kFastBits);
    if (v) atomicAdd(&hist[kH1 + hist_index(static_cast<int>(bin))], 1u);
    mine += v ? 1u : 0u;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(kFull, mine, off);
  if ((tid & 31) == 0 && mine != 0) {
    if (G == 1)
      atomicAdd(&ctl.ns, mine);
    else
      dsmem_add(map_rank(smem_addr(&ctl.ns), 0), mine);
  }
  __syncthreads();
  if (G > 1) merge_into_cta0(hist + kH1, mhist + kH1, kFastWords);
  // the sample has arrived: now the bulk of the slice, issued by the last warp
  // before the thresholds are looked for
  if (!prefetched) prefetch_slice(s, kThreads - 32);
  // sample ranks a few standard deviations either side of the expected sample rank
  // of the row's k-th key; CTA 0 finds their coarse bins
  uint32_t rs = 0, rs_lo = 0;
  if (rank == 0) {
    const uint32_t ns = ctl.ns;
    if (ns != 0) {
      // four standard deviations on lambda's side (a lambda above the k-th key
      // costs the exact tier: about 3e-5 of rows), three on the other (it only sets
      // the candidate-histogram bin width)
      // (approximate arithmetic is enough: any ranks give an exact result, these
      // only make the fast tier likely)
      const float mean =
          fmaxf(__fdividef(static_cast<float>(k) * static_cast<float>(ns), static_cast<float>(L)),
                1.0f);
      const float sd = mean * rsqrtf(mean);
      rs = min(static_cast<uint32_t>(ceilf(mean + 4.0f * sd)) + 2u, ns);
      const float lo = floorf(mean - 3.0f * sd);
      rs_lo = min(lo < 1.0f ? 1u : static_cast<uint32_t>(lo), rs);
    }
    block_find2<kFastBins / kThreads>((G > 1 ? mhist : hist) + kH1, rs, rs_lo, ns != 0, ctl);
    __syncthreads();
  }
  if (finder) {
    const uint32_t ns = ctl.ns;
    __syncwarp();
    if (tid == 0) {
      constexpr int kC = 32 - kFastBits;  // coarse bin width exponent
      if (ns != 0) {
        // fine window: coarse bins sel_t .. sel2_t in at most kFastBins fine bins
        const uint64_t span = static_cast<uint64_t>(ctl.sel2_t + 1 - ctl.sel_t) << kC;
        const int f = max(0, (64 - __clzll(static_cast<long long>(span - 1))) - kFastBits);
        ctl.win_lo = ctl.sel_t << kC;
        ctl.win_shift = static_cast<uint32_t>(f);
        ctl.win_above = ctl.sel2_above;  // sample keys above the window
      } else {  // no sample below the row's length: an empty window, lambda = 0
        ctl.sel2_t = 0;
        ctl.win_lo = 0;
        ctl.win_shift = kC;
        ctl.win_above = 0;
      }
    }
    __syncwarp();
    if (G > 1 && tid > 0 && tid < G) {
      dsmem_st(map_rank(smem_addr(&ctl.win_lo), tid), ctl.win_lo);
      dsmem_st(map_rank(smem_addr(&ctl.win_shift), tid), ctl.win_shift);
      dsmem_st(map_rank(smem_addr(&ctl.win_above), tid), ctl.win_above);
      dsmem_st(map_rank(smem_addr(&ctl.sel2_t), tid), ctl.sel2_t);
    }
  }
  if (G > 1)
    cluster_sync();
  else
    __syncthreads();

  // second sample round: fine bins over [win_lo, end of coarse bin sel2_t]
  const uint32_t win_lo = ctl.win_lo, f = ctl.win_shift, win_above = ctl.win_above;
  const uint64_t span =
      (static_cast<uint64_t>(ctl.sel2_t + 1) << (32 - kFastBits)) - static_cast<uint64_t>(win_lo);
#pragma unroll
  for (int i = 0; i < 4 * kSampleQuads; ++i) {
    const uint64_t d = static_cast<uint64_t>(sm.key[i]) - win_lo;  // wraps for keys below
    if (sample_valid(sm, i, L) && sm.key[i] >= win_lo && d < span)
      atomicAdd(&hist[kH2 + hist_index(static_cast<int>(d >> f))], 1u);
  }
  __syncthreads();
  if (G > 1) merge_into_cta0(hist + kH2, mhist + kH2, kFastWords);
  if (rank == 0) {
    block_find2<kFastBins / kThreads>((G > 1 ? mhist : hist) + kH2, rs != 0 ? rs - win_above : 0u,
                                      rs_lo - win_above, rs != 0, ctl);
    __syncthreads();
  }
  if (finder) {
    __syncwarp();
    if (tid == 0) {
      if (rs != 0) {
        // [lambda, lambda_hi] spans fewer than 1024 candidate bins
        const uint32_t lam = win_lo + (ctl.sel_t << f);
        const uint64_t hi =
            static_cast<uint64_t>(win_lo) + (static_cast<uint64_t>(ctl.sel2_t + 1) << f) - 1;
        const uint64_t gap = hi > lam ? hi - lam : 0;
        const int bits = 64 - __clzll(static_cast<long long>(gap));
        ctl.lambda = lam;
        ctl.lambda_shift = static_cast<uint32_t>(max(0, bits - (kCandBits - 1)));
        // (predict) the sample keys at or above lambda, scaled to the row: the filter's
        // expected candidate count. Far over the buffer (scores packed into a few
        // values), the filter pass would only find that out: the row goes to the exact
        // tier at once.
        if (predict) {
          const uint32_t at_or_above = win_above + ctl.sel_above + ctl.sel_count;
          const float expect = __fdividef(static_cast<float>(at_or_above) * static_cast<float>(L),
                                          static_cast<float>(max(ctl.ns, 1u)));
          ctl.skip_fast = expect > 2.0f * static_cast<float>(cap) ? 1u : 0u;
          // the exact tier then starts below the bits that lambda and lambda_hi share
          // (every bit when they are equal: scores packed into a few values)
          ctl.ex_shift = 32u - static_cast<uint32_t>(__clz(lam ^ static_cast<uint32_t>(hi)));
        }
      } else {
        ctl.lambda = 0;
        ctl.lambda_shift = 32 - kCandBits;
        if (predict) {
          ctl.skip_fast = 0;
          ctl.ex_shift = 32;
        }
      }
    }
    __syncwarp();
    if (G > 1 && tid > 0 && tid < G) {
      dsmem_st(map_rank(smem_addr(&ctl.lambda), tid), ctl.lambda);
      dsmem_st(map_rank(smem_addr(&ctl.lambda_shift), tid), ctl.lambda_shift);
      if (predict) {
        dsmem_st(map_rank(smem_addr(&ctl.skip_fast), tid), ctl.skip_fast);
        dsmem_st(map_rank(smem_addr(&ctl.ex_shift), tid), ctl.ex_shift);
      }
    }
  }
  if (G > 1)
    cluster_sync();
  else
    __syncthreads();
  *shift2 = ctl.lambda_shift;
  return ctl.lambda;
}

// F2: "key >= lambda" on raw fp32 bits. kPos: lambda is the key of a non-negative
// value, so the test is "(int)bits >= lambda ^ 2^31"; otherwise "bits <= ~lambda"
// (unsigned).
template <bool kPos>
__device__ __forceinline__ bool is_candidate(uint32_t bits, uint32_t thr) {
  if constexpr (kPos)
    return static_cast<int32_t>(bits) >= static_cast<int32_t>(thr);
  else
    return bits <= thr;
}

// The candidate histogram (bin = min((key - lambda) >> shift, kCandBins - 1)) of the
// n candidates in buf, counted by every thread (chist zero on entry; a barrier at the
// end). Counting it in the filters' per-candidate loops measured slower.
__device__ __forceinline__ void count_candidates(const uint2* buf, uint32_t n, uint32_t lambda,
                                                 uint32_t shift, uint32_t* chist) {
  uint32_t top = 0;  // the last bin, counted per warp
  for (uint32_t i = threadIdx.x; i < n; i += kThreads) {
    const uint32_t d = (buf[i].x - lambda) >> shift;
    if (d >= static_cast<uint32_t>(kCandBins - 1))
      ++top;
    else
      atomicAdd(&chist[hist_index(static_cast<int>(d))], 1u);
  }
  top = __reduce_add_sync(kFull, top);
  if ((threadIdx.x & 31) == 0 && top != 0) atomicAdd(&chist[hist_index(kCandBins - 1)], top);
  __syncthreads();
}

// F2, a row owned by one CTA: stream the row, keep per lane a 32-bit candidate
// mask per iteration (8 quads), and every MI iterations turn the masks into
// candidates written compactly into the buffer at slots from one reservation per
// warp and group on the CTA's counter (ctl.cand_cnt, zero on entry). Holding only
// masks lets the loads of a whole group be in flight together. The loads keep their
// lines in L1. Without kKeys only positions are written (entry .y; fill_candidates
// reads the values back afterwards, mostly from L1: keeping the lines there measured
// 0.5 us faster at one row, against streaming them past L1 and reading back from L2);
// with kKeys the masks are decoded
// every iteration (MI = 1) and each candidate's value is read back from L1 at
// once, so the entry gets its key (its histogram comes from count_candidates).
// Slots at or beyond `cap` are counted but not written.
template <bool kPos, bool kKeys>
__device__ __forceinline__ void filter_positions(const Slice& s, uint32_t lambda, uint2* buf,
                                                 uint32_t cap, Ctl& ctl) {
  const int tid = threadIdx.x;
  const uint32_t thr = kPos ? (lambda ^ 0x80000000u) : ~lambda;
  constexpr int U = kFilterUnroll;
  constexpr int MI = kKeys ? 1 : kMaskIters;
  constexpr int32_t kStep = U * kThreads;
  int32_t ej;
  const bool edge = edge_position(s, &ej) && is_candidate<kPos>(__float_as_uint(s.row[ej]), thr);
  bool first = true;
  for (int32_t gbase = 0; first || gbase < s.nq; gbase += MI * kStep) {
    uint32_t mk[MI];
#pragma unroll
    for (int it = 0; it < MI; ++it) {
      const int32_t base = gbase + it * kStep;
      uint32_t m = 0;
      if (base < s.nq) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int32_t q = base + u * kThreads + tid;
          x[u] = q < s.nq ? ld_keep(s.vec + q)
                          : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const bool ok = base + u * kThreads + tid < s.nq;
          m |= static_cast<uint32_t>(ok && is_candidate<kPos>(x[u].x, thr)) << (4 * u + 0);
          m |= static_cast<uint32_t>(ok && is_candidate<kPos>(x[u].y, thr)) << (4 * u + 1);
          m |= static_cast<uint32_t>(ok && is_candidate<kPos>(x[u].z, thr)) << (4 * u + 2);
          m |= static_cast<uint32_t>(ok && is_candidate<kPos>(x[u].w, thr)) << (4 * u + 3);
        }
      }
      mk[it] = m;
    }
    const bool with_edge = first && edge;
    uint32_t n = with_edge ? 1u : 0u;
#pragma unroll
    for (int it = 0; it < MI; ++it) n += static_cast<uint32_t>(__popc(mk[it]));
    uint32_t slot = warp_reserve(&ctl.cand_cnt, 0u, false, n);
    {
      auto put = [&](int32_t j) {
        if constexpr (kKeys) {
          const uint32_t key = order_key(__float_as_uint(__ldg(s.row + j)));  // from L1
          if (slot < cap) buf[slot] = make_uint2(key, static_cast<uint32_t>(j));
        } else {
          if (slot < cap) buf[slot].y = static_cast<uint32_t>(j);
        }
        ++slot;
      };
      if (with_edge) put(ej);
#pragma unroll
      for (int it = 0; it < MI; ++it) {
        uint32_t mm = mk[it];
        const int32_t base = gbase + it * kStep;
        while (mm != 0u) {
          const int b = __ffs(mm) - 1;
          mm &= mm - 1u;
          put(s.j0 + 4 * (base + (b >> 2) * kThreads + tid) + (b & 3));
        }
      }
    }
    first = false;
  }
}

// F2, a row owned by one CTA: the n buffered positions get their keys, read back
// (from L1, where the filter kept the row, or from L2) in batches of 2048, and the
// candidate histogram (bin = min((key - lambda) >> shift, kCandBins - 1)) is counted
// in `chist`, which is zero on entry. The last bin collects most candidates, so it is
// counted per warp (ballot) rather than by one shared atomic per candidate.
__device__ __forceinline__ void fill_candidates(const float* row, uint2* buf, uint32_t n,
                                                uint32_t lambda, uint32_t shift,
                                                uint32_t* chist, Ctl& ctl) {
  const int tid = threadIdx.x;
  // 2048 candidates per batch whatever the CTA size: one L2 round trip for the
  // candidate counts the fast tier normally sees
  constexpr int kPer = 2048 / kThreads;
  // the loop bound is the same for every thread (the ballot below needs whole warps)
  for (uint32_t base = 0; base < n; base += kPer * kThreads) {
    const uint32_t i0 = base + static_cast<uint32_t>(tid);
    uint32_t bits[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const uint32_t i = i0 + r * kThreads;
      bits[r] = i < n ? __float_as_uint(__ldg(row + buf[i].y)) : 0u;
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const uint32_t i = i0 + r * kThreads;
      const uint32_t key = order_key(bits[r]);
      const uint32_t d = (key - lambda) >> shift;
      const bool top = i < n && d >= static_cast<uint32_t>(kCandBins - 1);
      if (i < n) {
        buf[i].x = key;
        if (!top) atomicAdd(&chist[hist_index(static_cast<int>(d))], 1u);
      }
      const uint32_t b = __ballot_sync(kFull, top);
      if ((tid & 31) == 0 && b != 0)
        atomicAdd(&chist[hist_index(kCandBins - 1)], static_cast<uint32_t>(__popc(b)));
    }
  }
  __syncthreads();
}

// F2, a row split over a cluster: stream the slice; every element with key >=
// lambda goes, as (key, position), to CTA 0's buffer, so that CTA 0 does not have to
// read the keys back for the whole row (it counts their histogram from its buffer
// afterwards: counting per CTA and summing over the cluster measured 0.9 us slower on
// 262144-element rows). Slots come from one reservation per warp and iteration on
// CTA 0's counter through distributed shared memory; slots at or beyond `cap` are
// counted but not written. `remote`: this CTA is not CTA 0.
template <bool kPos>
__device__ __forceinline__ void filter_candidates(const Slice& s, uint32_t lambda, uint2* buf,
                                                  uint32_t buf_remote, uint32_t cnt_remote,
                                                  bool remote, uint32_t cap, Ctl& ctl) {
  const int tid = threadIdx.x;
  const uint32_t thr = kPos ? (lambda ^ 0x80000000u) : ~lambda;
  constexpr int U = kFilterUnroll;
  constexpr int32_t kStep = U * kThreads;
  auto put = [&](uint32_t slot, uint32_t bits, int32_t j) {
    const uint32_t key = order_key(bits);
    if (slot < cap) {
      if (remote)
        dsmem_st2(buf_remote + 8u * slot, key, static_cast<uint32_t>(j));
      else
        buf[slot] = make_uint2(key, static_cast<uint32_t>(j));
    }
  };
  {  // the unaligned head/tail element of this thread, if any
    int32_t ej;
    const bool e = edge_position(s, &ej);
    const uint32_t bits = e ? __float_as_uint(s.row[ej]) : 0u;
    const bool c = e && is_candidate<kPos>(bits, thr);
    const uint32_t slot = warp_reserve(&ctl.cand_cnt, cnt_remote, true, c ? 1u : 0u);
    if (c) put(slot, bits, ej);
  }
  for (int32_t base = 0; base < s.nq; base += kStep) {
    uint4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int32_t q = base + u * kThreads + tid;
      x[u] = q < s.nq ? ld_stream(s.vec + q) : make_uint4(0, 0, 0, 0);
    }
    uint32_t m = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool ok = base + u * kThreads + tid < s.nq;
      m |= static_cast<uint32_t>(ok && is_candidate<kPos>(x[u].x, thr)) << (4 * u + 0);
      m |= static_cast<uint32_t>(ok && is_candidate<kPos>(x[u].y, thr)) << (4 * u + 1);
      m |= static_cast<uint32_t>(ok && is_candidate<kPos>(x[u].z, thr)) << (4 * u + 2);
      m |= static_cast<uint32_t>(ok && is_candidate<kPos>(x[u].w, thr)) << (4 * u + 3);
    }
    uint32_t slot = warp_reserve(&ctl.cand_cnt, cnt_remote, true,
                                 static_cast<uint32_t>(__popc(m)));
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint32_t nib = (m >> (4 * u)) & 15u;
      const int32_t j = s.j0 + 4 * (base + u * kThreads + tid);
      while (nib != 0u) {
        const int c = __ffs(nib) - 1;
        nib &= nib - 1u;
        const uint32_t bits = c == 0 ? x[u].x : c == 1 ? x[u].y : c == 2 ? x[u].z : x[u].w;
        put(slot++, bits, j + c);
      }
    }
  }
}

// ------------------------------------------------------------------ selection in a buffer

__device__ __forceinline__ uint64_t hi_bits(uint64_t v, int p) { return p >= 64 ? 0ull : v >> p; }

// F3 / E3 (CTA 0 only): among the c buffered (key, position) entries, all with
// composite (key:~position) >> p == P, select the `need` largest composites and
// write them mapped to out[k_above + ...]. h is a scratch histogram.
template <int F>
__device__ __forceinline__ void select_in_buffer(const uint2* buf, uint32_t c, uint32_t need,
                                                 uint64_t P, int p, int32_t L, int32_t* out,
                                                 int32_t k, uint32_t k_above, const OutMap& m,
                                                 uint32_t* h, Ctl& ctl) {
  const int tid = threadIdx.x;
  auto compose = [](uint2 e) -> uint64_t {
    return (static_cast<uint64_t>(e.x) << 32) | static_cast<uint64_t>(~e.y);
  };
  const uint32_t want = need;  // entries to write
  if (need < c) {
    const int nb = 32 - __clz(L - 1);  // positions fit in nb bits (L >= 2 here)
    for (;;) {
      if (p == 32) {  // key resolved: the ~position bits above nb are all ones
        const int skip = 32 - nb;
        P = (P << skip) | ((1ull << skip) - 1ull);
        p = nb;
      }
      // Composites are unique (positions are), so the loop ends with the threshold
      // bin holding exactly what is still needed, at the latest when p reaches 0;
      // the test below only bounds the loop should that ever not hold.
      if (p <= 0) {
        if (tid == 0) guard_hit();
        break;
      }
      const int lo = p > 32 ? 32 : 0;
      const int w = min(kBufRoundBits, p - lo);
      const int np = p - w;
      const uint32_t mask = (1u << w) - 1u;
      for (int i = tid; i < hist_index(static_cast<int>(mask) + 1); i += kThreads) h[i] = 0;
      __syncthreads();
      for (uint32_t i = tid; i < c; i += kThreads) {
        const uint64_t v = compose(buf[i]);
        if (hi_bits(v, p) == P)
          atomicAdd(&h[hist_index(static_cast<int>(static_cast<uint32_t>(v >> np) & mask))], 1u);
      }
      __syncthreads();
      find_threshold(h, 1 << w, need, ctl);
      const uint32_t t = ctl.sel_t, above = ctl.sel_above, ct = ctl.sel_count;
      need -= above;
      P = (P << w) | t;
      p = np;
      if (ct == need) break;
    }
  }
  // every entry whose composite prefix is >= P is selected
  const uint32_t cpad = (c + kThreads - 1) / kThreads * kThreads;
  for (uint32_t i = tid; i < cpad; i += kThreads) {
    bool sel = false;
    uint2 e = make_uint2(0, 0);
    if (i < c) {
      e = buf[i];
      sel = hi_bits(compose(e), p) >= P;
    }
    const uint32_t slot = warp_reserve_bit(&ctl.out_cnt, sel);
    if (sel) {
      if (slot < want)
        emit<F>(out, k, k_above + slot, m, static_cast<int32_t>(e.y), e.x);
      else
        guard_hit();
    }
  }
}

// The k selected positions of a row, staged in shared memory slot by slot (slots
// [0, upto)), written to out at once: coalesced stores from every thread, and one
// copy of the mapping code. A slot holding no position of the row (possible only
// when the scores changed while the kernel ran) is written as -1.
template <int F>
__device__ __forceinline__ void write_slots(const int32_t* slots, uint32_t upto, int32_t L,
                                            int32_t* out, const OutMap& m) {
  if constexpr (form_of(F) == kPaged) {
    if (m.pt_smem != nullptr && m.ps_shift >= 0) {  // the usual case, with no branch per slot
      const int32_t sh = m.ps_shift, msk = m.ps - 1;
      for (uint32_t i = threadIdx.x; i < upto; i += kThreads) {
        const int32_t j = slots[i];
        const int32_t page = j >> sh;
        const bool ok = static_cast<uint32_t>(j) < static_cast<uint32_t>(L) && page < m.pt_n;
        out[i] = ok ? m.pt_smem[page] * m.ps + (j & msk) : -1;
      }
      return;
    }
  }
  for (uint32_t i = threadIdx.x; i < upto; i += kThreads) {
    const int32_t j = slots[i];
    out[i] = static_cast<uint32_t>(j) < static_cast<uint32_t>(L) ? map_pos<F>(m, j) : -1;
  }
}

// F3 (CTA 0 only): the filter left n candidates in buf and their histogram (bin =
// min((key - lambda) >> shift, kCandBins - 1)) in chist. Writes the k largest composites
// (key, ~position) mapped to out. h may be chist itself: it is used only after
// chist has been read. Launches without the values or sorted outputs stage the
// positions in `slots` (k words of shared memory that may overlap h but nothing
// else) and write them out at the end; the others emit each slot as it is decided.
template <int F>
__device__ __forceinline__ void select_candidates(const uint2* buf, uint32_t n, uint32_t k,
                                                  uint32_t* chist, uint32_t lambda,
                                                  uint32_t shift, uint2* list, uint32_t* h,
                                                  int32_t* slots, int32_t L, int32_t* out,
                                                  const OutMap& m, Ctl& ctl) {
  constexpr bool kSlots = !opts_of(F);
  const int tid = threadIdx.x;
  // slot s gets position j (key `key`)
  auto put = [&](uint32_t s, uint2 e) {
    if constexpr (kSlots)
      slots[s] = static_cast<int32_t>(e.y);
    else
      emit<F>(out, static_cast<int32_t>(k), s, m, static_cast<int32_t>(e.y), e.x);
  };
  block_find2<kCandBins / kThreads>(chist, k, 0u, false, ctl);
  __syncthreads();
  const uint32_t t = ctl.sel_t, above = ctl.sel_above, ct = ctl.sel_count;
  if (__builtin_expect(ct > static_cast<uint32_t>(kListCap), 0)) {
    select_in_buffer<F>(buf, n, k, 0ull, 64, L, out, static_cast<int32_t>(k), 0u, m, h, ctl);
    return;
  }
  // candidates above the threshold bin are winners; the bin's go to the list. Each
  // thread classifies up to kClsR entries of the buffer at once (entries base +
  // r kThreads + tid), held in registers; a block scan of the packed (winners, ties)
  // counts then gives each thread its first slot of each kind.
  constexpr int kClsR = 8;
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t run = 0;  // (winners, ties) slots taken by the earlier sweeps, packed
  for (uint32_t base = 0; base < n; base += static_cast<uint32_t>(kClsR * kThreads)) {
    uint2 e[kClsR];
    uint32_t wb = 0, tb = 0;
#pragma unroll
    for (int r = 0; r < kClsR; ++r) {
      const uint32_t i = base + static_cast<uint32_t>(r * kThreads + tid);
      const bool live = i < n;
      e[r] = live ? buf[i] : make_uint2(0u, 0u);
      const uint32_t b = min((e[r].x - lambda) >> shift, static_cast<uint32_t>(kCandBins - 1));
      wb |= static_cast<uint32_t>(live && b > t) << r;
      tb |= static_cast<uint32_t>(live && b == t) << r;
    }
    // winners number above < k and ties ct <= kListCap: each fits 16 bits
    const uint32_t mine = static_cast<uint32_t>(__popc(wb)) | (static_cast<uint32_t>(__popc(tb)) << 16);
    uint32_t x = mine;  // inclusive prefix over the warp's lanes
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) ctl.scan[warp] = x;
    __syncthreads();
    const uint32_t sw = lane < kWarps ? ctl.scan[lane] : 0u;
    const uint32_t first = run + __reduce_add_sync(kFull, lane < warp ? sw : 0u) + x - mine;
    run += __reduce_add_sync(kFull, sw);
    // entry r's slot: the first slot plus this thread's entries of its kind before r;
    // stores predicated on the entry's kind, the slots' bounds counted afterwards
    const uint32_t ws = first & 0xFFFFu, ts = first >> 16;
#pragma unroll
    for (int r = 0; r < kClsR; ++r) {
      const uint32_t below = (1u << r) - 1u;
      const uint32_t wr = ws + static_cast<uint32_t>(__popc(wb & below));
      const uint32_t tr = ts + static_cast<uint32_t>(__popc(tb & below));
      if (((wb >> r) & 1u) != 0u && wr < above) put(wr, e[r]);
      if (((tb >> r) & 1u) != 0u && tr < ct) list[tr] = e[r];
    }
    // slots past the bin's counts (only if the scores changed under the kernel)
    if (wb != 0u && ws + static_cast<uint32_t>(__popc(wb)) > above) guard_hit();
    if (tb != 0u && ts + static_cast<uint32_t>(__popc(tb)) > ct) guard_hit();
    if (base + static_cast<uint32_t>(kClsR * kThreads) < n) __syncthreads();  // ctl.scan again
  }
  __syncthreads();
  const uint32_t need = k - above;  // 1 <= need <= ct
  // entry o ranks before entry e: a larger key, or an equal key at a smaller position
  auto before = [](uint2 e, uint32_t ox, uint32_t oy) -> uint32_t {
    return static_cast<uint32_t>(ox > e.x) |
           (static_cast<uint32_t>(ox == e.x) & static_cast<uint32_t>(oy < e.y));
  };
  if (ct <= 32u) {  // order the bin by counting, one thread per entry
    if (static_cast<uint32_t>(tid) < ct) {
      const uint2 e = list[tid];
      uint32_t r = 0;
      for (uint32_t j = 0; j < ct; ++j) {
        const uint2 o = list[j];
        r += before(e, o.x, o.y);
      }
      if (r < need) put(above + r, e);
    }
    if constexpr (kSlots) {
      __syncthreads();
      write_slots<F>(slots, k, L, out, m);
    }
    return;
  }
  if (ct <= static_cast<uint32_t>(kRankDirect)) {
    // order the bin by counting: entry i takes slot above + (#entries ranked before
    // it). Each entry gets a group of g consecutive lanes (g a power of two, g * ct
    // <= kThreads, g <= ct and at most a warp) that split the comparisons and add
    // them up.
    int g = 32;
    while (g > 1 && (static_cast<uint32_t>(g) * ct > static_cast<uint32_t>(kThreads) ||
                     static_cast<uint32_t>(g) > ct))
      g >>= 1;
    const uint32_t i = static_cast<uint32_t>(tid) / static_cast<uint32_t>(g);
    const uint32_t part = static_cast<uint32_t>(tid) & static_cast<uint32_t>(g - 1);
    // the whole warp takes part in the shuffles; lanes past the last entry count nothing
    const bool live = i < ct;
    uint2 e = make_uint2(0u, 0u);
    uint32_t r = 0;
    if (live) {
      e = list[i];
      // two entries per 16-byte load: pairs (2q, 2q + 1), q = part, part + g, ...
      const uint4* pairs = reinterpret_cast<const uint4*>(list);
      const uint32_t npairs = ct >> 1;
      for (uint32_t q = part; q < npairs; q += static_cast<uint32_t>(g)) {
        const uint4 o = pairs[q];
        r += before(e, o.x, o.y) + before(e, o.z, o.w);
      }
      if ((ct & 1u) != 0u && part == static_cast<uint32_t>(g - 1)) {
        const uint2 o = list[ct - 1];
        r += before(e, o.x, o.y);
      }
    }
    if (tid < ((static_cast<int>(ct) * g + 31) & ~31)) {  // whole warps that hold an entry
      for (int off = g >> 1; off > 0; off >>= 1) r += __shfl_xor_sync(kFull, r, off);
      if (live && part == 0u && r < need) put(above + r, e);
    }
    if constexpr (kSlots) {
      __syncthreads();
      write_slots<F>(slots, k, L, out, m);
    }
    return;
  }
  if constexpr (kSlots) {  // the winners out first: h may overlap the slots
    write_slots<F>(slots, above, L, out, m);
    __syncthreads();
  }
  select_in_buffer<F>(list, ct, need, 0ull, 64, L, out, static_cast<int32_t>(k), above, m, h, ctl);
}

// ------------------------------------------------------------------ exact tier

// E2: winners (key >> shift > prefix) to out[win_base + ...], ties
// (key >> shift == prefix) to CTA 0's tie buffer at tie_base + ...
template <int F>
__device__ __forceinline__ void scatter_pass(const Slice& s, uint32_t prefix, int shift,
                                             int32_t* out, int32_t k, uint32_t win_base,
                                             uint32_t tie_base,
                                             uint2* ties, uint32_t ties_remote, bool remote,
                                             uint32_t cap, const OutMap& m, Ctl& ctl) {
  const int tid = threadIdx.x;
  auto put_tie = [&](uint32_t slot, uint32_t key, int32_t j) {
    if (slot >= cap) {
      guard_hit();
      return;
    }
    if (remote)
      dsmem_st2(ties_remote + 8u * slot, key, static_cast<uint32_t>(j));
    else
      ties[slot] = make_uint2(key, static_cast<uint32_t>(j));
  };
  {
    int32_t j;
    const bool ok = edge_position(s, &j);
    const uint32_t key = ok ? order_key(__float_as_uint(s.row[j])) : 0u;
    const bool win = ok && (key >> shift) > prefix;
    const bool tie = ok && (key >> shift) == prefix;
    const uint32_t ws = warp_reserve_bit(&ctl.win_cnt, win);
    const uint32_t ts = warp_reserve_bit(&ctl.tie_cnt, tie);
    if (win) emit<F>(out, k, win_base + ws, m, j, key);
    if (tie) put_tie(tie_base + ts, key, j);
  }
  for (int32_t base = 0; base < s.nq; base += kUnroll * kThreads) {
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t q = base + u * kThreads + tid;
      x[u] = q < s.nq ? ld_stream(s.vec + q) : make_uint4(0, 0, 0, 0);
    }
    uint32_t key[4 * kUnroll];
    uint32_t wb = 0, tb = 0;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const bool ok = base + u * kThreads + tid < s.nq;
      key[4 * u + 0] = order_key(x[u].x);
      key[4 * u + 1] = order_key(x[u].y);
      key[4 * u + 2] = order_key(x[u].z);
      key[4 * u + 3] = order_key(x[u].w);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t hi = key[4 * u + c] >> shift;
        wb |= static_cast<uint32_t>(ok && hi > prefix) << (4 * u + c);
        tb |= static_cast<uint32_t>(ok && hi == prefix) << (4 * u + c);
      }
    }
    if (__any_sync(kFull, (wb | tb) != 0u)) {
      uint32_t ws = warp_reserve(&ctl.win_cnt, 0u, false, __popc(wb));
      uint32_t ts = warp_reserve(&ctl.tie_cnt, 0u, false, __popc(tb));
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t j = s.j0 + 4 * (base + u * kThreads + tid);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int bit = 4 * u + c;
          if ((wb >> bit) & 1u) emit<F>(out, k, win_base + ws++, m, j + c, key[bit]);
          if ((tb >> bit) & 1u) put_tie(tie_base + ts++, key[bit], j + c);
        }
      }
    }
  }
}

// E4: key tau is exact and more elements than the tie buffer holds equal it.
// Each CTA scans its slice in position order, writes its winners (key > tau) and
// the first `quota` of its elements equal to tau.
template <int F>
__device__ __forceinline__ void emit_equal(const Slice& s, uint32_t tau, int32_t* out, int32_t k,
                                           uint32_t win_base, uint32_t eq_slot0,
                                           uint32_t quota, const OutMap& m, Ctl& ctl) {
  const int tid = threadIdx.x;
  uint32_t taken = 0;
  for (int32_t t0 = s.lo; t0 < s.hi; t0 += 4 * kThreads) {
    const int32_t j0 = t0 + 4 * tid;
    uint32_t key[4];
    uint32_t wb = 0, eb = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = j0 + u < s.hi;
      key[u] = ok ? order_key(__float_as_uint(s.row[j0 + u])) : 0u;
      wb |= static_cast<uint32_t>(ok && key[u] > tau) << u;
      eb |= static_cast<uint32_t>(ok && key[u] == tau) << u;
    }
    uint32_t ws = warp_reserve(&ctl.win_cnt, 0u, false, __popc(wb));
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if ((wb >> u) & 1u) emit<F>(out, k, win_base + ws++, m, j0 + u, key[u]);
    uint32_t total;
    uint32_t r = taken + block_excl_scan(__popc(eb), ctl, &total);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if ((eb >> u) & 1u) {
        if (r < quota) emit<F>(out, k, eq_slot0 + r, m, j0 + u, tau);
        ++r;
      }
    }
    taken += total;
  }
}

// ------------------------------------------------------------------ the kernel

// E1-E4: the exact tier over this CTA's slice s of a row of length L (CTA `rank` of
// a cluster of G). hist and, in CTA 0, mhist are zero on entry; buf holds `cap`
// (key, position) entries. Paged rows whose table was copied to shared memory
// (pages > 0 entries at pt_smem) wait for that copy here if nothing waited before.
// start_shift < 32: the first round looks only at keys whose bits above start_shift
// equal start_prefix (a window that the sample expects to hold the k-th key), and
// counts the keys above the window; if the k-th key is not in the window after all,
// the rounds start again from the top bits. The same value on every CTA of a cluster.
template <int F>
__device__ __forceinline__ void exact_tier(const Slice& s, int32_t L, int32_t k, int32_t* out,
                                           OutMap m, int32_t pages, int32_t* pt_smem, int G,
                                           int rank, uint32_t* hist, uint32_t* mhist, uint2* buf,
                                           uint32_t cap, Ctl& ctl, int start_shift = 32,
                                           uint32_t start_prefix = 0) {
  const int tid = threadIdx.x;
  if constexpr (form_of(F) == kPaged) {
    if (pages > 0 && m.pt_smem == nullptr) {  // the fast tier did not run
      cp_async_wait_all();
      __syncthreads();
      m.pt_smem = pt_smem;
    }
  }
  uint32_t need = static_cast<uint32_t>(k);  // winners still to find at or below the bin
  uint32_t prefix = 0;                       // known high bits of the threshold key
  int shift = 32;                            // prefix == threshold key >> shift
  uint32_t cnt = static_cast<uint32_t>(L);   // elements whose key >> shift == prefix
  uint32_t above_local = 0;                  // this CTA's elements above the bin
  uint32_t tie_local = 0;                    // this CTA's elements in the bin
  bool more = true;                          // another round is needed
  if (start_shift < 32) {
    // the window's round: keys >> start_shift above start_prefix are counted, keys equal
    // to it go to the histogram of their next w bits
    const int w = min(kRowRoundBits, start_shift);
    const int nshift = start_shift - w;
    const uint32_t mask = (1u << w) - 1u;
    uint32_t a = 0, in = 0;
    visit_keys(s, [&](bool ok, uint32_t key, int32_t) {
      const uint32_t hi = key >> start_shift;
      if (ok && hi == start_prefix) {
        atomicAdd(&hist[hist_index(static_cast<int>((key >> nshift) & mask))], 1u);
        ++in;
      }
      a += static_cast<uint32_t>(ok && hi > start_prefix);
    });
    const uint32_t a_cta = block_sum(a, ctl);
    const uint32_t in_cta = block_sum(in, ctl);
    uint32_t a_row = a_cta, in_row = in_cta;
    if (G > 1) {  // every CTA gets every CTA's two counts
      if (tid < G) {
        dsmem_st(map_rank(smem_addr(&ctl.xa[rank]), tid), a_cta);
        dsmem_st(map_rank(smem_addr(&ctl.xt[rank]), tid), in_cta);
      }
      cluster_sync();
      a_row = 0;
      in_row = 0;
      for (int r = 0; r < G; ++r) {
        a_row += ctl.xa[r];
        in_row += ctl.xt[r];
      }
    }
    if (a_row < need && need <= a_row + in_row) {  // the k-th key is in the window
      need -= a_row;
      const Sel sel = threshold_of(hist, mhist, 1 << w, need, G, rank, ctl);
      if (G == 1) {
        above_local = a_cta + sel.above;
        tie_local = sel.count;
      } else {
        uint32_t part = 0;
        for (int i = tid; i <= static_cast<int>(mask); i += kThreads)
          part += static_cast<uint32_t>(i) > sel.t ? hist[hist_index(i)] : 0u;
        tie_local = hist[hist_index(static_cast<int>(sel.t))];
        above_local = a_cta + block_sum(part, ctl);
      }
      need -= sel.above;
      prefix = (start_prefix << w) | sel.t;
      shift = nshift;
      cnt = sel.count;
      more = cnt > cap && shift != 0;
    } else {  // not: the rounds from the top bits (mhist is still zero)
      for (int i = tid; i < hist_index(static_cast<int>(mask) + 1); i += kThreads) hist[i] = 0;
      __syncthreads();
    }
  }
  while (more) {
    const int w = min(kRowRoundBits, shift);
    const int nshift = shift - w;
    const uint32_t mask = (1u << w) - 1u;
    if (shift != 32) {
      for (int i = tid; i < hist_index(static_cast<int>(mask) + 1); i += kThreads) hist[i] = 0;
      __syncthreads();
    }
    visit_keys(s, [&](bool ok, uint32_t key, int32_t) {
      if (ok && __funnelshift_rc(key, 0u, shift) == prefix)
        atomicAdd(&hist[hist_index(static_cast<int>((key >> nshift) & mask))], 1u);
    });
    __syncthreads();
    const Sel sel = threshold_of(hist, mhist, 1 << w, need, G, rank, ctl);
    if (G == 1) {
      above_local += sel.above;
      tie_local = sel.count;
    } else {
      uint32_t part = 0;
      for (int i = tid; i <= static_cast<int>(mask); i += kThreads)
        part += static_cast<uint32_t>(i) > sel.t ? hist[hist_index(i)] : 0u;
      tie_local = hist[hist_index(static_cast<int>(sel.t))];
      above_local += block_sum(part, ctl);
    }
    need -= sel.above;
    prefix = (prefix << w) | sel.t;
    shift = nshift;
    cnt = sel.count;
    more = cnt > cap && shift != 0;
  }

  const uint32_t k_above = static_cast<uint32_t>(k) - need;  // winners above the bin
  uint32_t win_base = 0, tie_base = 0;
  if (G > 1) {
    if (tid < G) {
      dsmem_st(map_rank(smem_addr(&ctl.xa[rank]), tid), above_local);
      dsmem_st(map_rank(smem_addr(&ctl.xt[rank]), tid), tie_local);
    }
    cluster_sync();
    for (int r = 0; r < rank; ++r) {
      win_base += ctl.xa[r];
      tie_base += ctl.xt[r];
    }
  }

  if (cnt <= cap) {
    const bool remote = G > 1 && rank != 0;
    const uint32_t ties_remote = G > 1 ? map_rank(smem_addr(buf), 0) : 0u;
    scatter_pass<F>(s, prefix, shift, out, k, win_base, tie_base, buf, ties_remote, remote, cap, m,
                    ctl);
    if (G > 1)
      cluster_sync();  // CTA 0 now holds every tie
    else
      __syncthreads();
    if (rank == 0)
      select_in_buffer<F>(buf, cnt, need, prefix, 32 + shift, L, out, k, k_above, m, hist, ctl);
  } else {
    // tie_base is this CTA's first position among the elements equal to prefix
    const uint32_t quota = tie_base >= need ? 0u : min(need - tie_base, tie_local);
    const uint32_t eq_slot0 = k_above + min(tie_base, need);
    emit_equal<F>(s, prefix, out, k, win_base, eq_slot0, quota, m, ctl);
  }
}

// ------------------------------------------------------------------ staged tier
//
// A row owned by one CTA whose aligned body holds at most kStagedQuads quads is
// copied whole into shared memory, starting at kernel start. One SM takes in data
// at a limited rate (about 25 bytes per clock, measured with plain and bulk loads
// alike), and filtering a row takes the SM about as long again in integer work; so
// the row must start arriving at once, and each part must be filtered as soon as it
// has landed:
//   - every thread first loads one quad of the sample: 16 runs of 512 bytes (one
//     per warp) spread evenly over the row, 2048 keys for 512 threads;
//   - the row is cut into chunks of kChunkQuads quads, one per thread, in passes of
//     kPassChunks chunks; each thread copies its own quad of each chunk to shared
//     memory with a 16-byte cp.async, one commit group per chunk. The first pass is
//     asked for before lambda is looked for, the second after (a thread that has
//     asked for much stalls until the memory system accepts its copies, and would
//     find lambda late). With the whole row staged (one CTA per SM) the second pass
//     has slots of its own; with half of it (two CTAs per SM) each thread copies
//     the second pass into its own first-pass slots once it has read them, and the
//     second half of the row is asked into L2 at kernel start;
//   - lambda is found from the sample while the chunks arrive;
//   - each thread flags its quad of each chunk that may hold a candidate (its
//     largest or smallest element against the threshold) once the chunk's group
//     has landed, then reads the flagged quads, about one in five, again for their
//     exact candidates; each thread reads back only what it copied itself, so no
//     barrier is needed;
//   - each warp reserves its candidates' slots once per pass and writes their keys
//     and positions into the candidate buffer; the candidate histogram is counted
//     from the buffer once the filter is done.
// For the raw and paged forms the copies cover the whole row stride and go out
// before the row's length has arrived; elements at or past it are ignored.
// Lambda comes from one round over the sample: the distance d = M - x in value of
// each sample element from the sample's largest one is binned by its fp32 exponent
// and the five bits after it (32 bins per power of two), in a window of 32 powers
// of two that ends at the sample's range. Distances in value, unlike in key space,
// do not jump where the scores change sign. If the bin holding the rs-th sample key
// holds more than kRefineCount sample keys (scores packed into a narrow band), a
// second round splits the window between the two sample ranks into 1024 equal key
// bins. Any lambda gives an exact result (the candidate count is verified); these
// only make the fast path likely. The candidate histogram and the selection are
// those of the fast tier (F2, F3). If the candidate count does not verify, the exact
// tier runs over the row.
#if TOPK_CTA_THREADS == 512
constexpr bool kHasStaged = true;
#else
constexpr bool kHasStaged = false;
#endif
constexpr int kChunkQuads = kThreads;                          // one quad per thread
constexpr int kPassChunks = 8;                                 // chunks of one pass
constexpr int kStagedChunks = 2 * kPassChunks;                 // chunks of a row at most
constexpr int32_t kStagedQuads = kStagedChunks * kChunkQuads;  // 8192 quads (32768 elements)
constexpr int kPtStaged = 512;                                 // page-table entries staged
constexpr uint32_t kRefineCount = 32;                          // sample keys in a bin: refine
constexpr int kLogSub = 5;                                     // bins per power of two: 2^kLogSub
constexpr int kDistShift = 23 - kLogSub;                       // fp32 bits below a log bin
// Shared memory of the staged tier (words): staging | sample histogram (1024 bins)
// | candidate histogram (2048 bins; also the second sample round's) | page table |
// candidate buffer. The staging area holds the whole row (kStagedChunks chunks: one
// CTA per SM) or half of it (kPassChunks chunks, two CTAs per SM: the second pass
// reuses the first pass's slots). Once the candidates are in the buffer, it holds
// the list of threshold-bin entries and the scratch histogram of the selection (or
// the exact tier's histogram).
template <bool kHalf>
__host__ __device__ constexpr int stage_words() { return (kHalf ? kPassChunks : kStagedChunks) * kChunkQuads * 4; }
template <bool kHalf>
__host__ __device__ constexpr int staged_fixed_words() { return stage_words<kHalf>() + kFastWords + kCandWords + kPtStaged; }
static_assert(kListWords + kHistWords + kMaxK <= stage_words<true>(),
              "list, scratch and output slots must fit the staging area");


// 128-bit read-only load issued where it stands (volatile: the compiler may not move
// it towards its use).
__device__ __forceinline__ uint4 ld_now(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t quad_elem(const uint4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// One candidate of the staged tier's filter: its key and position into the buffer at
// `slot` (if below cap); the candidate histogram is counted from the buffer afterwards.
__device__ __forceinline__ void staged_put_key(uint32_t bits, int32_t j, uint32_t slot, uint2* buf,
                                               uint32_t cap) {
  if (slot < cap) buf[slot] = make_uint2(order_key(bits), static_cast<uint32_t>(j));
}

// Candidate mask of quad v, quad q of the body whose first element is at row
// position j (bit c: element c is a candidate at a position below L).
template <bool kPos>
__device__ __forceinline__ uint32_t quad_cands(const uint4& v, int32_t q, int32_t nvec, int32_t j,
                                               int32_t L, uint32_t thr) {
  if (q >= nvec) return 0u;
  const int32_t left = L - j;  // elements of the quad below L
  const uint32_t lm = left >= 4 ? 0xFu : left <= 0 ? 0u : (1u << left) - 1u;
  return lm & (static_cast<uint32_t>(is_candidate<kPos>(v.x, thr)) |
               (static_cast<uint32_t>(is_candidate<kPos>(v.y, thr)) << 1) |
               (static_cast<uint32_t>(is_candidate<kPos>(v.z, thr)) << 2) |
               (static_cast<uint32_t>(is_candidate<kPos>(v.w, thr)) << 3));
}

// Asynchronous 16-byte copy global -> shared (both 16-byte aligned), L2 only.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_addr(smem_dst)), "l"(gsrc)
               : "memory");
}

// This thread's quads of chunks [c0, c0 + kPassChunks) of the body (vb, nvec quads)
// into slots [slot0, slot0 + kPassChunks) of the staging area, one commit group per
// chunk (empty for chunks past the body).
__device__ __forceinline__ void copy_pass(uint4* stage, int slot0, int c0, const uint4* vb,
                                          int32_t nvec) {
#pragma unroll
  for (int i = 0; i < kPassChunks; ++i) {
    const int32_t q = (c0 + i) * kChunkQuads + static_cast<int32_t>(threadIdx.x);
    if (q < nvec) cp_async16(stage + (slot0 + i) * kChunkQuads + threadIdx.x, vb + q);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
}

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// Waits until this thread's copy groups up to pass chunk i have landed, when kLater
// groups were committed after the pass's last chunk (i and kLater compile-time).
template <int kLater>
__device__ __forceinline__ void wait_pass_chunk(int i) {
  switch (i) {
    case 0: cp_async_wait_group<kLater + kPassChunks - 1>(); break;
    case 1: cp_async_wait_group<kLater + kPassChunks - 2>(); break;
    case 2: cp_async_wait_group<kLater + kPassChunks - 3>(); break;
    case 3: cp_async_wait_group<kLater + kPassChunks - 4>(); break;
    case 4: cp_async_wait_group<kLater + kPassChunks - 5>(); break;
    case 5: cp_async_wait_group<kLater + kPassChunks - 6>(); break;
    case 6: cp_async_wait_group<kLater + kPassChunks - 7>(); break;
    default: cp_async_wait_group<kLater>(); break;
  }
}
static_assert(kPassChunks == 8, "wait_pass_chunk spells out eight chunks");

// Whether quad v may hold a candidate: its largest element (signed compare, kPos) or
// its smallest (unsigned) against the filter threshold. Positions past the body or
// the row's length are not looked at here; the exact mask is taken afterwards.
template <bool kPos>
__device__ __forceinline__ bool quad_may(const uint4& v, uint32_t thr) {
  if constexpr (kPos) {
    const int32_t mx = max(max(static_cast<int32_t>(v.x), static_cast<int32_t>(v.y)),
                           max(static_cast<int32_t>(v.z), static_cast<int32_t>(v.w)));
    return mx >= static_cast<int32_t>(thr);
  } else {
    return min(min(v.x, v.y), min(v.z, v.w)) <= thr;
  }
}

// F2 on one pass of staged chunks (every thread), in two levels: this thread's quad
// of each chunk c0 + i (slot slot0 + i) is flagged if it may hold a candidate, once
// the chunk's copy group has landed (kLater groups were committed after the pass);
// then the flagged quads, about one in five, are read again for their exact
// candidates (positions below L), which go with this thread's edge element (when
// `edge`) to buf, as (key, position), at slots from one reservation per warp on
// ctl.cand_cnt.
template <bool kPos, int kLater>
__device__ __forceinline__ void filter_pass(const uint4* stage, int slot0, int c0, int32_t nvec,
                                            int32_t head, int32_t L, bool edge, int32_t ej,
                                            uint32_t ebits, uint32_t lambda, uint2* buf,
                                            uint32_t cap, Ctl& ctl) {
  const int tid = threadIdx.x;
  const uint32_t thr = kPos ? (lambda ^ 0x80000000u) : ~lambda;
  uint32_t fl = 0;  // bit i: this thread's quad of pass chunk i may hold a candidate
#pragma unroll
  for (int i = 0; i < kPassChunks; ++i) {
    wait_pass_chunk<kLater>(i);
    fl |= static_cast<uint32_t>(quad_may<kPos>(stage[(slot0 + i) * kChunkQuads + tid], thr)) << i;
  }
  // exact masks of the flagged quads: bits 4 i .. 4 i + 3 for pass chunk i
  uint32_t m = 0;
  while (fl != 0u) {
    const int i = __ffs(fl) - 1;
    fl &= fl - 1u;
    const int32_t q = (c0 + i) * kChunkQuads + tid;
    m |= quad_cands<kPos>(stage[(slot0 + i) * kChunkQuads + tid], q, nvec, head + 4 * q, L, thr)
         << (4 * i);
  }
  const bool ec = edge && is_candidate<kPos>(ebits, thr);
  uint32_t slot = warp_reserve(&ctl.cand_cnt, 0u, false,
                               static_cast<uint32_t>(__popc(m)) + (ec ? 1u : 0u));
  if (ec) staged_put_key(ebits, ej, slot++, buf, cap);
  while (m != 0u) {
    const int bit = __ffs(m) - 1;
    m &= m - 1u;
    const int i = bit >> 2, e = bit & 3;
    const int32_t q = (c0 + i) * kChunkQuads + tid;
    staged_put_key(quad_elem(stage[(slot0 + i) * kChunkQuads + tid], e), head + 4 * q + e, slot++,
                   buf, cap);
  }
}

// The second sample round of staged_lambda (every thread; the same sample quad v at
// row position j, `in` as there): 1024 equal key bins over [wlo, whi] (keys above
// it counted apart) in chist's region, which is cleared again afterwards. Returns
// lambda and sets *shift; when rs falls above the window (rounding), the first round's
// (wlo, shift1) stands. Kept out of line, as it runs only for scores packed into a
// narrow band.
__device__ __noinline__ uint32_t staged_refine(uint4 v, int32_t j, bool in, int32_t L, uint32_t rs,
                                               uint32_t rs_lo, uint32_t wlo, uint32_t whi,
                                               uint32_t shift1, uint32_t* chist, Ctl& ctl,
                                               uint32_t* shift) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int f = max(0, (32 - __clz(static_cast<int>(whi - wlo))) - kFastBits);
  uint32_t above = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (!(in && j + c < L)) continue;
    const uint32_t key = order_key(quad_elem(v, c));
    if (key > whi)
      ++above;
    else if (key >= wlo)
      atomicAdd(&chist[hist_index(static_cast<int>((key - wlo) >> f))], 1u);
  }
  above = __reduce_add_sync(kFull, above);
  if (lane == 0) ctl.wcnt[warp] = above;
  __syncthreads();  // (also: every thread has read the first round's bins)
  uint32_t na = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) na += ctl.wcnt[w];
  const bool go = rs > na, two = rs_lo > na;
  block_find2<kFastBins / kThreads>(chist, go ? rs - na : 0u, two ? rs_lo - na : 0u, two, ctl);
  __syncthreads();
  uint32_t lam = wlo, sh = shift1;
  if (go) {
    lam = wlo + (ctl.sel_t << f);
    const uint64_t top =
        static_cast<uint64_t>(wlo) + (static_cast<uint64_t>(ctl.sel2_t + 1u) << f) - 1u;
    const uint32_t hi = two ? static_cast<uint32_t>(min(top, static_cast<uint64_t>(whi))) : whi;
    const uint32_t gap = hi > lam ? hi - lam : 0u;
    sh = static_cast<uint32_t>(max(0, (32 - __clz(static_cast<int>(gap))) - (kCandBits - 1)));
  }
  for (int i = tid; i < kCandWords; i += kThreads) chist[i] = 0;
  __syncthreads();
  *shift = sh;
  return lam;
}

// Lambda from the sample (every thread of the CTA; thread t holds sample quad v,
// whose first element is at row position j, when `in`). shist is zero on entry;
// chist is zero on entry and on return. Returns lambda; *shift gets the
// candidate-histogram bin width exponent.
__device__ __forceinline__ uint32_t staged_lambda(const uint4& v, int32_t j, bool in, int32_t L,
                                                  uint32_t k, uint32_t* shist, uint32_t* chist,
                                                  Ctl& ctl, uint32_t* shift) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t key[4];
  bool ok[4];
  uint32_t mx = 0, mn = 0xFFFFFFFFu, cnt = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    key[c] = order_key(quad_elem(v, c));
    ok[c] = in && j + c < L;
    if (ok[c]) {
      mx = max(mx, key[c]);
      mn = min(mn, key[c]);
      ++cnt;
    }
  }
  mx = __reduce_max_sync(kFull, mx);
  mn = __reduce_min_sync(kFull, mn);
  cnt = __reduce_add_sync(kFull, cnt);
  if (lane == 0) {
    ctl.wmax[warp] = mx;
    ctl.wmin[warp] = mn;
    ctl.wcnt[warp] = cnt;
  }
  __syncthreads();
  // the CTA's values: lane l < kWarps reads warp l's, then a warp reduction
  const bool own = lane < kWarps;
  const uint32_t M = __reduce_max_sync(kFull, own ? ctl.wmax[lane] : 0u);
  const uint32_t Mn = __reduce_min_sync(kFull, own ? ctl.wmin[lane] : 0xFFFFFFFFu);
  const uint32_t ns = __reduce_add_sync(kFull, own ? ctl.wcnt[lane] : 0u);
  // first sample round: log bins of the distance in value from the largest sample element, in
  // the 32 powers of two below the sample's range (index 1023 - bin, so that larger
  // scores have higher indices); distances past the window share its end bins
  const float Mv = __uint_as_float(key_bits(M));
  const float range = Mv - __uint_as_float(key_bits(Mn));
  const bool usable = ns != 0 && isfinite(range);
  const int32_t base = static_cast<int32_t>(__float_as_uint(range) >> kDistShift) + 1 - (kFastBins - 1);
  if (usable) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (!ok[c]) continue;
      const float d = Mv - __uint_as_float(key_bits(key[c]));
      // NaN and infinite distances (non-finite scores) fall into the last bin
      const int32_t raw = isfinite(d) ? static_cast<int32_t>(__float_as_uint(d) >> kDistShift)
                                      : INT32_MAX - kFastBins;
      const int32_t bin = min(max(raw - base, 0), kFastBins - 1);
      atomicAdd(&shist[hist_index(kFastBins - 1 - bin)], 1u);
    }
  }
  __syncthreads();
  // the sample ranks: four standard deviations below the expected sample rank of the
  // row's k-th key (lambda's side) and three above (the candidate-histogram width)
  uint32_t rs = 0, rs_lo = 0;
  if (usable) {
    const float mean =
        fmaxf(__fdividef(static_cast<float>(k) * static_cast<float>(ns), static_cast<float>(L)), 1.0f);
    const float sd = mean * rsqrtf(mean);
    rs = min(static_cast<uint32_t>(ceilf(mean + 4.0f * sd)) + 2u, ns);
    const float lo = floorf(mean - 3.0f * sd);
    rs_lo = min(lo < 1.0f ? 1u : static_cast<uint32_t>(lo), rs);
  }
  block_find2<kFastBins / kThreads>(shist, rs, rs_lo, usable, ctl);
  __syncthreads();
  // every thread: lambda and the candidate-histogram bin width from the bins found
  if (!usable) {
    *shift = 32 - kCandBits;
    return 0u;
  }
  // the distances at a window bin's edges (bins 0 and kFastBins - 1 are open)
  const int32_t bs = kFastBins - 1 - static_cast<int32_t>(ctl.sel_t);
  const int32_t bl = kFastBins - 1 - static_cast<int32_t>(ctl.sel2_t);
  const int32_t ehi = bs + base + 1, elo = bl + base;
  const float dhi = bs >= kFastBins - 1 ? __uint_as_float(0x7F800000u)
                    : ehi <= 0          ? 0.0f
                                        : __uint_as_float((static_cast<uint32_t>(ehi) << kDistShift) - 1u);
  const float dlo = bl <= 0 || elo <= 0 ? 0.0f
                                        : __uint_as_float(static_cast<uint32_t>(elo) << kDistShift);
  // keys of M - d, lambda rounded down and lambda_hi up by a few key units
  const float xlo = Mv - dhi, xhi = Mv - dlo;
  const uint32_t klo = isnan(xlo) ? 0u : order_key(__float_as_uint(xlo));
  const uint32_t khi = isnan(xhi) ? M : order_key(__float_as_uint(xhi));
  const uint32_t lam = klo > 2u ? klo - 2u : 0u;
  const uint32_t lam_hi = min(khi + 2u < khi ? khi : khi + 2u, M);
  const uint32_t gap = lam_hi > lam ? lam_hi - lam : 0u;
  const uint32_t sh =
      static_cast<uint32_t>(max(0, (32 - __clz(static_cast<int>(gap))) - (kCandBits - 1)));
  if (__builtin_expect(ctl.sel_count > kRefineCount && lam_hi > lam, 0))
    return staged_refine(v, j, in, L, rs, rs_lo, lam, lam_hi, sh, chist, ctl, shift);
  *shift = sh;
  return lam;
}

// One row of problem p on the staged tier (one CTA, no cluster).
template <int F>
__device__ __forceinline__ void staged_row(const Params& p, int row, uint32_t* dyn, Ctl& ctl) {
  constexpr bool kHalf = (F & kHalfStage) != 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint4* stage = reinterpret_cast<uint4*>(dyn);
  uint32_t* shist = dyn + stage_words<kHalf>();   // sample histogram (kFastBins, padded)
  uint32_t* chist = shist + kFastWords;            // candidate histogram (kCandBins, padded)
  int32_t* pt_smem = reinterpret_cast<int32_t*>(chist + kCandWords);
  uint2* buf = reinterpret_cast<uint2*>(pt_smem + kPtStaged);
  const uint32_t cap = static_cast<uint32_t>(p.tie_cap);

  allow_next_grid();
  for (int i = tid; i < kFastWords + kCandWords; i += kThreads) shist[i] = 0;
  if (tid == 0) {
    ctl.win_cnt = 0;
    ctl.tie_cnt = 0;
    ctl.out_cnt = 0;
    ctl.cand_cnt = 0;
  }
  __syncthreads();  // cleared memory before any use
  wait_prior_grids();

  const int32_t seq = p.seq_lens[row];
  int32_t start = 0;
  if constexpr (form_of(F) == kRagged || form_of(F) == kWindow) start = p.row_starts[row];

  // the row's data and the length its layout covers: raw and paged rows lay out the
  // whole stride at once; ragged and window rows wait for their start and length
  const float* rowp;
  int32_t span;
  if constexpr (form_of(F) == kRagged) {
    rowp = p.scores + start;
    span = max(seq, 0);
  } else if constexpr (form_of(F) == kWindow) {
    const int64_t hi = min(static_cast<int64_t>(max(seq, 0)), p.row_stride);
    const int64_t lo = min(static_cast<int64_t>(max(start, 0)), hi);
    rowp = p.scores + static_cast<int64_t>(row) * p.row_stride + lo;
    span = static_cast<int32_t>(hi - lo);
  } else {
    rowp = p.scores + static_cast<int64_t>(row) * p.row_stride;
    span = static_cast<int32_t>(p.row_stride);
  }
  const Slice lay = make_slice(rowp, span, 0, 1);
  const uint4* vb = lay.vec;  // the aligned body: nvec quads from row position head
  const int32_t nvec = lay.nvec, head = lay.n_head;
  const bool fits = nvec <= kStagedQuads;
  // the sample first (run `warp` of 16 spread over the body), then the early chunks
  const int32_t qs = static_cast<int32_t>((static_cast<int64_t>(nvec) * warp) / kWarps) + lane;
  const bool sin = fits && qs < nvec;
  const uint4 sv = sin ? ld_now(vb + qs) : make_uint4(0, 0, 0, 0);
  if (fits) copy_pass(stage, 0, 0, vb, nvec);
  if constexpr (kHalf) {  // the second half towards L2, from the last warp
    const int32_t q1 = min(nvec, kPassChunks * kChunkQuads);
    const uint32_t bytes = fits ? 16u * static_cast<uint32_t>(nvec - q1) : 0u;
    const uint32_t piece = static_cast<uint32_t>(kPrefetchBytes);
    const uint32_t off = static_cast<uint32_t>(tid - (kThreads - 32)) * piece;
    if (tid >= kThreads - 32 && off < bytes)
      prefetch_l2(reinterpret_cast<const char*>(vb + q1) + off, min(piece, bytes - off));
  }
  // paged: the page table of the span's pages (at most the table's row stride)
  int32_t pages = 0;
  if constexpr (form_of(F) == kPaged) {
    const int64_t up = static_cast<int64_t>(span) + p.page_size - 1;
    const int64_t np = min(p.page_shift >= 0 ? up >> p.page_shift : up / p.page_size, p.pt_stride);
    if (np <= kPtStaged) {
      pages = static_cast<int32_t>(np);
      const int32_t* pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
      for (int32_t i = tid; i < pages; i += kThreads) cp_async4(pt_smem + i, pt_row + i);
    }
  }

  OutMap m;
  m.pt_row = nullptr;
  m.pt_smem = nullptr;
  m.pt_n = 0;
  m.ps = p.page_size;
  m.ps_shift = p.page_shift;
  m.rstart = 0;
  m.values = opts_of(F) && p.values != nullptr ? p.values + static_cast<int64_t>(row) * p.k
                                               : nullptr;
  m.staged = opts_of(F) && p.staged != nullptr ? p.staged + static_cast<int64_t>(row) * p.k
                                               : nullptr;
  int32_t L;
  if constexpr (form_of(F) == kRagged) {
    m.rstart = start;
    L = span;
  } else if constexpr (form_of(F) == kWindow) {
    m.rstart = static_cast<int32_t>(rowp - (p.scores + static_cast<int64_t>(row) * p.row_stride));
    L = span;
  } else {
    L = static_cast<int32_t>(min(static_cast<int64_t>(max(seq, 0)), p.row_stride));
  }
  if constexpr (form_of(F) == kPaged) {
    m.pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
    const int64_t up = static_cast<int64_t>(L) + p.page_size - 1;
    const int64_t np = p.page_shift >= 0 ? up >> p.page_shift : up / p.page_size;
    m.pt_n = static_cast<int32_t>(min(np, p.pt_stride));
    if (np > p.pt_stride && tid == 0) guard_hit();
  }
  const int32_t k = p.k;
  int32_t* out = p.out + static_cast<int64_t>(row) * k;

  if (__builtin_expect(!fits, 0)) {  // a ragged or window row longer than its hint promised
    cp_async_wait_all();
    for (int i = tid; i < kHistWords; i += kThreads) dyn[i] = 0;
    __syncthreads();
    exact_tier<F>(make_slice(rowp, L, 0, 1), L, k, out, m, pages, pt_smem, 1, 0, dyn, nullptr, buf,
                  cap, ctl);
    return;
  }

  if (__builtin_expect(L <= k, 0)) {  // every position is selected; the rest of the row is -1
    const bool keys = opts_of(F) && (m.values != nullptr || m.staged != nullptr);
    for (int32_t i = tid; i < k; i += kThreads) {
      if (i < L)
        emit<F>(out, k, static_cast<uint32_t>(i), m, i, keys ? order_key(__float_as_uint(rowp[i])) : 0u);
      else
        emit_pad<F>(out, static_cast<uint32_t>(i), m);
    }
    cp_async_wait_all();  // nothing may still be copying into shared memory at exit
    return;
  }

  // this thread's unaligned head or tail element, if any: positions [0, head) and
  // [head + 4 nvec, L)
  int32_t ej = 0;
  bool edge = false;
  {
    const int32_t tail0 = head + 4 * nvec;
    if (tid < head && tid < L) {
      ej = tid;
      edge = true;
    } else if (tid >= 4 && tid - 4 < L - tail0) {
      ej = tail0 + (tid - 4);
      edge = true;
    }
  }
  const uint32_t ebits = edge ? __float_as_uint(rowp[ej]) : 0u;

  // ---- lambda from the sample (rows that fit the buffer: every element)
  uint32_t lambda = 0, shift2 = 32 - kCandBits;
  if (static_cast<uint32_t>(L) > cap)
    lambda = staged_lambda(sv, head + 4 * qs, sin, L, static_cast<uint32_t>(k), shist, chist, ctl,
                           &shift2);

  // ---- the second pass's copies, and the filter of each chunk as it lands
  const bool pos = lambda >= 0x80000000u;
  if constexpr (!kHalf) {  // the whole row in the staging area
    copy_pass(stage, kPassChunks, kPassChunks, vb, nvec);
    if (pos) {
      filter_pass<true, kPassChunks>(stage, 0, 0, nvec, head, L, edge, ej, ebits, lambda, buf, cap, ctl);
      filter_pass<true, 0>(stage, kPassChunks, kPassChunks, nvec, head, L, false, 0, 0u, lambda, buf,
                           cap, ctl);
    } else {
      filter_pass<false, kPassChunks>(stage, 0, 0, nvec, head, L, edge, ej, ebits, lambda, buf, cap, ctl);
      filter_pass<false, 0>(stage, kPassChunks, kPassChunks, nvec, head, L, false, 0, 0u, lambda, buf,
                            cap, ctl);
    }
  } else {  // half the row: the second pass into this thread's first-pass slots
    if (pos)
      filter_pass<true, 0>(stage, 0, 0, nvec, head, L, edge, ej, ebits, lambda, buf, cap, ctl);
    else
      filter_pass<false, 0>(stage, 0, 0, nvec, head, L, edge, ej, ebits, lambda, buf, cap, ctl);
    copy_pass(stage, 0, kPassChunks, vb, nvec);
    if (pos)
      filter_pass<true, 0>(stage, 0, kPassChunks, nvec, head, L, false, 0, 0u, lambda, buf, cap, ctl);
    else
      filter_pass<false, 0>(stage, 0, kPassChunks, nvec, head, L, false, 0, 0u, lambda, buf, cap, ctl);
  }
  cp_async_wait_all();  // the page table
  if constexpr (form_of(F) == kPaged) {
    if (pages > 0) m.pt_smem = pt_smem;  // visible to all threads after the barrier below
  }
  __syncthreads();
  const uint32_t n_cand = ctl.cand_cnt;
  uint2* list = reinterpret_cast<uint2*>(dyn);  // the staging area is free from here on
  uint32_t* scratch = dyn + kListWords;
  // the candidate histogram, from the buffer
  if (n_cand >= static_cast<uint32_t>(k) && n_cand <= cap)
    count_candidates(buf, n_cand, lambda, shift2, chist);
  if (__builtin_expect(n_cand >= static_cast<uint32_t>(k) && n_cand <= cap, 1)) {

    select_candidates<F>(buf, n_cand, static_cast<uint32_t>(k), chist, lambda, shift2, list, scratch,
                         reinterpret_cast<int32_t*>(scratch + kHistWords), L, out, m, ctl);
    return;
  }
  // too few (lambda above the k-th key) or too many candidates: exact tier
  for (int i = tid; i < kHistWords; i += kThreads) dyn[i] = 0;
  __syncthreads();
  exact_tier<F>(make_slice(rowp, L, 0, 1), L, k, out, m, pages, pt_smem, 1, 0, dyn, nullptr, buf,
                cap, ctl);
}

// One row of problem p, this CTA's slice of it (CTA `rank` of a cluster of G).
template <int F>
__device__ __forceinline__ void row_body(const Params& p, int row, int G, int rank, uint32_t* dyn,
                                         Ctl& ctl) {
  const int tid = threadIdx.x;

  // shared memory: histogram | list | page table | cluster-sum histogram (G > 1) |
  // candidate/tie buffer
  uint32_t* hist = dyn;
  uint2* list = reinterpret_cast<uint2*>(dyn + kHistWords);
  int32_t* pt_smem = reinterpret_cast<int32_t*>(dyn + kHistWords + kListWords);
  uint32_t* mhist = dyn + kHistWords + kListWords + kPtCap;
  uint2* buf =
      reinterpret_cast<uint2*>(dyn + (G > 1 ? 2 : 1) * kHistWords + kListWords + kPtCap);
  const uint32_t cap = static_cast<uint32_t>(p.tie_cap);

  allow_next_grid();
  // independent of the row: clear the histograms and counters (overlapping the
  // previous kernel's tail), then wait for it before touching any buffer
  for (int i = tid; i < kHistWords; i += kThreads) hist[i] = 0;
  if (G > 1 && rank == 0)
    for (int i = tid; i < kHistWords; i += kThreads) mhist[i] = 0;
  if (tid == 0) {
    ctl.win_cnt = 0;
    ctl.tie_cnt = 0;
    ctl.out_cnt = 0;
    ctl.cand_cnt = 0;
    ctl.ns = 0;
    ctl.lambda = 0;
    ctl.lambda_shift = 0;
  }

  wait_prior_grids();

  // the row's length (and start) first: everything waits for them
  const int32_t seq = p.seq_lens[row];
  int32_t start = 0;  // ragged: row offset; window: window start
  if constexpr (form_of(F) == kRagged || form_of(F) == kWindow) start = p.row_starts[row];
  // raw, paged: the row's start does not depend on its length, so the sample is
  // loaded (over the whole row stride; elements at or past the length are ignored
  // later) while the length is still on its way
  Sample sm;
  bool sample_loaded = false;
  if constexpr (form_of(F) == kRaw || form_of(F) == kPaged) {
    if (p.use_filter && p.row_stride > static_cast<int64_t>(p.tie_cap) && p.row_stride <= INT32_MAX) {
      const Slice whole = make_slice(p.scores + static_cast<int64_t>(row) * p.row_stride,
                                     static_cast<int32_t>(p.row_stride), rank, G);
      load_sample(whole, sm);
      // right behind the sample: the whole stride towards L2 (from the last warp)
      prefetch_slice(whole, kThreads - 32);
      sample_loaded = true;
    }
  }

  OutMap m;
  m.pt_row = nullptr;
  m.pt_smem = nullptr;
  m.pt_n = 0;
  m.ps = p.page_size;
  m.ps_shift = p.page_shift;
  m.rstart = 0;
  m.values = opts_of(F) && p.values != nullptr ? p.values + static_cast<int64_t>(row) * p.k
                                               : nullptr;
  m.staged = opts_of(F) && p.staged != nullptr ? p.staged + static_cast<int64_t>(row) * p.k
                                               : nullptr;
  const float* rowp;
  int32_t L;
  if constexpr (form_of(F) == kRagged) {
    m.rstart = start;
    rowp = p.scores + m.rstart;
    L = max(seq, 0);
  } else if constexpr (form_of(F) == kWindow) {  // columns [lo, hi) of the row, clamped to it
    const int64_t hi = min(static_cast<int64_t>(max(seq, 0)), p.row_stride);
    const int64_t lo = min(static_cast<int64_t>(max(start, 0)), hi);
    m.rstart = static_cast<int32_t>(lo);
    rowp = p.scores + static_cast<int64_t>(row) * p.row_stride + lo;
    L = static_cast<int32_t>(hi - lo);
  } else {
    rowp = p.scores + static_cast<int64_t>(row) * p.row_stride;
    L = static_cast<int32_t>(min(static_cast<int64_t>(max(seq, 0)), p.row_stride));
  }
  if constexpr (form_of(F) == kPaged) {
    m.pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
    // the row's pages; a table row narrower than that is read only up to its stride
    const int64_t up = static_cast<int64_t>(L) + p.page_size - 1;
    const int64_t np = p.page_shift >= 0 ? up >> p.page_shift : up / p.page_size;
    m.pt_n = static_cast<int32_t>(min(np, p.pt_stride));
    if (np > p.pt_stride && rank == 0 && tid == 0) guard_hit();
  }
  const int32_t k = p.k;
  int32_t* out = p.out + static_cast<int64_t>(row) * k;

  if (L <= k) {  // every position is selected; the rest of the row is -1
    const int32_t s0 = static_cast<int32_t>(static_cast<int64_t>(k) * rank / G);
    const int32_t s1 = static_cast<int32_t>(static_cast<int64_t>(k) * (rank + 1) / G);
    const bool keys = opts_of(F) && (m.values != nullptr || m.staged != nullptr);
    for (int32_t i = s0 + tid; i < s1; i += kThreads) {
      if (i < L)
        emit<F>(out, k, static_cast<uint32_t>(i), m, i,
                keys ? order_key(__float_as_uint(rowp[i])) : 0u);
      else
        emit_pad<F>(out, static_cast<uint32_t>(i), m);
    }
    return;
  }

  const Slice s = make_slice(rowp, L, rank, G);
  const bool sampled = p.use_filter && static_cast<uint32_t>(L) > cap;
  if (sampled && !sample_loaded) load_sample(s, sm);
  // paged: CTA 0, which writes the fast tier's output, copies the row's page table
  // to shared memory asynchronously (waited for after the sample); the other CTAs
  // of a cluster, and rows of more than kPtCap pages, read it from global memory
  int32_t pages = 0;
  if constexpr (form_of(F) == kPaged) {
    if (rank == 0 && m.pt_n <= kPtCap) {
      pages = m.pt_n;
      for (int32_t i = tid; i < pages; i += kThreads) cp_async4(pt_smem + i, m.pt_row + i);
    }
  }
  // pull the whole slice towards L2; every pass below then reads L2. A sampled row
  // does this once its sample has arrived (inside sample_lambda), so that the
  // sample loads do not queue behind the bulk traffic of every row.
  if (!sampled) prefetch_slice(s);
  if (G > 1)
    cluster_sync();  // all CTAs running; CTA 0's histograms and counters cleared
  else
    __syncthreads();

  // ---------------- fast tier
  uint32_t lam_x = 0, shift_x = 0;  // lambda and its candidate-bin width, kept for the exact tier
  bool overflow = false;            // the filter found more candidates than the buffer holds
  if (p.use_filter) {
    uint32_t shift2 = 32 - kCandBits;  // rows that skip the sample: the top key bits
    // rows split over a cluster (the long rows of the adversarial workloads) let the
    // sample predict an overflowing filter; single-CTA rows measured slower with the check
    constexpr bool kPredict = (F & kSingle) == 0;
    const uint32_t lambda =
        sampled ? sample_lambda(sm, s, sample_loaded, L, static_cast<uint32_t>(k), G, rank, hist,
                                mhist, ctl, &shift2, cap, kPredict)
                : 0u;
    lam_x = lambda;
    shift_x = shift2;
    if (!(kPredict && sampled && ctl.skip_fast != 0u)) {  // else the exact tier at once
      if constexpr (form_of(F) == kPaged) {
        if (pages > 0) {
          cp_async_wait_all();
          m.pt_smem = pt_smem;  // visible to all threads after the next barrier
        }
      }
      uint32_t n_cand;
      uint32_t* chist = hist + kHC;
      if (G == 1) {
        constexpr bool kKeys = (F & kKeysInFilter) != 0;
        if (lambda >= 0x80000000u)
          filter_positions<true, kKeys>(s, lambda, buf, cap, ctl);
        else
          filter_positions<false, kKeys>(s, lambda, buf, cap, ctl);
        __syncthreads();
        n_cand = ctl.cand_cnt;
        if (!kKeys && n_cand >= static_cast<uint32_t>(k) && n_cand <= cap)
          fill_candidates(rowp, buf, n_cand, lambda, shift2, chist, ctl);
        if (kKeys && n_cand >= static_cast<uint32_t>(k) && n_cand <= cap)
          count_candidates(buf, n_cand, lambda, shift2, chist);

      } else {
        const bool remote = rank != 0;
        const uint32_t buf_remote = map_rank(smem_addr(buf), 0);
        const uint32_t cnt_remote = map_rank(smem_addr(&ctl.cand_cnt), 0);
        if (lambda >= 0x80000000u)
          filter_candidates<true>(s, lambda, buf, buf_remote, cnt_remote, remote, cap, ctl);
        else
          filter_candidates<false>(s, lambda, buf, buf_remote, cnt_remote, remote, cap, ctl);
        cluster_sync();  // every candidate is in CTA 0's buffer; the counter is final
        if (rank == 0 && tid < G) dsmem_st(map_rank(smem_addr(&ctl.n_cand), tid), ctl.cand_cnt);
        cluster_sync();
        n_cand = ctl.n_cand;
        if (rank == 0 && n_cand >= static_cast<uint32_t>(k) && n_cand <= cap)
          count_candidates(buf, n_cand, lambda, shift2, chist);

      }
      overflow = n_cand > cap;
      if (__builtin_expect(n_cand >= static_cast<uint32_t>(k) && n_cand <= cap, 1)) {
        if (rank == 0)
          select_candidates<F>(buf, n_cand, static_cast<uint32_t>(k), chist, lambda, shift2, list,
                               hist, reinterpret_cast<int32_t*>(hist), L, out, m, ctl);
        return;
      }
    }
    // too few (lambda above the k-th key) or too many candidates, or too many expected:
    // exact tier
    for (int i = tid; i < kHistWords; i += kThreads) hist[i] = 0;
    if (G > 1) {
      if (rank == 0)
        for (int i = tid; i < kHistWords; i += kThreads) mhist[i] = 0;
      cluster_sync();
    } else {
      __syncthreads();
    }
  }

  // ---------------- exact tier (hist and, for CTA 0, mhist are zero here); a row whose
  // sample predicted an overflowing filter starts from the sample's window, and a
  // single-CTA row whose filter overflowed from the bits that the ends of its candidate
  // bins' span, [lambda, lambda + 2^(shift + kCandBits - 1)), share
  int x_start = 32;
  uint32_t start_prefix = 0;
  if constexpr ((F & kSingle) == 0) {
    if (p.use_filter && static_cast<uint32_t>(L) > cap && ctl.skip_fast != 0u) {
      x_start = static_cast<int>(ctl.ex_shift);
      start_prefix = x_start < 32 ? ctl.lambda >> x_start : 0u;
    }
  } else {
    if (overflow) {
      const uint64_t end = static_cast<uint64_t>(lam_x) + (1ull << (shift_x + kCandBits - 1)) - 1;
      const uint32_t hi = end > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(end);
      x_start = 32 - __clz(lam_x ^ hi);
      start_prefix = x_start < 32 ? lam_x >> x_start : 0u;
    }
  }
  exact_tier<F>(s, L, k, out, m, pages, pt_smem, G, rank, hist, mhist, buf, cap, ctl, x_start,
                start_prefix);
}

// ------------------------------------------------------------------ chip-wide split
//
// Small batches of long rows: each row is split over split_s CTAs anywhere on the
// chip (not one cluster), in two kernels. The filter kernel's CTAs each take the
// same sampled threshold of the whole row and store their slice's candidates in the
// workspace; the select kernel (one CTA per row, after the filter kernel) gathers
// them and selects. A row whose candidates do not fit (a CTA's share over
// split_cap, or the row's over gather_cap) or fall short of k takes the exact tier
// on the select CTA.

// The row's data, valid length and output map (page table not staged).
template <int F>
__device__ __forceinline__ void row_view(const Params& p, int row, int32_t seq, int32_t start,
                                         const float** rowp, int32_t* L, OutMap* m) {
  m->pt_row = nullptr;
  m->pt_smem = nullptr;
  m->pt_n = 0;
  m->ps = p.page_size;
  m->ps_shift = p.page_shift;
  m->rstart = 0;
  m->values = nullptr;
  m->staged = nullptr;
  if constexpr (form_of(F) == kRagged) {
    m->rstart = start;
    *rowp = p.scores + start;
    *L = max(seq, 0);
  } else if constexpr (form_of(F) == kWindow) {
    const int64_t hi = min(static_cast<int64_t>(max(seq, 0)), p.row_stride);
    const int64_t lo = min(static_cast<int64_t>(max(start, 0)), hi);
    m->rstart = static_cast<int32_t>(lo);
    *rowp = p.scores + static_cast<int64_t>(row) * p.row_stride + lo;
    *L = static_cast<int32_t>(hi - lo);
  } else {
    *rowp = p.scores + static_cast<int64_t>(row) * p.row_stride;
    *L = static_cast<int32_t>(min(static_cast<int64_t>(max(seq, 0)), p.row_stride));
  }
  if constexpr (form_of(F) == kPaged) {
    m->pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
    const int64_t up = static_cast<int64_t>(*L) + p.page_size - 1;
    const int64_t np = p.page_shift >= 0 ? up >> p.page_shift : up / p.page_size;
    m->pt_n = static_cast<int32_t>(min(np, p.pt_stride));
  }
}

// Filter CTA `part` (of p.split_s) of row `row`. Shared memory: histogram | buffer of
// split_cap candidates.
template <int F>
__device__ __forceinline__ void split_filter_part(const Params& p, int row, int part, uint32_t* dyn,
                                                  Ctl& ctl) {
  const int tid = threadIdx.x;
  const int S = p.split_s;
  uint32_t* hist = dyn;
  uint2* buf = reinterpret_cast<uint2*>(dyn + kHistWords);
  const uint32_t cap = static_cast<uint32_t>(p.split_cap);
  allow_next_grid();
  for (int i = tid; i < kHistWords; i += kThreads) hist[i] = 0;
  if (tid == 0) {
    ctl.cand_cnt = 0;
    ctl.ns = 0;
    ctl.lambda = 0;
    ctl.lambda_shift = 0;
  }
  wait_prior_grids();  // the workspace is free once the previous launch has ended
  const int32_t seq = p.seq_lens[row];
  int32_t start = 0;
  if constexpr (form_of(F) == kRagged || form_of(F) == kWindow) start = p.row_starts[row];
  // raw, paged: the sample of the whole stride while the length is on its way
  // a sample four times the streaming tier's (8192 keys): the threshold lies
  // closer to the k-th key, so the select CTA gathers fewer candidates
  SampleT<4 * kSampleQuads> sm;
  bool sample_loaded = false;
  if constexpr (form_of(F) == kRaw || form_of(F) == kPaged) {
    if (p.row_stride > static_cast<int64_t>(p.gather_cap) && p.row_stride <= INT32_MAX) {
      load_sample(make_slice(p.scores + static_cast<int64_t>(row) * p.row_stride,
                             static_cast<int32_t>(p.row_stride), 0, 1),
                  sm);
      sample_loaded = true;
    }
  }
  const float* rowp;
  int32_t L;
  OutMap m;
  row_view<F>(p, row, seq, start, &rowp, &L, &m);
  const int32_t k = p.k;
  uint2* hdr = reinterpret_cast<uint2*>(p.split_ws);
  int32_t* counts =
      reinterpret_cast<int32_t*>(static_cast<char*>(p.split_ws) + split_counts_offset(p.batch));
  uint2* entries =
      reinterpret_cast<uint2*>(static_cast<char*>(p.split_ws) + split_entries_offset(p.batch, S));
  const int64_t cell = static_cast<int64_t>(row) * S + part;
  if (L <= k) {  // the select CTA writes such rows alone
    if (tid == 0) counts[cell] = 0;
    return;
  }
  const Slice s = make_slice(rowp, L, part, S);
  // rows that fit the select CTA's buffer skip the sample: every element is a candidate
  const bool sampled = static_cast<uint32_t>(L) > static_cast<uint32_t>(p.gather_cap);
  if (sampled && !sample_loaded) load_sample(make_slice(rowp, L, 0, 1), sm);
  prefetch_slice(s, kThreads - 32);
  __syncthreads();  // the cleared histogram and counters
  uint32_t shift2 = 32 - kCandBits;
  const uint32_t lambda =
      sampled ? sample_lambda(sm, s, true, L, static_cast<uint32_t>(k), 1, 0, hist, nullptr, ctl, &shift2)
              : 0u;
  if (lambda >= 0x80000000u)
    filter_positions<true, true>(s, lambda, buf, cap, ctl);
  else
    filter_positions<false, true>(s, lambda, buf, cap, ctl);
  __syncthreads();
  const uint32_t n = ctl.cand_cnt;
  const uint32_t stored = min(n, cap);
  uint2* dst = entries + cell * cap;
  for (uint32_t i = static_cast<uint32_t>(tid); i < stored; i += kThreads) dst[i] = buf[i];
  if (tid == 0) {
    counts[cell] = static_cast<int32_t>(min(n, static_cast<uint32_t>(INT32_MAX)));
    if (part == 0) hdr[row] = make_uint2(lambda, shift2);
  }
}

// The select cluster of row `row` (G CTAs, this one `rank`): CTA 0 gathers the filter
// CTAs' candidates (and their histogram) and selects, the others end; a row whose
// candidates did not fit, or fell short of k, runs the exact tier on the whole cluster
// (every CTA reads the same counts, so all take the same branch). Shared memory as
// row_body's for a cluster of G, with a buffer of gather_cap candidates.
template <int F>
__device__ __forceinline__ void split_select_row(const Params& p, int row, int G, int rank,
                                                 uint32_t* dyn, Ctl& ctl) {
  const int tid = threadIdx.x;
  const int S = p.split_s;
  uint32_t* hist = dyn;
  uint2* list = reinterpret_cast<uint2*>(dyn + kHistWords);
  int32_t* pt_smem = reinterpret_cast<int32_t*>(dyn + kHistWords + kListWords);
  uint32_t* mhist = dyn + kHistWords + kListWords + kPtCap;
  uint2* buf = reinterpret_cast<uint2*>(dyn + (G > 1 ? 2 : 1) * kHistWords + kListWords + kPtCap);
  const uint32_t gcap = static_cast<uint32_t>(p.gather_cap);
  allow_next_grid();
  for (int i = tid; i < kHistWords; i += kThreads) hist[i] = 0;
  if (G > 1 && rank == 0)
    for (int i = tid; i < kHistWords; i += kThreads) mhist[i] = 0;
  if (tid == 0) {
    ctl.win_cnt = 0;
    ctl.tie_cnt = 0;
    ctl.out_cnt = 0;
    ctl.cand_cnt = 0;
  }
  wait_prior_grids();  // the filter kernel's candidates (and whatever the inputs wait for)
  // the parts' counts and the row's threshold, read together with the row's length
  // (meaningless for rows of at most k elements, which do not use them)
  const uint2* hdr = reinterpret_cast<const uint2*>(p.split_ws);
  const int32_t* counts = reinterpret_cast<const int32_t*>(static_cast<const char*>(p.split_ws) +
                                                           split_counts_offset(p.batch));
  const int32_t c = tid < S ? counts[static_cast<int64_t>(row) * S + tid] : 0;
  const uint2 lh = hdr[row];
  const int32_t seq = p.seq_lens[row];
  int32_t start = 0;
  if constexpr (form_of(F) == kRagged || form_of(F) == kWindow) start = p.row_starts[row];
  const float* rowp;
  int32_t L;
  OutMap m;
  row_view<F>(p, row, seq, start, &rowp, &L, &m);
  const int32_t k = p.k;
  int32_t* out = p.out + static_cast<int64_t>(row) * k;
  if constexpr (form_of(F) == kPaged) {
    const int64_t up = static_cast<int64_t>(L) + p.page_size - 1;
    if ((p.page_shift >= 0 ? up >> p.page_shift : up / p.page_size) > p.pt_stride && tid == 0 &&
        rank == 0)
      guard_hit();
  }
  // CTA 0, which writes the selection, stages the page table
  int32_t pages = 0;
  if constexpr (form_of(F) == kPaged) {
    if (rank == 0 && m.pt_n <= kPtCap) {
      pages = m.pt_n;
      for (int32_t i = tid; i < pages; i += kThreads) cp_async4(pt_smem + i, m.pt_row + i);
    }
  }
  if (L <= k) {  // each CTA writes its share of the slots
    cp_async_wait_all();
    __syncthreads();
    if (pages > 0) m.pt_smem = pt_smem;
    const int32_t s0 = static_cast<int32_t>(static_cast<int64_t>(k) * rank / G);
    const int32_t s1 = static_cast<int32_t>(static_cast<int64_t>(k) * (rank + 1) / G);
    for (int32_t i = s0 + tid; i < s1; i += kThreads) {
      if (i < L)
        emit<F>(out, k, static_cast<uint32_t>(i), m, i, 0u);
      else
        emit_pad<F>(out, static_cast<uint32_t>(i), m);
    }
    return;
  }
  const uint2* entries = reinterpret_cast<const uint2*>(static_cast<const char*>(p.split_ws) +
                                                        split_entries_offset(p.batch, S));
  const uint32_t scap = static_cast<uint32_t>(p.split_cap);
  // the parts' counts: an exclusive scan over the first S threads (S <= kThreads)
  uint32_t total = 0;
  const uint32_t off = block_excl_scan(static_cast<uint32_t>(c), ctl, &total);
  const bool over = __syncthreads_or(static_cast<uint32_t>(c) > scap) != 0;
  if (__builtin_expect(over || total < static_cast<uint32_t>(k) || total > gcap, 0)) {
    // exact tier over the whole row on the cluster (hist and, for CTA 0, mhist are zero)
    if (G > 1)
      cluster_sync();  // every CTA running, its histograms cleared
    else
      __syncthreads();
    // too many candidates: the k-th key is at or above lambda and most likely within the
    // candidate bins' span, [lambda, lambda + 2^(shift + kCandBits - 1)), so the exact
    // tier starts from the bits that this span's ends share
    int x_start = 32;
    uint32_t x_prefix = 0;
    if (over || total > gcap) {
      const uint64_t end = static_cast<uint64_t>(lh.x) + (1ull << (lh.y + kCandBits - 1)) - 1;
      const uint32_t hi = end > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(end);
      x_start = 32 - __clz(lh.x ^ hi);
      x_prefix = x_start < 32 ? lh.x >> x_start : 0u;
    }
    exact_tier<F>(make_slice(rowp, L, rank, G), L, k, out, m, pages, pt_smem, G, rank, hist, mhist,
                  buf, min(gcap, static_cast<uint32_t>(kTieCapMax)), ctl, x_start, x_prefix);
    return;
  }
  if (rank != 0) return;  // CTA 0 selects
  int32_t* part_off = reinterpret_cast<int32_t*>(list);  // S + 1 offsets, then the scan is read
  if (tid < S) part_off[tid] = static_cast<int32_t>(off);
  if (tid == 0) part_off[S] = static_cast<int32_t>(total);
  cp_async_wait_all();
  __syncthreads();
  if (pages > 0) m.pt_smem = pt_smem;
  const uint32_t lambda = lh.x, shift = lh.y;
  uint32_t* chist = hist + kHC;
  // gather: kThreads / S threads per part, each taking every (kThreads / S)-th entry
  // of it, eight loads in flight at a time
  uint32_t top = 0;
  {
    const int tpp = kThreads / S;  // S is a power of two <= kMaxSplit <= kThreads
    const int part = tid / tpp, sub = tid % tpp;
    const uint32_t cnt = static_cast<uint32_t>(part_off[part + 1] - part_off[part]);
    const uint2* src = entries + (static_cast<int64_t>(row) * S + part) * scap;
    uint2* dst = buf + part_off[part];
    for (uint32_t b = static_cast<uint32_t>(sub); b < cnt; b += 8u * static_cast<uint32_t>(tpp)) {
      uint2 e[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t i = b + static_cast<uint32_t>(u * tpp);
        e[u] = i < cnt ? src[i] : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t i = b + static_cast<uint32_t>(u * tpp);
        if (i < cnt) {
          dst[i] = e[u];
          const uint32_t d = (e[u].x - lambda) >> shift;
          if (d >= static_cast<uint32_t>(kCandBins - 1))
            ++top;
          else
            atomicAdd(&chist[hist_index(static_cast<int>(d))], 1u);
        }
      }
    }
  }
  top = __reduce_add_sync(kFull, top);
  if ((tid & 31) == 0 && top != 0) atomicAdd(&chist[hist_index(kCandBins - 1)], top);
  __syncthreads();  // buffer, histogram; the offsets in list are read no more
  select_candidates<F>(buf, total, static_cast<uint32_t>(k), chist, lambda, shift, list, hist,
                       reinterpret_cast<int32_t*>(hist), L, out, m, ctl);
}

// One cluster of G CTAs per row (with kSingle: one CTA, G = 1 at compile time).
template <int F>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) topk_rows_kernel(const Params p) {
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ Ctl ctl;
  if constexpr ((F & kStaged) != 0) {
    staged_row<F>(p, static_cast<int>(blockIdx.x), dyn, ctl);
  } else if constexpr ((F & kSingle) != 0) {
    row_body<F>(p, static_cast<int>(blockIdx.x), 1, 0, dyn, ctl);
  } else {
    const int G = static_cast<int>(cluster_nctarank());
    row_body<F>(p, static_cast<int>(blockIdx.x) / G, G, static_cast<int>(cluster_ctarank()), dyn,
                ctl);
  }
}

// Several problems of one form in one launch: the clusters take the problems' rows
// in order (problem i owns rows [row_begin[i], row_begin[i + 1])). Each CTA copies
// its problem's parameters to shared memory once.
template <int F>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    topk_group_kernel(const __grid_constant__ GroupParams gp) {
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ Ctl ctl;
  __shared__ Params prob;
  const int G = static_cast<int>(cluster_nctarank());
  const int item = static_cast<int>(blockIdx.x) / G;
  int i = 0;
  while (i + 1 < gp.n && gp.row_begin[i + 1] <= item) ++i;
  if (threadIdx.x == 0) prob = gp.probs[i];
  __syncthreads();
  if constexpr ((F & kStaged) != 0)
    staged_row<F>(prob, item - gp.row_begin[i], dyn, ctl);
  else
    row_body<F>(prob, item - gp.row_begin[i], G, static_cast<int>(cluster_ctarank()), dyn, ctl);
}

// The chip-wide split's two kernels (split_filter_part, split_select_row).
template <int F>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) topk_split_filter_kernel(const Params p) {
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ Ctl ctl;
  const int S = p.split_s;
  split_filter_part<F>(p, static_cast<int>(blockIdx.x) / S, static_cast<int>(blockIdx.x) % S, dyn, ctl);
}
template <int F>
__global__ void __launch_bounds__(kThreads, 1) topk_split_select_kernel(const Params p) {
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ Ctl ctl;
  const int G = static_cast<int>(cluster_nctarank());
  split_select_row<F>(p, static_cast<int>(blockIdx.x) / G, G, static_cast<int>(cluster_ctarank()),
                      dyn, ctl);
}

// The sort pass of the sorted output (one CTA per row, after the selection kernel):
// the row's k staged (key, position) pairs are ordered by the composite (key,
// ~position), largest first, so equal keys come by smaller position first and the
// padding pairs (composite 0) last, with a bitonic network in shared memory; then
// out (mapped) and values are written in that order.
constexpr int kSortMax = 2048;  // the largest k
template <int F>
__global__ void __launch_bounds__(kThreads) topk_sort_kernel(const Params p) {
  __shared__ uint64_t v[kSortMax];
  const int row = static_cast<int>(blockIdx.x);
  const int tid = threadIdx.x;
  const int k = p.k;
  allow_next_grid();
  wait_prior_grids();  // the staged pairs come from the selection kernel
  int n = 1;
  while (n < k) n <<= 1;
  const uint2* st = p.staged + static_cast<int64_t>(row) * k;
  for (int i = tid; i < n; i += kThreads) {
    uint64_t c = 0;
    if (i < k) {
      const uint2 e = st[i];
      c = (static_cast<uint64_t>(e.x) << 32) | static_cast<uint64_t>(~e.y);
    }
    v[i] = c;
  }
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = tid; i < n; i += kThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const uint64_t a = v[i], b = v[j];
          const bool desc = (i & size) == 0;  // this run is ordered largest first
          if (desc ? a < b : a > b) {
            v[i] = b;
            v[j] = a;
          }
        }
      }
    }
  }
  __syncthreads();
  OutMap m;
  m.pt_row = form_of(F) == kPaged ? p.page_table + static_cast<int64_t>(row) * p.pt_stride : nullptr;
  m.pt_smem = nullptr;
  // every staged position lies on a page below the row's page count; entries past
  // the table's row stride are not read (the selection kernel counted that row)
  m.pt_n = static_cast<int32_t>(min(p.pt_stride, static_cast<int64_t>(INT32_MAX)));
  m.ps = p.page_size;
  m.ps_shift = p.page_shift;
  m.rstart = 0;
  m.values = p.values != nullptr ? p.values + static_cast<int64_t>(row) * k : nullptr;
  m.staged = nullptr;
  if constexpr (form_of(F) == kRagged) {
    m.rstart = p.row_starts[row];
  } else if constexpr (form_of(F) == kWindow) {  // the window's first column, as the selection took it
    const int64_t hi = min(static_cast<int64_t>(max(p.seq_lens[row], 0)), p.row_stride);
    m.rstart = static_cast<int32_t>(min(static_cast<int64_t>(max(p.row_starts[row], 0)), hi));
  }
  int32_t* out = p.out + static_cast<int64_t>(row) * k;
  for (int i = tid; i < k; i += kThreads) {
    const uint64_t c = v[i];
    if (c == 0)
      emit_pad<F>(out, static_cast<uint32_t>(i), m);
    else
      emit<F>(out, k, static_cast<uint32_t>(i), m, static_cast<int32_t>(~static_cast<uint32_t>(c)),
              static_cast<uint32_t>(c >> 32));
  }
}

// Dynamic shared memory of a launch: the rows kernels' layout for clusters of g, or
// the staged tier's.
constexpr size_t rows_smem_bytes(int g, int tie_cap) {
  return sizeof(uint32_t) * static_cast<size_t>(kHistWords * (g > 1 ? 2 : 1) + kListWords + kPtCap) +
         sizeof(uint2) * static_cast<size_t>(tie_cap);
}
// The chip-wide split's filter CTA: histogram | its candidate buffer.
constexpr size_t split_filter_smem_bytes(int split_cap) {
  return sizeof(uint32_t) * static_cast<size_t>(kHistWords) + sizeof(uint2) * static_cast<size_t>(split_cap);
}
template <bool kHalf>
constexpr size_t staged_smem_bytes(int tie_cap) {
  return sizeof(uint32_t) * static_cast<size_t>(staged_fixed_words<kHalf>()) +
         sizeof(uint2) * static_cast<size_t>(tie_cap);
}

#ifdef TOPK_FORM
// ---------------------------------------------------------------- one form's kernels
//
// Each form's kernels are compiled in an object of their own (TOPK_FORM = the form),
// so that the objects build in parallel; the object without TOPK_FORM holds the
// dispatch by form below.

// Dynamic shared memory of a kernel with template argument F.
template <int F>
constexpr size_t kernel_smem_bytes(int g, int tie_cap) {
  return (F & kStaged) == 0        ? rows_smem_bytes(g, tie_cap)
         : (F & kHalfStage) != 0   ? staged_smem_bytes<true>(tie_cap)
                                   : staged_smem_bytes<false>(tie_cap);
}

template <int F, class Kernel, class Arg>
cudaError_t launch_clusters(Kernel kernel, const Arg& arg, int64_t rows, int g, int tie_cap,
                            cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows * g), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kernel_smem_bytes<F>(g, tie_cap);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(g);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

template <int F>
cudaError_t launch_group_form(const GroupParams& gp, int g, cudaStream_t stream) {
  return launch_clusters<F>(topk_group_kernel<F>, gp, gp.row_begin[gp.n], g, gp.probs[0].tie_cap,
                            stream);
}

template <int F>
cudaError_t launch_rows_form(const Params& p, int g, cudaStream_t stream) {
  return launch_clusters<F>(topk_rows_kernel<F>, p, p.batch, g, p.tie_cap, stream);
}

template <class Kernel>
cudaError_t prepare_kernel(Kernel kernel, size_t smem = rows_smem_bytes(2, kTieCapMax)) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

constexpr int kForm = TOPK_FORM;
static_assert(kForm >= kRaw && kForm <= kWindow, "TOPK_FORM must be a Form");

}  // namespace

#if TOPK_FORM == 0
#define TOPK_FORM_NS raw
#elif TOPK_FORM == 1
#define TOPK_FORM_NS paged
#elif TOPK_FORM == 2
#define TOPK_FORM_NS ragged
#else
#define TOPK_FORM_NS window
#endif

namespace TOPK_FORM_NS {

cudaError_t prepare_device() {
  constexpr int F = kForm;
  cudaError_t e = prepare_kernel(topk_rows_kernel<F>);
  if (e == cudaSuccess) e = prepare_kernel(topk_rows_kernel<F | kSingle>);
  if (e == cudaSuccess) e = prepare_kernel(topk_rows_kernel<F | kSingle | kKeysInFilter>);
  if (e == cudaSuccess) e = prepare_kernel(topk_group_kernel<F>);
  if (e == cudaSuccess) e = prepare_kernel(topk_group_kernel<F | kKeysInFilter>);
  if (e == cudaSuccess) e = prepare_kernel(topk_group_kernel<F | kOpts | kKeysInFilter>);
  if (e == cudaSuccess) e = prepare_kernel(topk_group_kernel<F | kOpts>);
  if (e == cudaSuccess)
    e = prepare_kernel(topk_split_filter_kernel<F>, split_filter_smem_bytes(kSplitCapMax));
  if (e == cudaSuccess)
    e = prepare_kernel(topk_split_select_kernel<F>, rows_smem_bytes(2, kGatherCapMax));
  if constexpr (kHasStaged) {
    const size_t full = staged_smem_bytes<false>(kTieCapMax), half = staged_smem_bytes<true>(kTieCapMax);
    if (e == cudaSuccess) e = prepare_kernel(topk_rows_kernel<F | kSingle | kStaged>, full);
    if (e == cudaSuccess) e = prepare_kernel(topk_group_kernel<F | kStaged>, full);
    if (e == cudaSuccess) e = prepare_kernel(topk_group_kernel<F | kOpts | kStaged>, full);
    if (e == cudaSuccess) e = prepare_kernel(topk_rows_kernel<F | kSingle | kStaged | kHalfStage>, half);
    if (e == cudaSuccess) e = prepare_kernel(topk_group_kernel<F | kStaged | kHalfStage>, half);
    if (e == cudaSuccess) e = prepare_kernel(topk_group_kernel<F | kOpts | kStaged | kHalfStage>, half);
  }
  return e;
}

cudaError_t launch(const Params& p, int g, bool keys_in_filter, int staged, cudaStream_t stream) {
  constexpr int F = kForm;
  if constexpr (kHasStaged) {
    if (g == 1 && staged == 1) return launch_rows_form<F | kSingle | kStaged>(p, 1, stream);
    if (g == 1 && staged == 2) return launch_rows_form<F | kSingle | kStaged | kHalfStage>(p, 1, stream);
  } else {
    if (staged != 0) return cudaErrorInvalidValue;
  }
  if (g == 1 && keys_in_filter) return launch_rows_form<F | kSingle | kKeysInFilter>(p, 1, stream);
  if (g == 1) return launch_rows_form<F | kSingle>(p, 1, stream);
  return launch_rows_form<F>(p, g, stream);
}

cudaError_t launch_group(const GroupParams& gp, int g, bool opts, bool keys_in_filter, int staged,
                         cudaStream_t stream) {
  constexpr int F = kForm;
  if constexpr (kHasStaged) {
    if (staged == 1 && g == 1)
      return opts ? launch_group_form<F | kOpts | kStaged>(gp, g, stream)
                  : launch_group_form<F | kStaged>(gp, g, stream);
    if (staged == 2 && g == 1)
      return opts ? launch_group_form<F | kOpts | kStaged | kHalfStage>(gp, g, stream)
                  : launch_group_form<F | kStaged | kHalfStage>(gp, g, stream);
  } else {
    if (staged != 0) return cudaErrorInvalidValue;
  }
  const bool keys = keys_in_filter && g == 1;
  if (opts)
    return keys ? launch_group_form<F | kOpts | kKeysInFilter>(gp, g, stream)
                : launch_group_form<F | kOpts>(gp, g, stream);
  return keys ? launch_group_form<F | kKeysInFilter>(gp, g, stream)
              : launch_group_form<F>(gp, g, stream);
}

cudaError_t launch_split(const Params& p, cudaStream_t stream) {
  constexpr int F = kForm;
  if (p.split_s < 1 || p.split_s > kMaxSplit || (p.split_s & (p.split_s - 1)) != 0 ||
      p.split_cap < 0 || p.split_cap > kSplitCapMax || p.gather_cap < 0 || p.split_g < 1 ||
      p.split_g > kMaxCluster || (p.split_g & (p.split_g - 1)) != 0 ||
      p.gather_cap > kGatherCapMax || p.split_ws == nullptr || p.values != nullptr ||
      p.staged != nullptr)
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(p.batch) * p.split_s), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = split_filter_smem_bytes(p.split_cap);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, topk_split_filter_kernel<F>, p);
  if (e != cudaSuccess) return e;
  // the select kernel: one cluster of split_g CTAs per row
  cudaLaunchAttribute attr2[2];
  attr2[0] = attr[0];
  attr2[1].id = cudaLaunchAttributeClusterDimension;
  attr2[1].val.clusterDim.x = static_cast<unsigned>(p.split_g);
  attr2[1].val.clusterDim.y = 1;
  attr2[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(p.batch) * p.split_g), 1, 1);
  cfg.dynamicSmemBytes = rows_smem_bytes(p.split_g, p.gather_cap);
  cfg.attrs = attr2;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, topk_split_select_kernel<F>, p);
}

cudaError_t max_active_clusters(int g, int* n) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(g), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = rows_smem_bytes(g, kTieCapMax);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(g);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, topk_rows_kernel<kForm>, &cfg);
}

cudaError_t sort_rows(const Params& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_sort_kernel<kForm | kOpts>, p);
}

cudaError_t guard_hits(unsigned int* hits) {
  return cudaMemcpyFromSymbol(hits, g_guard_hits, sizeof(unsigned int));
}

cudaError_t reset_guard_hits() {
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_guard_hits, &zero, sizeof(unsigned int));
}

}  // namespace TOPK_FORM_NS
#undef TOPK_FORM_NS

#else
// ---------------------------------------------------------------- dispatch by form

}  // namespace

size_t smem_bytes(int g, int tie_cap) { return rows_smem_bytes(g, tie_cap); }

bool staged_fits(int64_t row_len) {
  return kHasStaged && row_len > 0 && row_len <= 4 * static_cast<int64_t>(kStagedQuads);
}

cudaError_t prepare_device() {
  cudaError_t e = raw::prepare_device();
  if (e == cudaSuccess) e = paged::prepare_device();
  if (e == cudaSuccess) e = ragged::prepare_device();
  if (e == cudaSuccess) e = window::prepare_device();
  return e;
}

cudaError_t launch(Form form, const Params& p, int g, bool keys_in_filter, int staged,
                   cudaStream_t stream) {
  switch (form) {
    case kRaw: return raw::launch(p, g, keys_in_filter, staged, stream);
    case kPaged: return paged::launch(p, g, keys_in_filter, staged, stream);
    case kRagged: return ragged::launch(p, g, keys_in_filter, staged, stream);
    case kWindow: return window::launch(p, g, keys_in_filter, staged, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_group(Form form, const GroupParams& gp, int g, bool opts,
                         bool keys_in_filter, int staged, cudaStream_t stream) {
  switch (form) {
    case kRaw: return raw::launch_group(gp, g, opts, keys_in_filter, staged, stream);
    case kPaged: return paged::launch_group(gp, g, opts, keys_in_filter, staged, stream);
    case kRagged: return ragged::launch_group(gp, g, opts, keys_in_filter, staged, stream);
    case kWindow: return window::launch_group(gp, g, opts, keys_in_filter, staged, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_split(Form form, const Params& p, cudaStream_t stream) {
  switch (form) {
    case kRaw: return raw::launch_split(p, stream);
    case kPaged: return paged::launch_split(p, stream);
    case kRagged: return ragged::launch_split(p, stream);
    case kWindow: return window::launch_split(p, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t max_active_clusters(int g, int* n) { return raw::max_active_clusters(g, n); }

cudaError_t sort_rows(Form form, const Params& p, cudaStream_t stream) {
  switch (form) {
    case kRaw: return raw::sort_rows(p, stream);
    case kPaged: return paged::sort_rows(p, stream);
    case kRagged: return ragged::sort_rows(p, stream);
    case kWindow: return window::sort_rows(p, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t guard_hits(unsigned int* hits) {
  unsigned int a = 0, b = 0, c = 0, d = 0;
  cudaError_t e = raw::guard_hits(&a);
  if (e == cudaSuccess) e = paged::guard_hits(&b);
  if (e == cudaSuccess) e = ragged::guard_hits(&c);
  if (e == cudaSuccess) e = window::guard_hits(&d);
  *hits = a + b + c + d;
  return e;
}

cudaError_t reset_guard_hits() {
  cudaError_t e = raw::reset_guard_hits();
  if (e == cudaSuccess) e = paged::reset_guard_hits();
  if (e == cudaSuccess) e = ragged::reset_guard_hits();
  if (e == cudaSuccess) e = window::reset_guard_hits();
  return e;
}

#endif  // TOPK_FORM

}  // namespace TOPK_CTA_NS
}  // namespace topk_gb300
