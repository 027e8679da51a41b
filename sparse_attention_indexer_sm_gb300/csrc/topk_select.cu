// Exact per-row top-k selection of fp32 indexer scores on GB300 (sm_103a).
//
// One thread-block cluster of G CTAs (G = 1, 2, 4, 8 or 16) owns one row; each
// CTA owns a contiguous slice of it. The steps follow the exact "coop" top-k of
// the sglang PR #37591 summary page (section "实现拆解" (implementation
// breakdown) item 1 and the coop_topk_kernel excerpt under "关键源码片段"),
// re-planned for this machine:
//
//  1. key      every fp32 becomes its order-preserving 32-bit key (negatives
//              bit-inverted, the rest with the sign bit set: unsigned order ==
//              float order; PR #37591 page, order_key32).
//  2. round 0  a 4096-bin shared-memory histogram of the top 12 key bits over the
//              slice, read from HBM with 128-bit loads. With G > 1 the slices'
//              histograms are summed into CTA 0 through distributed shared
//              memory; CTA 0 finds the threshold bin with a block-wide suffix
//              scan and sends it back (the page's "binary search for the threshold
//              bucket" computes the same bin).
//  3. more     while the threshold bin holds more elements than the tie buffer,
//     rounds   one more histogram of the next 12 (then 8) key bits restricted to
//              that bin narrows it (the page's second, 4-bit round does the same
//              job; this build uses wider rounds so that fewer passes are needed
//              when values concentrate).
//  4. scatter  elements above the threshold bin are winners and go straight to the
//              output, mapped; elements in it go to the shared tie buffer of CTA 0
//              (the page's "scatter pass"). Both use one shared atomic per warp.
//  5. refine   CTA 0 selects the missing winners among the ties by radix rounds on
//              the 64-bit composite (key, ~position): the rest of the key first,
//              then the position, so equal keys go to the smaller position (the
//              page's "radix sort of the ties on the full fp32 key").
//  6. rescan   when even the full 32-bit key leaves more equal elements than the
//              tie buffer holds (88% identical values, say), no element is
//              dropped: every CTA re-reads its slice in position order and takes
//              its quota of the equal elements by a block-wide prefix count (the
//              page's "overflow rescan of the whole row").
//
// No step waits on another CTA except through the hardware cluster barrier, so
// there is no spin loop, no global workspace and no inter-launch dependency.

#include <cstdint>

#include "topk_select.cuh"

namespace topk_gb300 {
namespace {

constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;            // 128-bit loads in flight per thread per step
constexpr int kRowRoundBits = 12;     // histogram width of the passes over the row
constexpr int kBufRoundBits = 10;     // histogram width of the rounds over the ties
constexpr unsigned kFull = 0xFFFFFFFFu;

struct Ctl {
  uint32_t scan[kWarps];              // per-warp partials of block scans
  uint32_t sel_t, sel_above, sel_count;  // threshold bin of the current round
  uint32_t win_cnt, tie_cnt, out_cnt;    // slot counters
  uint32_t xa[kMaxCluster];           // per-CTA winners (cluster exchange)
  uint32_t xt[kMaxCluster];           // per-CTA threshold-bin elements
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

__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" :: "r"(addr), "r"(a), "r"(b)
               : "memory");
}

// 128-bit read-only load that does not allocate in L1 (each byte is read once
// per pass; a second pass finds it in L2).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Reserve n consecutive slots of *counter for this lane; one atomic per warp.
// Must be called by all 32 lanes.
__device__ __forceinline__ uint32_t warp_reserve(uint32_t* counter, uint32_t n) {
  const int lane = threadIdx.x & 31;
  uint32_t x = n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
  const uint32_t total = __shfl_sync(kFull, x, 31);
  uint32_t base = 0;
  if (total != 0) {
    if (lane == 31) base = atomicAdd(counter, total);
    base = __shfl_sync(kFull, base, 31);
  }
  return base + x - n;
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
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
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

// Threshold bin of histogram h[0, nbins): the bin t where the count from the top
// reaches `need` (need <= sum of h). Writes t, the count strictly above t and
// h[t] into ctl.sel_*; all threads see them on return.
__device__ __forceinline__ void find_threshold(const uint32_t* h, int nbins, uint32_t need,
                                               Ctl& ctl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nbins >= kThreads ? nbins / kThreads : 1;
  const int b0 = tid * per;
  uint32_t s = 0;
  if (b0 < nbins)
    for (int i = 0; i < per; ++i) s += h[b0 + i];
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
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t c = h[b0 + i];
      if (acc + c >= need) {
        ctl.sel_t = static_cast<uint32_t>(b0 + i);
        ctl.sel_above = acc;
        ctl.sel_count = c;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ row slices

// This CTA's part of a row: a 16-byte-aligned body of 4-element quads split
// evenly over the cluster, plus the unaligned head (CTA 0) and tail (last CTA).
struct Slice {
  const float* row;
  const uint4* vec;       // quad 0 of the aligned body
  int64_t q0, q1;         // this CTA's quads
  int32_t vec0;           // row position of quad 0
  int32_t n_head;         // positions [0, n_head) belong to this CTA
  int32_t tail0, n_tail;  // positions [tail0, tail0 + n_tail) belong to this CTA
  int32_t lo, hi;         // the CTA's positions as one range [lo, hi)
};

__device__ __forceinline__ Slice make_slice(const float* row, int32_t L, int rank, int G) {
  Slice s;
  s.row = row;
  const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row) >> 2) & 3u;
  int32_t head = static_cast<int32_t>((4u - mis) & 3u);
  if (head > L) head = L;
  const int64_t nvec = static_cast<int64_t>(L - head) >> 2;
  s.vec0 = head;
  s.vec = reinterpret_cast<const uint4*>(row + head);
  s.q0 = nvec * rank / G;
  s.q1 = nvec * (rank + 1) / G;
  const int32_t tail0 = head + static_cast<int32_t>(nvec * 4);
  s.n_head = rank == 0 ? head : 0;
  s.tail0 = tail0;
  s.n_tail = rank == G - 1 ? L - tail0 : 0;
  s.lo = rank == 0 ? 0 : head + static_cast<int32_t>(s.q0 * 4);
  s.hi = rank == G - 1 ? L : head + static_cast<int32_t>(s.q1 * 4);
  return s;
}

// Calls f(valid, key, position) for every position of the slice. Control flow is
// block-uniform; `valid` is false for padding lanes.
template <class F>
__device__ __forceinline__ void visit_keys(const Slice& s, F&& f) {
  const int tid = threadIdx.x;
  {
    bool ok = false;
    int32_t j = 0;
    if (tid < s.n_head) {
      ok = true;
      j = tid;
    } else if (tid >= 4 && tid - 4 < s.n_tail) {
      ok = true;
      j = s.tail0 + (tid - 4);
    }
    const uint32_t key = ok ? order_key(__float_as_uint(s.row[j])) : 0u;
    f(ok, key, j);
  }
  for (int64_t base = s.q0; base < s.q1; base += static_cast<int64_t>(kUnroll) * kThreads) {
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t q = base + static_cast<int64_t>(u) * kThreads + tid;
      x[u] = q < s.q1 ? ld_stream(s.vec + q) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t q = base + static_cast<int64_t>(u) * kThreads + tid;
      const bool ok = q < s.q1;
      const int32_t j = s.vec0 + 4 * static_cast<int32_t>(q);
      f(ok, order_key(x[u].x), j);
      f(ok, order_key(x[u].y), j + 1);
      f(ok, order_key(x[u].z), j + 2);
      f(ok, order_key(x[u].w), j + 3);
    }
  }
}

// ------------------------------------------------------------------ output map

struct OutMap {
  const int32_t* pt_row;  // paged: this row's page table
  int32_t ps;             // page size
  int32_t ps_shift;       // log2(ps) or -1
  int32_t rstart;         // ragged: row start in the packed buffer
};

template <int F>
__device__ __forceinline__ int32_t map_pos(const OutMap& m, int32_t j) {
  if constexpr (F == kPaged) {
    int32_t page, off;
    if (m.ps_shift >= 0) {
      page = j >> m.ps_shift;
      off = j & (m.ps - 1);
    } else {
      page = j / m.ps;
      off = j - page * m.ps;
    }
    return __ldg(m.pt_row + page) * m.ps + off;
  } else if constexpr (F == kRagged) {
    return m.rstart + j;
  } else {
    return j;
  }
}

// ------------------------------------------------------------------ passes

// Step 4: winners (key >> shift > prefix) to out[win_base + ...], ties
// (key >> shift == prefix) to the tie buffer at tie_base + ... (CTA 0's buffer,
// through distributed shared memory when G > 1).
template <int F>
__device__ __forceinline__ void scatter_pass(const Slice& s, uint32_t prefix, int shift,
                                             int32_t* out, uint32_t win_base, uint32_t tie_base,
                                             uint2* ties, uint32_t ties_remote, bool remote,
                                             const OutMap& m, Ctl& ctl) {
  const int tid = threadIdx.x;
  auto put_tie = [&](uint32_t slot, uint32_t key, int32_t j) {
    if (remote)
      dsmem_st2(ties_remote + 8u * slot, key, static_cast<uint32_t>(j));
    else
      ties[slot] = make_uint2(key, static_cast<uint32_t>(j));
  };
  {  // unaligned head and tail, at most one position per thread
    bool ok = false;
    int32_t j = 0;
    if (tid < s.n_head) {
      ok = true;
      j = tid;
    } else if (tid >= 4 && tid - 4 < s.n_tail) {
      ok = true;
      j = s.tail0 + (tid - 4);
    }
    const uint32_t key = ok ? order_key(__float_as_uint(s.row[j])) : 0u;
    const bool win = ok && (key >> shift) > prefix;
    const bool tie = ok && (key >> shift) == prefix;
    const uint32_t ws = warp_reserve(&ctl.win_cnt, win ? 1u : 0u);
    const uint32_t ts = warp_reserve(&ctl.tie_cnt, tie ? 1u : 0u);
    if (win) out[win_base + ws] = map_pos<F>(m, j);
    if (tie) put_tie(tie_base + ts, key, j);
  }
  for (int64_t base = s.q0; base < s.q1; base += static_cast<int64_t>(kUnroll) * kThreads) {
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t q = base + static_cast<int64_t>(u) * kThreads + tid;
      x[u] = q < s.q1 ? ld_stream(s.vec + q) : make_uint4(0, 0, 0, 0);
    }
    uint32_t key[4 * kUnroll];
    uint32_t wb = 0, tb = 0;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t q = base + static_cast<int64_t>(u) * kThreads + tid;
      const bool ok = q < s.q1;
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
      uint32_t ws = warp_reserve(&ctl.win_cnt, __popc(wb));
      uint32_t ts = warp_reserve(&ctl.tie_cnt, __popc(tb));
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t q = base + static_cast<int64_t>(u) * kThreads + tid;
        const int32_t j = s.vec0 + 4 * static_cast<int32_t>(q);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int bit = 4 * u + c;
          if ((wb >> bit) & 1u) out[win_base + ws++] = map_pos<F>(m, j + c);
          if ((tb >> bit) & 1u) put_tie(tie_base + ts++, key[bit], j + c);
        }
      }
    }
  }
}

// Step 5 (CTA 0 only): among the c ties (all with key >> shift == prefix) select
// the `need` largest composites (key, ~position) and write them to
// out[k_above + ...].
template <int F>
__device__ __forceinline__ void refine_ties(const uint2* ties, uint32_t c, uint32_t need,
                                            int shift, uint32_t prefix, int32_t L, int32_t* out,
                                            uint32_t k_above, const OutMap& m, uint32_t* h,
                                            Ctl& ctl) {
  const int tid = threadIdx.x;
  auto compose = [](uint2 e) -> uint64_t {
    return (static_cast<uint64_t>(e.x) << 32) | static_cast<uint64_t>(~e.y);
  };
  uint64_t P = prefix;   // known high bits of the composite: composite >> p == P
  int p = 32 + shift;
  if (need < c) {
    const int nb = 32 - __clz(L - 1);  // positions fit in nb bits (L >= 2 here)
    for (;;) {
      if (p == 32) {  // key resolved: the ~position bits above nb are all ones
        const int skip = 32 - nb;
        P = (P << skip) | ((1ull << skip) - 1ull);
        p = nb;
      }
      const int lo = p > 32 ? 32 : 0;
      const int w = min(kBufRoundBits, p - lo);
      const int np = p - w;
      const uint32_t mask = (1u << w) - 1u;
      for (int i = tid; i <= static_cast<int>(mask); i += kThreads) h[i] = 0;
      __syncthreads();
      for (uint32_t i = tid; i < c; i += kThreads) {
        const uint64_t v = compose(ties[i]);
        if ((v >> p) == P) atomicAdd(&h[static_cast<uint32_t>(v >> np) & mask], 1u);
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
  // every tie whose composite prefix is >= P is selected
  const uint32_t cpad = (c + kThreads - 1) / kThreads * kThreads;
  for (uint32_t i = tid; i < cpad; i += kThreads) {
    bool sel = false;
    uint2 e = make_uint2(0, 0);
    if (i < c) {
      e = ties[i];
      sel = (compose(e) >> p) >= P;
    }
    const uint32_t slot = warp_reserve(&ctl.out_cnt, sel ? 1u : 0u);
    if (sel) out[k_above + slot] = map_pos<F>(m, static_cast<int32_t>(e.y));
  }
}

// Step 6: key tau is exact and more elements than the tie buffer holds equal it.
// Each CTA scans its slice in position order, writes its winners (key > tau) and
// the first `quota` of its elements equal to tau.
template <int F>
__device__ __forceinline__ void emit_equal(const Slice& s, uint32_t tau, int32_t* out,
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
    uint32_t ws = warp_reserve(&ctl.win_cnt, __popc(wb));
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if ((wb >> u) & 1u) out[win_base + ws++] = map_pos<F>(m, j0 + u);
    uint32_t total;
    uint32_t r = taken + block_excl_scan(__popc(eb), ctl, &total);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if ((eb >> u) & 1u) {
        if (r < quota) out[eq_slot0 + r] = map_pos<F>(m, j0 + u);
        ++r;
      }
    }
    taken += total;
  }
}

// ------------------------------------------------------------------ the kernel

template <int F>
__global__ void __launch_bounds__(kThreads, 2) topk_rows_kernel(const Params p) {
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ Ctl ctl;
  const int tid = threadIdx.x;
  const int G = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int row = static_cast<int>(blockIdx.x) / G;

  OutMap m;
  m.pt_row = nullptr;
  m.ps = p.page_size;
  m.ps_shift = p.page_shift;
  m.rstart = 0;
  const int32_t seq = p.seq_lens[row];
  const float* rowp;
  int32_t L;
  if constexpr (F == kRagged) {
    m.rstart = p.row_starts[row];
    rowp = p.scores + m.rstart;
    L = max(seq, 0);
  } else {
    rowp = p.scores + static_cast<int64_t>(row) * p.row_stride;
    L = static_cast<int32_t>(min(static_cast<int64_t>(max(seq, 0)), p.row_stride));
  }
  if constexpr (F == kPaged) m.pt_row = p.page_table + static_cast<int64_t>(row) * p.pt_stride;
  const int32_t k = p.k;
  int32_t* out = p.out + static_cast<int64_t>(row) * k;

  if (L <= k) {  // every position is selected; the rest of the row is -1
    const int32_t s0 = static_cast<int32_t>(static_cast<int64_t>(k) * rank / G);
    const int32_t s1 = static_cast<int32_t>(static_cast<int64_t>(k) * (rank + 1) / G);
    for (int32_t i = s0 + tid; i < s1; i += kThreads) out[i] = i < L ? map_pos<F>(m, i) : -1;
    return;
  }

  uint32_t* hist = dyn;                                   // this CTA's histogram
  uint32_t* mhist = dyn + kMaxBins;                       // cluster sum (CTA 0, G > 1)
  uint2* ties = reinterpret_cast<uint2*>(dyn + (G > 1 ? 2 : 1) * kMaxBins);

  if (tid == 0) {
    ctl.win_cnt = 0;
    ctl.tie_cnt = 0;
    ctl.out_cnt = 0;
  }
  if (G > 1) {
    if (rank == 0)
      for (int i = tid; i < kMaxBins; i += kThreads) mhist[i] = 0;
    cluster_sync();  // all CTAs running, CTA 0's sum histogram cleared
  }
  const Slice s = make_slice(rowp, L, rank, G);

  // Steps 2-3: radix rounds over the row until the threshold bin fits the tie
  // buffer (or the key is exhausted).
  uint32_t need = static_cast<uint32_t>(k);  // winners still to find at or below the bin
  uint32_t prefix = 0;                       // known high bits of the threshold key
  int shift = 32;                            // prefix == threshold key >> shift
  uint32_t cnt = static_cast<uint32_t>(L);   // elements whose key >> shift == prefix
  uint32_t above_local = 0;                  // this CTA's elements above the bin
  uint32_t tie_local = 0;                    // this CTA's elements in the bin
  for (;;) {
    const int w = min(kRowRoundBits, shift);
    const int nshift = shift - w;
    const uint32_t mask = (1u << w) - 1u;
    for (int i = tid; i <= static_cast<int>(mask); i += kThreads) hist[i] = 0;
    __syncthreads();
    visit_keys(s, [&](bool ok, uint32_t key, int32_t) {
      if (ok && __funnelshift_rc(key, 0u, shift) == prefix)
        atomicAdd(&hist[(key >> nshift) & mask], 1u);
    });
    __syncthreads();
    uint32_t t, above, c;
    if (G == 1) {
      find_threshold(hist, 1 << w, need, ctl);
      t = ctl.sel_t;
      above = ctl.sel_above;
      c = ctl.sel_count;
      above_local += above;
      tie_local = c;
    } else {
      const uint32_t m0 = map_rank(smem_addr(mhist), 0);
      for (int i = tid; i <= static_cast<int>(mask); i += kThreads) {
        const uint32_t v = hist[i];
        if (v != 0) dsmem_add(m0 + 4u * static_cast<uint32_t>(i), v);
      }
      cluster_sync();
      if (rank == 0) {
        find_threshold(mhist, 1 << w, need, ctl);
        if (tid > 0 && tid < G) {
          dsmem_st(map_rank(smem_addr(&ctl.sel_t), tid), ctl.sel_t);
          dsmem_st(map_rank(smem_addr(&ctl.sel_above), tid), ctl.sel_above);
          dsmem_st(map_rank(smem_addr(&ctl.sel_count), tid), ctl.sel_count);
        }
        for (int i = tid; i <= static_cast<int>(mask); i += kThreads) mhist[i] = 0;
      }
      cluster_sync();
      t = ctl.sel_t;
      above = ctl.sel_above;
      c = ctl.sel_count;
      uint32_t part = 0;
      for (int i = tid; i <= static_cast<int>(mask); i += kThreads)
        part += static_cast<uint32_t>(i) > t ? hist[i] : 0u;
      tie_local = hist[t];
      above_local += block_sum(part, ctl);
    }
    need -= above;
    prefix = (prefix << w) | t;
    shift = nshift;
    cnt = c;
    if (cnt <= static_cast<uint32_t>(p.tie_cap) || shift == 0) break;
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

  if (cnt <= static_cast<uint32_t>(p.tie_cap)) {
    const bool remote = G > 1 && rank != 0;
    const uint32_t ties_remote = G > 1 ? map_rank(smem_addr(ties), 0) : 0u;
    scatter_pass<F>(s, prefix, shift, out, win_base, tie_base, ties, ties_remote, remote, m, ctl);
    if (G > 1)
      cluster_sync();  // CTA 0 now holds every tie
    else
      __syncthreads();
    if (rank == 0) refine_ties<F>(ties, cnt, need, shift, prefix, L, out, k_above, m, hist, ctl);
  } else {
    // tie_base is this CTA's first position among the elements equal to prefix
    const uint32_t quota = tie_base >= need ? 0u : min(need - tie_base, tie_local);
    const uint32_t eq_slot0 = k_above + min(tie_base, need);
    emit_equal<F>(s, prefix, out, win_base, eq_slot0, quota, m, ctl);
  }
}

template <int F>
cudaError_t launch_form(const Params& p, int g, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * static_cast<unsigned>(g), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes(g, p.tie_cap);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(g);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_rows_kernel<F>, p);
}

template <int F>
cudaError_t prepare_form() {
  cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel<F>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_bytes(2, kTieCapMax)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(topk_rows_kernel<F>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace

size_t smem_bytes(int g, int tie_cap) {
  return sizeof(uint32_t) * kMaxBins * (g > 1 ? 2 : 1) + sizeof(uint2) * static_cast<size_t>(tie_cap);
}

cudaError_t prepare_device() {
  cudaError_t e = prepare_form<kRaw>();
  if (e == cudaSuccess) e = prepare_form<kPaged>();
  if (e == cudaSuccess) e = prepare_form<kRagged>();
  return e;
}

cudaError_t launch(Form form, const Params& p, int g, cudaStream_t stream) {
  switch (form) {
    case kRaw: return launch_form<kRaw>(p, g, stream);
    case kPaged: return launch_form<kPaged>(p, g, stream);
    case kRagged: return launch_form<kRagged>(p, g, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace topk_gb300
