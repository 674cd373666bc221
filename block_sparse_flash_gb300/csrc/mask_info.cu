// mask_info.cu -- builds the sparse execution table (MaskInfo) on the GPU.
//
// "Pallas Kernels and Splash Attention" (CMU 11-868 Lecture 13 notes):
//   §6.1  blocks of the mask are empty (skip), full (no element mask) or
//         partial (element mask needed);
//   §6.2  MaskInfo: block_mask, the active rows / columns, the deduplicated
//         partial patterns and mask_next, bounds_start / bounds_end;
//   §6.4  segment IDs (q_id == kv_id) joined with causal / local by AND.
//
// Pipeline (all kernels on the caller's stream):
//   K1 seg_summary   per q-block / kv-block min and max segment id (and the
//                    counters cleared)
//   K2 classify      exact allowed-element count of every block -> class,
//                    per-row active / partial counts, allowed pairs; blocks
//                    the summaries cannot decide go to count_deferred (one
//                    CTA per block, the key block's IDs staged in shared memory)
//   K3 scan_order    row_ptr (CSR), partial offsets, and the rows by
//                    descending active count (the attention's work order)
//      compact       active lists in row-major, kv-ascending order, bounds
//   K4 partial_hash  a content hash of each partial block's element pattern
//      dedup         first partial with identical content (hash prefilter,
//                    exact word-by-word comparison)
//      scan_finalize pattern index of each first occurrence, mask_next
//      materialize   the patterns, bit-packed (the byte form of
//                    partial_mask_blocks is expanded on the host when the
//                    table is copied there)
// The pattern buffer is sized from a bound known before the build (no host
// wait) unless that bound exceeds kPatternBudgetBytes; then the build waits
// once for the exact pattern count.  Band-only masks (no segment IDs) take
// the classes in closed form.  Small band tables run the whole pipeline as
// one single-CTA kernel (build_small_kernel); other tables up to 4M blocks
// as one persistent cooperative kernel whose phases are separated by a grid
// barrier (build_grid_kernel); larger ones as the chain of kernels above.
#include <algorithm>
#include <atomic>
#include <climits>
#include <mutex>

#include "internal.h"

namespace {

struct DevMask {
  int32_t causal;
  int64_t wl, wr;
  const int32_t *qseg, *kvseg;
  int64_t Lq, Lk, nq, nk;
  int32_t bq, bk, nbm;
  int32_t ragged;  // Lq or Lk is not a multiple of its block: the grid is padded
};

// The band part of the joint mask for query i: allowed keys j lie in [lo, hi]
// intersected with [c0, c1].  Padding of a ragged grid (queries i >= Lq, keys
// j >= Lk) is masked ("Pallas Kernels and Splash Attention" §2.3: ragged
// edges are padded so that every block has the same size).
__device__ __forceinline__ void band_range(const DevMask &m, int64_t i, int64_t c0, int64_t c1,
                                           int64_t &lo, int64_t &hi) {
  lo = c0;
  hi = min(c1, m.Lk - 1);
  if (m.causal) hi = min(hi, i);
  if (m.wl >= 0) lo = max(lo, i - m.wl);
  if (m.wr >= 0) hi = min(hi, i + m.wr);
  if (i >= m.Lq) hi = lo - 1;
}

// 32 mask bits of query i against keys j0 .. j0+31 (bit t = key j0 + t).
__device__ __forceinline__ uint32_t row_word(const DevMask &m, int32_t bm, int64_t i, int32_t sq,
                                             int64_t j0) {
  int64_t lo, hi;
  band_range(m, i, j0, j0 + 31, lo, hi);
  if (hi < lo) return 0u;
  uint32_t bits = 0u;
  if (m.qseg == nullptr) {
    int64_t n = hi - lo + 1;  // 1..32 contiguous bits starting at lo - j0
    uint32_t run = n >= 32 ? 0xffffffffu : ((1u << n) - 1u);
    bits = run << (lo - j0);
  } else {
    const int32_t *kv = m.kvseg + (int64_t)bm * m.Lk;
    for (int64_t j = lo; j <= hi; ++j)
      if (kv[j] == sq) bits |= 1u << (j - j0);
  }
  return bits;
}

__device__ __forceinline__ int32_t q_segment(const DevMask &m, int32_t bm, int64_t i) {
  return (m.qseg && i < m.Lq) ? m.qseg[(int64_t)bm * m.Lq + i] : 0;  // padding rows: unused
}

// q_segment issued as a volatile load of the read-only segment array, so
// that a batch of them stays where it is written (the compiler would
// otherwise sink each load to its first use, one memory latency per row)
__device__ __forceinline__ int32_t q_segment_early(const DevMask &m, int32_t bm, int64_t i) {
  if (!(m.qseg && i < m.Lq)) return 0;
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(m.qseg + (int64_t)bm * m.Lq + i));
  return v;
}

// The band part in closed form: key j is allowed for query i iff
// i - W <= j <= i + A, with A = 0 for causal (and min with the right window)
// and W the left window; an unbounded side is kBandInf.
constexpr int64_t kBandInf = (int64_t)1 << 60;

__device__ __forceinline__ void band_limits(const DevMask &m, int64_t &A, int64_t &W) {
  A = kBandInf;
  if (m.causal) A = 0;
  if (m.wr >= 0) A = min(A, m.wr);
  W = m.wl >= 0 ? m.wl : kBandInf;
}

// Class of block (r, c) under the band alone (0 empty, 1 partial, 2 full).
// Rows i in [r0, r1] and keys j in [c0, c1]: the block holds an allowed pair
// iff some row i has i + A >= c0 and i - W <= c1; it is full iff every row has
// lo(i) = max(c0, i - W) = c0 and hi(i) = min(c1, i + A) = c1, i.e. iff
// r1 - W <= c0 and r0 + A >= c1 (lo and hi are nondecreasing in i).  On a
// ragged grid the rows and keys are first clipped to the sequences, and a
// block with padding is never full.
__device__ __forceinline__ int band_block_class(const DevMask &m, int64_t A, int64_t W, int64_t r, int64_t c) {
  const int64_t r0 = r * m.bq, r1 = r0 + m.bq - 1, c0 = c * m.bk, c1 = c0 + m.bk - 1;
  const int64_t r1v = min(r1, m.Lq - 1), c1v = min(c1, m.Lk - 1);
  if (max(r0, c0 - A) > min(r1v, c1v + W)) return 0;
  return (r1v == r1 && c1v == c1 && r1 - W <= c0 && r0 + A >= c1) ? 2 : 1;
}

// Allowed keys of query i under the band alone.
__device__ __forceinline__ int64_t band_row_count(const DevMask &m, int64_t A, int64_t W, int64_t i) {
  if (i >= m.Lq) return 0;
  return max((int64_t)0, min(m.Lk - 1, i + A) - max((int64_t)0, i - W) + 1);
}

// Segment IDs of key block c of batch row bm, staged in shared memory by the
// whole CTA (keys past Lk are never read: band_range clips them).  Returns,
// to every thread, whether the block's IDs are non-decreasing (then the keys
// with a given ID form one run, found by binary search).
__device__ __forceinline__ bool stage_kv_ids(const DevMask &m, int32_t bm, int64_t c, int32_t *s_kv) {
  const int64_t n = min((int64_t)m.bk, m.Lk - c * m.bk);  // real keys of the block
  for (int32_t t = threadIdx.x; t < m.bk; t += blockDim.x) {
    const int64_t j = c * m.bk + t;
    s_kv[t] = j < m.Lk ? m.kvseg[(int64_t)bm * m.Lk + j] : 0;
  }
  __syncthreads();
  bool sorted = true;
  for (int32_t t = threadIdx.x; t + 1 < n; t += blockDim.x) sorted &= s_kv[t] <= s_kv[t + 1];
  return __syncthreads_and(sorted) != 0;
}

// The run [a, b] (block offsets) of keys with ID sq in a sorted staged block
// of n real keys (empty: a > b).
__device__ __forceinline__ void sorted_run(const int32_t *s_kv, int32_t n, int32_t sq, int32_t &a, int32_t &b) {
  int32_t lo = 0, hi = n;  // first index with s_kv >= sq
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (s_kv[mid] < sq) lo = mid + 1; else hi = mid;
  }
  a = lo;
  hi = n;  // first index with s_kv > sq
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (s_kv[mid] <= sq) lo = mid + 1; else hi = mid;
  }
  b = lo - 1;
}

// For a block whose n real keys have non-decreasing IDs (s_kv, staged), the
// run [ra, rb] of keys with ID sq (the caller's query ID; each lane its own)
// is ra = #(IDs < sq), rb = #(IDs <= sq) - 1: counted by ballots over the
// keys lane, lane+32, .. (bk <= 128), one pass per distinct sq in the warp.
// Warp-collective; it replaces two binary searches of dependent shared-memory
// loads per row.
__device__ __forceinline__ void sorted_run_warp(const int32_t *s_kv, int32_t n, int32_t sq, int32_t &ra,
                                                int32_t &rb) {
  const int lane = threadIdx.x & 31;
  int32_t kid[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) kid[j] = s_kv[lane + 32 * j];
  unsigned todo = 0xffffffffu;
  while (todo != 0u) {  // warp-uniform
    const int32_t v = __shfl_sync(0xffffffffu, sq, __ffs(todo) - 1);
    int32_t lt = 0, le = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool valid = lane + 32 * j < n;
      lt += __popc(__ballot_sync(0xffffffffu, valid && kid[j] < v));
      le += __popc(__ballot_sync(0xffffffffu, valid && kid[j] <= v));
    }
    if (sq == v) {
      ra = lt;
      rb = le - 1;
    }
    todo &= ~__ballot_sync(0xffffffffu, sq == v);
  }
}

// row_word with the key block's segment IDs staged in shared memory (its
// first key is c0): 32 mask bits of query i (segment id sq) against keys
// j0 .. j0+31.  For a sorted block, run = [ra, rb] is the row's run of keys
// with ID sq (block offsets, from sorted_run) and the word is one range of bits.
__device__ __forceinline__ uint32_t row_word_staged(const DevMask &m, int64_t i, int32_t sq, int64_t c0, int64_t j0,
                                                    const int32_t *s_kv, bool sorted, int32_t ra, int32_t rb) {
  int64_t lo, hi;
  band_range(m, i, j0, j0 + 31, lo, hi);
  if (sorted) {
    lo = max(lo, c0 + ra);
    hi = min(hi, c0 + rb);
    if (hi < lo) return 0u;
    const int64_t n = hi - lo + 1;
    return (n >= 32 ? 0xffffffffu : ((1u << n) - 1u)) << (lo - j0);
  }
  uint32_t bits = 0u;
  for (int64_t j = lo; j <= hi; ++j) bits |= (uint32_t)(s_kv[j - c0] == sq) << (j - j0);
  return bits;
}

// Real keys of key block c (fewer than bk only in the last block of a ragged Lk).
__device__ __forceinline__ int32_t block_keys(const DevMask &m, int64_t c) {
  return (int32_t)min((int64_t)m.bk, m.Lk - c * m.bk);
}

// ---------------------------------------------------------------- K1
// One warp per q-block or kv-block of batch row bm (warp index `warp` within
// the row).  Also clears the per-row counters.
__device__ __forceinline__ void seg_summary_warp(const DevMask &m, int64_t warp, int32_t bm, int32_t *qsum,
                                                 int32_t *kvsum, int32_t *row_cnt, int32_t *row_pcnt) {
  const int lane = threadIdx.x & 31;
  const bool isq = warp < m.nq;
  if (isq && lane == 0) {
    row_cnt[(int64_t)bm * m.nq + warp] = 0;
    row_pcnt[(int64_t)bm * m.nq + warp] = 0;
  }
  const int64_t blk = isq ? warp : warp - m.nq;
  // the last block of a ragged sequence holds fewer positions
  const int32_t n = (int32_t)(isq ? min((int64_t)m.bq, m.Lq - blk * m.bq) : min((int64_t)m.bk, m.Lk - blk * m.bk));
  const int32_t *seg = isq ? m.qseg + (int64_t)bm * m.Lq + blk * m.bq
                           : m.kvseg + (int64_t)bm * m.Lk + blk * m.bk;
  int32_t mn = INT_MAX, mx = INT_MIN;
  for (int32_t x = lane; x < n; x += 32) {
    int32_t s = seg[x];
    mn = min(mn, s);
    mx = max(mx, s);
  }
  for (int off = 16; off; off >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if (lane == 0) {
    int32_t *dst = isq ? qsum + ((int64_t)bm * m.nq + blk) * 2 : kvsum + ((int64_t)bm * m.nk + blk) * 2;
    dst[0] = mn;
    dst[1] = mx;
  }
}

// Also clears the totals that classify_kernel adds to.
__global__ void seg_summary_kernel(DevMask m, int32_t *qsum, int32_t *kvsum, int32_t *row_cnt, int32_t *row_pcnt,
                                   unsigned long long *counters) {
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 8) counters[threadIdx.x] = 0ull;
  if (warp >= m.nq + m.nk) return;
  seg_summary_warp(m, warp, (int32_t)blockIdx.y, qsum, kvsum, row_cnt, row_pcnt);
}

// ---------------------------------------------------------------- K2
// One thread per block (bm, r, c); a CTA covers 128 blocks of one row.
constexpr int kClassifyThreads = 128;

// Blocks the segment summaries cannot decide (both a shared and a differing
// segment id possible) are appended to `deferred` (block index row * nk + c;
// counters[5] counts the appends) for count_deferred_kernel, which counts each
// with a whole CTA.  Blocks beyond the list's capacity `defer_cap` (or all of
// them, with deferred == nullptr) are counted here, element by element.
// The CTA (any multiple of 32 threads up to 1024) classifies blocks
// xc*blockDim .. of row r of batch row bm, one thread per block.
__device__ void classify_body(const DevMask &m, int64_t xc, int64_t r, int32_t bm, const int32_t *qsum,
                              const int32_t *kvsum, int8_t *block_mask, int32_t *row_cnt, int32_t *row_pcnt,
                              unsigned long long *counters, int32_t *deferred, int64_t defer_cap) {
  const int64_t c = xc * blockDim.x + threadIdx.x;
  const int64_t row = (int64_t)bm * m.nq + r;
  int64_t cnt = 0;
  int cls = 0;
  bool undecided = false;  // segment summaries leave the block's class open
  if (m.qseg == nullptr) {
    // band only: classes in closed form; the allowed pairs are counted per
    // query row by the first CTA of the row (cnt is then a row count)
    int64_t A, W;
    band_limits(m, A, W);
    if (c < m.nk) {
      cls = band_block_class(m, A, W, r, c);
      block_mask[row * m.nk + c] = (int8_t)cls;
    }
    if (xc == 0)
      for (int32_t di = threadIdx.x; di < m.bq; di += blockDim.x) cnt += band_row_count(m, A, W, r * m.bq + di);
  } else if (c < m.nk) {
    // the band's allowed pairs of the block: none or all of them in closed
    // form; a band-partial block's are summed row by row below, by its warp
    int64_t A, W;
    band_limits(m, A, W);
    if (band_block_class(m, A, W, r, c) == 2) cnt = (int64_t)m.bq * m.bk;
  }
  if (m.qseg != nullptr) {
    // band-partial blocks: their rows' band counts summed by the whole warp
    // (one such block per lane at a time; lanes take rows lane, lane+32, ...)
    int64_t A, W;
    band_limits(m, A, W);
    const bool bpart = c < m.nk && band_block_class(m, A, W, r, c) == 1;
    unsigned need = __ballot_sync(0xffffffffu, bpart);
    const int lane = threadIdx.x & 31;
    while (need != 0u) {
      const int src = __ffs(need) - 1;
      need &= need - 1u;
      const int64_t cc = __shfl_sync(0xffffffffu, c, src);
      int64_t part = 0;
      for (int32_t di = lane; di < m.bq; di += 32) {
        int64_t lo, hi;
        band_range(m, r * m.bq + di, cc * m.bk, cc * m.bk + m.bk - 1, lo, hi);
        if (hi >= lo) part += hi - lo + 1;
      }
      for (int off = 16; off; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      if (lane == src) cnt = part;
    }
  }
  if (m.qseg != nullptr && c < m.nk && cnt > 0) {
    const int32_t qmn = qsum[row * 2], qmx = qsum[row * 2 + 1];
    const int32_t kmn = kvsum[((int64_t)bm * m.nk + c) * 2], kmx = kvsum[((int64_t)bm * m.nk + c) * 2 + 1];
    if (qmx < kmn || kmx < qmn) {
      cnt = 0;  // no segment id in common
    } else if (!(qmn == qmx && kmn == kmx && qmn == kmn)) {
      undecided = true;  // handled below, with the whole warp
    }
    // (both constant and equal: the band count stands)
  }
  if (m.qseg != nullptr) {
    // undecided blocks: counted by count_deferred_kernel while the list has
    // room (slots reserved with one atomic per warp), else here element by element
    const unsigned um = __ballot_sync(0xffffffffu, undecided && deferred != nullptr);
    unsigned long long base = 0;
    if (um) {
      const int leader = __ffs(um) - 1;
      if ((int)(threadIdx.x & 31) == leader) base = atomicAdd(&counters[5], (unsigned long long)__popc(um));
      base = __shfl_sync(0xffffffffu, base, leader);
    }
    if (undecided) {
      const unsigned long long slot =
          deferred != nullptr ? base + __popc(um & ((1u << (threadIdx.x & 31)) - 1u)) : ~0ull;
      if (slot < (unsigned long long)defer_cap) {
        deferred[slot] = (int32_t)(row * m.nk + c);
        cnt = -1;
      } else {
        const int64_t c0 = c * m.bk, c1 = c0 + m.bk - 1;
        const int32_t *kv = m.kvseg + (int64_t)bm * m.Lk;
        cnt = 0;
        for (int32_t di = 0; di < m.bq; ++di) {
          const int64_t i = r * m.bq + di;
          const int32_t sq = q_segment(m, bm, i);
          int64_t lo, hi;
          band_range(m, i, c0, c1, lo, hi);
          for (int64_t j = lo; j <= hi; ++j) cnt += (kv[j] == sq);
        }
      }
    }
    if (cnt < 0) {
      cnt = 0;  // deferred: class and counts come from count_deferred_kernel
      cls = 0;
    } else if (c < m.nk) {
      cls = cnt == 0 ? 0 : (cnt == (int64_t)m.bq * m.bk ? 2 : 1);
      block_mask[row * m.nk + c] = (int8_t)cls;
    }
  }
  // reduce within the CTA (all threads share the row)
  int na = cls != 0, np = cls == 1;
  unsigned long long ns = (unsigned long long)cnt;
  for (int off = 16; off; off >>= 1) {
    na += __shfl_xor_sync(0xffffffffu, na, off);
    np += __shfl_xor_sync(0xffffffffu, np, off);
    ns += __shfl_xor_sync(0xffffffffu, ns, off);
  }
  __shared__ int sa[32], sp[32];
  __shared__ unsigned long long ss[32];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sa[w] = na;
    sp[w] = np;
    ss[w] = ns;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int ta = 0, tp = 0;
    unsigned long long ts = 0;
    for (int x = 0; x < (int)(blockDim.x >> 5); ++x) {
      ta += sa[x];
      tp += sp[x];
      ts += ss[x];
    }
    if (ta) atomicAdd(&row_cnt[row], ta);
    if (tp) atomicAdd(&row_pcnt[row], tp);
    if (ts) atomicAdd(&counters[3], ts);
  }
  __syncthreads();  // sa / sp / ss are rewritten by the CTA's next call
}

__global__ void __launch_bounds__(kClassifyThreads)
classify_kernel(DevMask m, const int32_t *qsum, const int32_t *kvsum, int8_t *block_mask,
                int32_t *row_cnt, int32_t *row_pcnt, unsigned long long *counters, int32_t *deferred,
                int64_t defer_cap) {
  classify_body(m, blockIdx.x, blockIdx.y, (int32_t)blockIdx.z, qsum, kvsum, block_mask, row_cnt, row_pcnt,
                counters, deferred, defer_cap);
}

// One CTA (kClassifyThreads threads, one per query row of the block) per
// deferred block: the allowed pairs of row i are the keys of the row's band
// range with i's segment id; the block's class and its row / total counts are
// then added like classify_kernel's.
__device__ void count_deferred_body(const DevMask &m, const int32_t *deferred, int64_t defer_cap, int8_t *block_mask,
                                    int32_t *row_cnt, int32_t *row_pcnt, unsigned long long *counters, int64_t bid,
                                    int64_t nb) {
  __shared__ unsigned long long part[32];
  __shared__ int32_t s_kv[128];  // the block's key segment IDs (bk <= 128)
  const int64_t n = min((int64_t)counters[5], defer_cap);
  const int di = threadIdx.x, lane = di & 31;
  for (int64_t x = bid; x < n; x += nb) {
    const int64_t idx = deferred[x];
    const int64_t row = idx / m.nk, c = idx - row * m.nk;
    const int32_t bm = (int32_t)(row / m.nq);
    const int64_t r = row - (int64_t)bm * m.nq;
    // (the first row's query ID is loaded beside the key IDs)
    const int32_t sq0 = di < m.bq ? q_segment_early(m, bm, r * m.bq + di) : 0;
    const bool sorted = stage_kv_ids(m, bm, c, s_kv);
    unsigned long long cnt = 0;
    // (bq and the block's thread count are multiples of 32: the loop's trip
    // count is the same for every lane of a warp, as sorted_run_warp needs)
    for (int32_t d = di; d < m.bq; d += blockDim.x) {
      const int64_t i = r * m.bq + d;
      int64_t lo, hi;
      band_range(m, i, c * m.bk, c * m.bk + m.bk - 1, lo, hi);
      const int32_t sq = d == di ? sq0 : q_segment(m, bm, i);
      int32_t a = 0, b = -1;
      if (sorted) sorted_run_warp(s_kv, block_keys(m, c), sq, a, b);
      if (hi >= lo) {
        if (sorted)
          cnt += (unsigned long long)max((int64_t)0, min(hi, c * m.bk + b) - max(lo, c * m.bk + a) + 1);
        else
          for (int64_t j = lo; j <= hi; ++j) cnt += (s_kv[j - c * m.bk] == sq);
      }
    }
    for (int off = 16; off; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    if (lane == 0) part[di >> 5] = cnt;
    __syncthreads();
    if (di == 0) {
      unsigned long long t = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += part[w];
      const int cls = t == 0 ? 0 : (t == (unsigned long long)m.bq * m.bk ? 2 : 1);
      block_mask[idx] = (int8_t)cls;
      if (cls != 0) atomicAdd(&row_cnt[row], 1);
      if (cls == 1) atomicAdd(&row_pcnt[row], 1);
      if (t) atomicAdd(&counters[3], t);
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kClassifyThreads)
count_deferred_kernel(DevMask m, const int32_t *deferred, int64_t defer_cap, int8_t *block_mask, int32_t *row_cnt,
                      int32_t *row_pcnt, unsigned long long *counters) {
  count_deferred_body(m, deferred, defer_cap, block_mask, row_cnt, row_pcnt, counters, blockIdx.x, gridDim.x);
}

// ---------------------------------------------------------------- scans
// Single-CTA exclusive scan of one or two int32 arrays (1024 threads).
__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  return x;
}

// Returns the exclusive prefix of x within the CTA and the CTA total.
__device__ __forceinline__ int block_excl_scan(int x, int &total, int *warp_buf) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = warp_incl_scan(x);
  if (lane == 31) warp_buf[w] = incl;
  __syncthreads();
  if (w == 0) {
    int v = lane < nw ? warp_buf[lane] : 0;
    int vi = warp_incl_scan(v);
    if (lane < nw) warp_buf[lane] = vi - v;
    if (lane == 31) warp_buf[32] = vi;
  }
  __syncthreads();
  int ex = warp_buf[w] + incl - x;
  total = warp_buf[32];
  __syncthreads();
  return ex;
}

// Exclusive prefix within the CTA of 64-bit values (two 32-bit counts packed
// in one word: their sums never carry into each other) and the CTA total.
__device__ __forceinline__ unsigned long long block_excl_scan64(unsigned long long x, unsigned long long &total,
                                                                unsigned long long *warp_buf) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned long long incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_buf[w] = incl;
  __syncthreads();
  if (w == 0) {
    const unsigned long long v = lane < nw ? warp_buf[lane] : 0ull;
    unsigned long long vi = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, vi, off);
      if (lane >= off) vi += y;
    }
    if (lane < nw) warp_buf[lane] = vi - v;
    if (lane == 31) warp_buf[32] = vi;
  }
  __syncthreads();
  const unsigned long long ex = warp_buf[w] + incl - x;
  total = warp_buf[32];
  __syncthreads();
  return ex;
}

__device__ __forceinline__ void scan_rows_body(int64_t R, const int32_t *row_cnt, const int32_t *row_pcnt,
                                               int32_t *row_ptr, int32_t *prow_ptr, unsigned long long *counters) {
  __shared__ int buf_a[33], buf_p[33];
  int carry_a = 0, carry_p = 0, mx = 0;
  for (int64_t base = 0; base < R; base += blockDim.x) {
    const int64_t x = base + threadIdx.x;
    const int a = x < R ? row_cnt[x] : 0;
    const int p = x < R ? row_pcnt[x] : 0;
    mx = max(mx, a);
    int ta, tp;
    const int ea = block_excl_scan(a, ta, buf_a);
    const int ep = block_excl_scan(p, tp, buf_p);
    if (x < R) {
      row_ptr[x] = carry_a + ea;
      prow_ptr[x] = carry_p + ep;
    }
    carry_a += ta;
    carry_p += tp;
  }
  for (int off = 16; off; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  __shared__ int smx[32];
  if ((threadIdx.x & 31) == 0) smx[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = max(t, smx[w]);
    row_ptr[R] = carry_a;
    prow_ptr[R] = carry_p;
    counters[0] = (unsigned long long)carry_a;
    counters[1] = (unsigned long long)carry_p;
    counters[4] = (unsigned long long)t;
  }
}

// ---------------------------------------------------------------- K3 compact
// One warp per row (b_mask, r): columns in chunks of 32, ballots give each
// active block its position.
// g0 .. gend: the row's range of the active lists; k0: its first partial index
__device__ __forceinline__ void compact_warp(const DevMask &m, int64_t row, int32_t g0, int32_t gend, int32_t k0,
                                             const int8_t *block_mask, int32_t *active_rows, int32_t *active_cols,
                                             int32_t *mask_next, uint8_t *bounds_start, uint8_t *bounds_end,
                                             int32_t *part_row, int32_t *part_col, int32_t *part_g) {
  const int lane = threadIdx.x & 31;
  const int32_t r = (int32_t)(row % m.nq);
  int32_t g = g0, k = k0;
  const unsigned lt = (1u << lane) - 1u;
  // the row's classes are loaded 256 columns (8 chunks) at a time, then placed
  for (int64_t cb0 = 0; cb0 < m.nk; cb0 += 256) {
    int cl[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int64_t c = cb0 + 32 * t + lane;
      cl[t] = c < m.nk ? block_mask[row * m.nk + c] : 0;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int64_t cb = cb0 + 32 * t;
      if (cb >= m.nk) break;
      const int64_t c = cb + lane;
      const int cls = cl[t];
      const unsigned act = __ballot_sync(0xffffffffu, cls != 0);
      const unsigned par = __ballot_sync(0xffffffffu, cls == 1);
      if (cls != 0) {
        const int32_t pos = g + __popc(act & lt);
        active_rows[pos] = r;
        active_cols[pos] = (int32_t)c;
        mask_next[pos] = -1;
        bounds_start[pos] = (uint8_t)(pos == g0);
        bounds_end[pos] = (uint8_t)(pos == gend - 1);
        if (cls == 1) {
          const int32_t kk = k + __popc(par & lt);
          part_row[kk] = (int32_t)row;
          part_col[kk] = (int32_t)c;
          part_g[kk] = pos;
        }
      }
      g += __popc(act);
      k += __popc(par);
    }
  }
}

__global__ void compact_kernel(DevMask m, int64_t R, const int8_t *block_mask,
                               const int32_t *row_ptr, const int32_t *prow_ptr,
                               int32_t *active_rows, int32_t *active_cols, int32_t *mask_next,
                               uint8_t *bounds_start, uint8_t *bounds_end, int32_t *part_row,
                               int32_t *part_col, int32_t *part_g) {
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= R) return;
  compact_warp(m, row, row_ptr[row], row_ptr[row + 1], prow_ptr[row], block_mask, active_rows, active_cols,
               mask_next, bounds_start, bounds_end, part_row, part_col, part_g);
}

// ---------------------------------------------------------------- K4 patterns
constexpr uint64_t kHashBasis = 0xcbf29ce484222325ull;
constexpr uint64_t kHashPrime = 0x100000001b3ull;

__device__ __forceinline__ uint64_t hash_step(uint64_t h, uint64_t x) { return (h ^ x) * kHashPrime; }

// Content hash of a partial block: an FNV hash per row (over the row's mask
// words), mixed with the row index by the splitmix64 finalizer (Steele, Lea
// and Flood, 2014) and summed over the rows.  A sum reduces in parallel (a
// sequential fold over 128 rows costs ~10k cycles); equal contents give equal
// hashes, and the hash only pre-filters the exact comparison.
__device__ __forceinline__ uint64_t row_hash_term(uint64_t rowh, int32_t di) {
  uint64_t z = rowh + (uint64_t)(di + 1) * 0x9e3779b97f4a7c15ull;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// One CTA per partial block, grid-stride; thread di < bq takes query row di
// (a CTA of more threads leaves the others idle).
__device__ void partial_hash_body(const DevMask &m, const unsigned long long *counters, const int32_t *part_row,
                                  const int32_t *part_col, uint64_t *part_hash, int64_t bid, int64_t nb) {
  __shared__ uint64_t wsum[8];  // bq <= 256 threads
  __shared__ int32_t s_kv[128];  // the block's key segment IDs (bk <= 128)
  const int64_t Ap = (int64_t)counters[1];
  const int di = threadIdx.x;
  const bool act = di < m.bq;
  for (int64_t k = bid; k < Ap; k += nb) {
    const int64_t row = part_row[k];
    const int32_t bm = (int32_t)(row / m.nq);
    const int64_t r = row % m.nq, c = part_col[k];
    if (m.qseg == nullptr && !m.ragged) {
      // band only: the diagonal offset identifies the content exactly (see
      // build_small_kernel), and serves as the "hash"
      if (di == 0) part_hash[k] = (uint64_t)(c * m.bk - r * m.bq);
      continue;
    }
    const bool sorted = m.qseg != nullptr ? stage_kv_ids(m, bm, c, s_kv) : false;
    uint64_t t = 0;
    if (act) {  // whole warps (bq is a multiple of 32)
      const int64_t i = r * m.bq + di;
      const int32_t sq = q_segment(m, bm, i);
      int32_t ra = 0, rb = -1;
      if (sorted) sorted_run(s_kv, block_keys(m, c), sq, ra, rb);
      uint64_t h = kHashBasis;
      for (int32_t w = 0; w < m.bk / 32; ++w)
        h = hash_step(h, m.qseg != nullptr
                             ? row_word_staged(m, i, sq, c * m.bk, c * m.bk + w * 32, s_kv, sorted, ra, rb)
                             : row_word(m, bm, i, sq, c * m.bk + w * 32));
      t = warp_sum_u64(row_hash_term(h, di));
    }
    if (act && (di & 31) == 0) wsum[di >> 5] = t;
    __syncthreads();
    if (di == 0) {
      uint64_t H = 0;
      for (int x = 0; x < m.bq / 32; ++x) H += wsum[x];
      part_hash[k] = H;
    }
    __syncthreads();
  }
}

__global__ void partial_hash_kernel(DevMask m, const unsigned long long *counters, const int32_t *part_row,
                                    const int32_t *part_col, uint64_t *part_hash) {
  partial_hash_body(m, counters, part_row, part_col, part_hash, blockIdx.x, gridDim.x);
}

// CTA-wide exact comparison of two partial blocks' patterns: each thread
// compares (row, 32-key word) pieces of both blocks; every thread of the CTA
// must call it and gets the same result.  With segment IDs, s_kv_a / s_kv_b
// hold the two blocks' key IDs (staged by the caller).
__device__ bool patterns_equal(const DevMask &m, const int32_t *part_row, const int32_t *part_col, int64_t ka,
                               int64_t kb, const int32_t *s_kv_a, const int32_t *s_kv_b, bool sorted_a,
                               bool sorted_b) {
  const int64_t rowa = part_row[ka], rowb = part_row[kb];
  const int32_t bma = (int32_t)(rowa / m.nq), bmb = (int32_t)(rowb / m.nq);
  const int64_t ra = rowa % m.nq, rb = rowb % m.nq, ca = part_col[ka], cb = part_col[kb];
  const int32_t words = m.bk / 32;
  bool same = true;
  for (int32_t x = threadIdx.x; x < m.bq * words && same; x += blockDim.x) {
    const int32_t di = x / words, w = x - di * words;
    const int64_t ia = ra * m.bq + di, ib = rb * m.bq + di;
    if (m.qseg != nullptr) {
      const int32_t sa = q_segment(m, bma, ia), sb = q_segment(m, bmb, ib);
      int32_t a0 = 0, a1 = -1, b0 = 0, b1 = -1;
      if (sorted_a) sorted_run(s_kv_a, block_keys(m, ca), sa, a0, a1);
      if (sorted_b) sorted_run(s_kv_b, block_keys(m, cb), sb, b0, b1);
      same = row_word_staged(m, ia, sa, ca * m.bk, ca * m.bk + w * 32, s_kv_a, sorted_a, a0, a1) ==
             row_word_staged(m, ib, sb, cb * m.bk, cb * m.bk + w * 32, s_kv_b, sorted_b, b0, b1);
    } else
      same = row_word(m, bma, ia, 0, ca * m.bk + w * 32) == row_word(m, bmb, ib, 0, cb * m.bk + w * 32);
  }
  return __syncthreads_and(same) != 0;
}

// One CTA per partial block k (grid-stride): rep[k] = the first k' <= k with
// identical content.  Earlier blocks of equal hash are the candidates, tried
// in ascending order; each exact comparison uses the whole CTA.
constexpr int kDedupThreads = 256;
__device__ void dedup_body(const DevMask &m, const unsigned long long *counters, const int32_t *part_row,
                           const int32_t *part_col, const uint64_t *part_hash, int32_t *part_rep, int64_t bid,
                           int64_t nb) {
  __shared__ uint32_t s_ball[kDedupThreads / 32];
  __shared__ int32_t s_kv_a[128], s_kv_b[128];  // key segment IDs of block k and of the candidate
  const int64_t Ap = (int64_t)counters[1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // band-only whole blocks: equal diagonal offsets (the "hash") mean equal content
  const bool by_offset = m.qseg == nullptr && !m.ragged;
  for (int64_t k = bid; k < Ap; k += nb) {
    const uint64_t h = part_hash[k];
    int64_t rep = k;  // uniform over the CTA
    bool staged_a = false, sorted_a = false, sorted_b = false;
    for (int64_t base = 0; base < k && rep == k; base += kDedupThreads) {
      const int64_t kp = base + tid;
      const unsigned b = __ballot_sync(0xffffffffu, kp < k && part_hash[kp] == h);
      if (lane == 0) s_ball[warp] = b;
      __syncthreads();
      for (int w = 0; w < kDedupThreads / 32 && rep == k; ++w) {
        unsigned cand = s_ball[w];
        while (cand && rep == k) {
          const int64_t kc = base + 32 * w + (__ffs(cand) - 1);
          cand &= cand - 1u;
          if (by_offset) {
            rep = kc;
            continue;
          }
          if (m.qseg != nullptr) {
            // (patterns_equal ends with a CTA barrier, so the previous
            // comparison has finished reading the staged IDs)
            if (!staged_a) {
              const int64_t row = part_row[k];
              sorted_a = stage_kv_ids(m, (int32_t)(row / m.nq), part_col[k], s_kv_a);
              staged_a = true;
            }
            sorted_b = stage_kv_ids(m, (int32_t)(part_row[kc] / m.nq), part_col[kc], s_kv_b);
          }
          if (patterns_equal(m, part_row, part_col, k, kc, s_kv_a, s_kv_b, sorted_a, sorted_b)) rep = kc;
        }
      }
      __syncthreads();  // s_ball is rewritten by the next chunk
    }
    if (tid == 0) part_rep[k] = (int32_t)rep;
  }
}

__global__ void __launch_bounds__(kDedupThreads)
dedup_kernel(DevMask m, const unsigned long long *counters, const int32_t *part_row, const int32_t *part_col,
             const uint64_t *part_hash, int32_t *part_rep) {
  dedup_body(m, counters, part_row, part_col, part_hash, part_rep, blockIdx.x, gridDim.x);
}

// Pattern indices (one CTA): an exclusive scan of the first-occurrence flags
// in partial order gives each representative its pattern index (P = the
// total); then every partial block's mask_next and the pattern list
// (partial index of pattern u).
// The pattern indices (one CTA): part_pidx[k] = the first occurrences among
// partial blocks 0 .. k-1, and their total P in counters[2].
__device__ void scan_reps_body(unsigned long long *counters, const int32_t *part_rep, int32_t *part_pidx) {
  __shared__ int buf[33];
  const int64_t Ap = (int64_t)counters[1];
  int carry = 0;
  for (int64_t base = 0; base < Ap; base += blockDim.x) {
    const int64_t k = base + threadIdx.x;
    const int f = (k < Ap && part_rep[k] == k) ? 1 : 0;
    int tot;
    const int ex = block_excl_scan(f, tot, buf);
    if (k < Ap) part_pidx[k] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) counters[2] = (unsigned long long)carry;
}

__device__ void scan_finalize_body(unsigned long long *counters, const int32_t *part_g, const int32_t *part_rep,
                                   int32_t *part_pidx, int32_t *mask_next, int32_t *rep_list) {
  const int64_t Ap = (int64_t)counters[1];
  scan_reps_body(counters, part_rep, part_pidx);
  __syncthreads();  // part_pidx is complete
  for (int64_t k = threadIdx.x; k < Ap; k += blockDim.x) {
    const int32_t rep = part_rep[k];
    const int32_t u = part_pidx[rep];
    mask_next[part_g[k]] = u;
    if (rep == k) rep_list[u] = (int32_t)k;
  }
}

__global__ void __launch_bounds__(1024)
scan_finalize_kernel(unsigned long long *counters, const int32_t *part_g, const int32_t *part_rep,
                     int32_t *part_pidx, int32_t *mask_next, int32_t *rep_list) {
  scan_finalize_body(counters, part_g, part_rep, part_pidx, mask_next, rep_list);
}

// One CTA (bq threads) per pattern: its bit-packed rows (word w of row di
// holds keys 32w .. 32w+31).  The pattern count is read on the device
// (counters[2]) and never exceeds the buffer capacity `cap` (a count above
// it is reported and clipped).
__device__ void materialize_body(const DevMask &m, const unsigned long long *counters, int64_t cap,
                                 const int32_t *rep_list, const int32_t *part_row, const int32_t *part_col,
                                 uint32_t *pattern_bits, uint32_t *err, int64_t bid, int64_t nb) {
  __shared__ int32_t s_kv[128];  // the block's key segment IDs (bk <= 128)
  const int di = threadIdx.x;
  const bool act = di < m.bq;  // thread di takes row di (others idle)
  const int32_t words = m.bk / 32;
  int64_t P = (int64_t)counters[2];
  if (P > cap) {
    if (bid == 0 && di == 0 && err) atomicOr(err, SPLASH_DEV_BAD_TABLE);
    P = cap;
  }
  for (int64_t u = bid; u < P; u += nb) {
    const int64_t k = rep_list[u];
    const int64_t row = part_row[k];
    const int32_t bm = (int32_t)(row / m.nq);
    const int64_t r = row % m.nq, c = part_col[k];
    const bool sorted = m.qseg != nullptr ? stage_kv_ids(m, bm, c, s_kv) : false;
    if (act) {
      const int64_t i = r * m.bq + di;
      const int32_t sq = q_segment(m, bm, i);
      int32_t ra = 0, rb = -1;
      if (sorted) sorted_run(s_kv, block_keys(m, c), sq, ra, rb);
      uint32_t *bits = pattern_bits + (u * m.bq + di) * words;
      for (int32_t w = 0; w < words; ++w)
        bits[w] = m.qseg != nullptr ? row_word_staged(m, i, sq, c * m.bk, c * m.bk + w * 32, s_kv, sorted, ra, rb)
                                    : row_word(m, bm, i, sq, c * m.bk + w * 32);
    }
    if (m.qseg != nullptr) __syncthreads();  // s_kv is restaged for the next pattern
  }
}

__global__ void materialize_kernel(DevMask m, const unsigned long long *counters, int64_t cap,
                                   const int32_t *rep_list, const int32_t *part_row,
                                   const int32_t *part_col, uint32_t *pattern_bits, uint32_t *err) {
  materialize_body(m, counters, cap, rep_list, part_row, part_col, pattern_bits, err, blockIdx.x, gridDim.x);
}

// ---------------------------------------------------------------- row order
// Rows sorted by descending active-block count, ties in ascending row order
// (a stable counting sort): the attention kernel takes its work longest row
// first.  One CTA; `hist` is a global scratch array of nk+1 counters.
constexpr int kOrderSmem = 4096;  // bins and rows the row order keeps in shared memory

__device__ __forceinline__ void row_order_body(int64_t R, int64_t nk, const int32_t *row_cnt_g, int32_t *hist_g,
                                               int32_t *row_order) {
  __shared__ int buf[33];
  __shared__ int s_hist[kOrderSmem], s_rows[kOrderSmem];
  // bins and counts in shared memory when they fit (the global scratch otherwise)
  const bool in_smem = nk + 1 <= kOrderSmem && R <= kOrderSmem;
  int32_t *hist = in_smem ? s_hist : hist_g;
  const int32_t *row_cnt = in_smem ? s_rows : row_cnt_g;
  for (int64_t b = threadIdx.x; b <= nk; b += blockDim.x) hist[b] = 0;
  if (in_smem)
    for (int64_t x = threadIdx.x; x < R; x += blockDim.x) s_rows[x] = row_cnt_g[x];
  __syncthreads();
  for (int64_t x = threadIdx.x; x < R; x += blockDim.x) atomicAdd(&hist[row_cnt[x]], 1);
  __syncthreads();
  // exclusive scan over bins nk, nk-1, ..., 0 (descending counts first)
  int carry = 0;
  for (int64_t base = 0; base <= nk; base += blockDim.x) {
    const int64_t x = base + threadIdx.x;
    const int64_t bin = nk - x;
    const int h = x <= nk ? hist[bin] : 0;
    int tot;
    const int ex = block_excl_scan(h, tot, buf);
    if (x <= nk) hist[bin] = carry + ex;
    carry += tot;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const unsigned lt = (1u << lane) - 1u;
    for (int64_t base = 0; base < R; base += 32) {
      const int64_t x = base + lane;
      const bool valid = x < R;
      const int c = valid ? row_cnt[x] : -1 - lane;  // invalid lanes get unique keys
      const unsigned peers = __match_any_sync(0xffffffffu, c);
      const int pos = valid ? hist[c] + __popc(peers & lt) : 0;
      __syncwarp();
      if (valid) {
        row_order[pos] = (int32_t)x;
        if ((peers & lt) == 0) hist[c] += __popc(peers);
      }
      __syncwarp();
    }
  }
}

// row_ptr and the partial offsets, then the row order, in one CTA (both need
// only the per-row counts).
__global__ void __launch_bounds__(1024)
scan_order_kernel(int64_t R, int64_t nk, const int32_t *row_cnt, const int32_t *row_pcnt, int32_t *row_ptr,
                  int32_t *prow_ptr, unsigned long long *counters, int32_t *hist, int32_t *row_order) {
  scan_rows_body(R, row_cnt, row_pcnt, row_ptr, prow_ptr, counters);
  __syncthreads();
  row_order_body(R, nk, row_cnt, hist, row_order);
}

// ---------------------------------------------------------------- one-launch build
// The pipeline K1 .. materialize as one persistent kernel: every CTA runs each
// phase on its share of the work (the bodies above with a grid stride; the
// row and pattern-index scans are counted per warp up to the limits below,
// and beyond them run on CTA 0), and a grid-wide barrier separates the
// phases.  It replaces nine dependent launches, each of which costs a few
// microseconds of launch and drain latency at these sizes.  The launch is cooperative, so
// that every CTA is resident and the barrier can complete; the barrier itself
// is this file's own, with a bounded wait: a CTA that waits longer than
// kGridBarrierNs sets SPLASH_DEV_TIMEOUT_BUILD and stops (the others then
// time out at their next barrier too), so the kernel always ends.
constexpr int kGridThreads = 256;
constexpr uint64_t kGridBarrierNs = 2000000000ull;  // 2 s
constexpr int64_t kGridMaxBlocks = (int64_t)1 << 22;  // larger tables take the launch chain
constexpr int64_t kGridMaxPartials = 65536;
constexpr int64_t kGridRowwiseMaxRows = 2048;  // rows a warp scans to place its own row
// Up to this many partial blocks the first occurrences are also marked in a
// bitmap (after the barrier's two words), from which each warp counts its
// block's pattern index itself; larger tables take the single-CTA scan.
constexpr int64_t kGridWarpScanMaxPartials = 2048;
constexpr int kGridSyncWords = 2 + (int)(kGridWarpScanMaxPartials / 32);

struct GridArgs {
  int32_t *qsum, *kvsum;
  int8_t *block_mask;
  int32_t *row_cnt, *row_pcnt, *row_ptr, *prow_ptr, *row_hist, *row_order;
  int32_t *active_rows, *active_cols, *mask_next;
  uint8_t *bounds_start, *bounds_end;
  int32_t *part_row, *part_col, *part_g, *part_rep, *part_pidx, *rep_list;
  uint64_t *part_hash;
  unsigned long long *counters;
  uint32_t *pattern_bits;
  int64_t cap_patterns, NB;
  // each partial block's mask words (the layout of pattern_bits, indexed by
  // partial block), and a hash table: key = content hash (0 = empty slot),
  // value = the smallest partial index with that hash
  uint32_t *part_bits;
  unsigned long long *ht_key;
  int32_t *ht_val;
  int64_t ht_mask;  // table size - 1 (a power of two, at least twice the partial blocks)
  // [kGridSyncWords], zero at launch: the grid barrier's arrival counter, a
  // spare word, and the first-occurrence bitmap (bit k: partial block k is
  // the first of its content, for k < kGridWarpScanMaxPartials)
  unsigned int *sync;
  uint32_t *err;
};

// Warp-level K4 phases of the one-launch build.  hash: the warp computes the
// mask words of partial block k once (into part_bits), their content hash,
// and enters the hash in the table with the block's index (the table keeps
// the smallest).  dedup: the smallest index c with the same hash is the first
// block of identical content whenever the two blocks' words are equal (all
// blocks of equal content have equal hashes); otherwise (a hash collision)
// the earlier blocks of equal hash are compared in ascending order.  So the
// result is exact, and the usual cost is one comparison per block.
__device__ __forceinline__ void stage_kv_ids_warp(const DevMask &m, int32_t bm, int64_t c, int32_t *s_kv, bool &sorted) {
  const int lane = threadIdx.x & 31;
  const int64_t n = min((int64_t)m.bk, m.Lk - c * m.bk);
  for (int32_t t = lane; t < m.bk; t += 32) {
    const int64_t j = c * m.bk + t;
    s_kv[t] = j < m.Lk ? m.kvseg[(int64_t)bm * m.Lk + j] : 0;
  }
  __syncwarp();
  bool ok = true;
  for (int32_t t = lane; t + 1 < n; t += 32) ok &= s_kv[t] <= s_kv[t + 1];
  sorted = __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ unsigned long long table_key(uint64_t h) { return h != 0 ? h : 1ull; }


__device__ void hash_warp(const DevMask &m, const GridArgs &a, int64_t k, int32_t *s_kv) {
  const int lane = threadIdx.x & 31;
  const int32_t words = m.bk / 32;
  const int64_t row = a.part_row[k];
  const int32_t bm = (int32_t)(row / m.nq);
  const int64_t r = row % m.nq, c = a.part_col[k];
  // band-only whole blocks: the diagonal offset identifies the content
  // exactly (no words are stored; materialize computes them)
  const bool by_offset = m.qseg == nullptr && !m.ragged;
  // the query IDs of this lane's rows (di = lane + 32 x, bq <= 256) are
  // loaded together, beside the key IDs, instead of one per row
  int32_t sqr[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) sqr[x] = (lane + 32 * x < m.bq) ? q_segment_early(m, bm, r * m.bq + lane + 32 * x) : 0;
  bool sorted = false;
  if (m.qseg != nullptr) stage_kv_ids_warp(m, bm, c, s_kv, sorted);
  uint32_t *dst = a.part_bits + k * m.bq * words;
  uint64_t t = 0;
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    const int32_t di = lane + 32 * x;
    if (di >= m.bq || by_offset) break;
    const int64_t i = r * m.bq + di;
    const int32_t sq = sqr[x];
    int32_t ra = 0, rb = -1;
    if (sorted) sorted_run_warp(s_kv, block_keys(m, c), sq, ra, rb);  // warp-uniform
    uint64_t h = kHashBasis;
    for (int32_t w = 0; w < words; ++w) {
      const uint32_t wv = m.qseg != nullptr
                              ? row_word_staged(m, i, sq, c * m.bk, c * m.bk + w * 32, s_kv, sorted, ra, rb)
                              : row_word(m, bm, i, sq, c * m.bk + w * 32);
      dst[di * words + w] = wv;
      h = hash_step(h, wv);
    }
    t += row_hash_term(h, di);
  }
  t = warp_sum_u64(t);
  const unsigned long long key =
      by_offset ? ((unsigned long long)(c * m.bk - r * m.bq) ^ 0x8000000000000000ull) : table_key(t);
  if (lane == 0) {
    a.part_hash[k] = key;
    int64_t slot = (int64_t)(key & (unsigned long long)a.ht_mask);
    for (int64_t probe = 0; probe <= a.ht_mask; ++probe) {  // the table is at most half full
      const unsigned long long prev = atomicCAS(&a.ht_key[slot], 0ull, key);
      if (prev == 0ull || prev == key) {
        atomicMin(&a.ht_val[slot], (int32_t)k);
        break;
      }
      slot = (slot + 1) & a.ht_mask;
    }
  }
  __syncwarp();  // s_kv is restaged for the warp's next block
}

// Whether partial blocks ka and kb have equal words (warp-wide result).
__device__ __forceinline__ bool words_equal(const DevMask &m, const GridArgs &a, int64_t ka, int64_t kb) {
  const int64_t n = (int64_t)m.bq * (m.bk / 32);
  const uint32_t *pa = a.part_bits + ka * n, *pb = a.part_bits + kb * n;
  bool same = true;
  for (int64_t x = threadIdx.x & 31; x < n; x += 32) same &= pa[x] == pb[x];
  return __all_sync(0xffffffffu, same);
}

__device__ void dedup_warp(const DevMask &m, const GridArgs &a, int64_t k) {
  const int lane = threadIdx.x & 31;
  const unsigned long long key = a.part_hash[k];
  const bool by_offset = m.qseg == nullptr && !m.ragged;
  int64_t slot = (int64_t)(key & (unsigned long long)a.ht_mask);
  int64_t c = k;
  for (int64_t probe = 0; probe <= a.ht_mask; ++probe) {
    if (a.ht_key[slot] == key) {
      c = a.ht_val[slot];
      break;
    }
    slot = (slot + 1) & a.ht_mask;
  }
  int64_t rep = k;
  if (c < k && (by_offset || words_equal(m, a, k, c))) {
    rep = c;
  } else if (c < k) {
    // a hash collision: earlier blocks of equal hash, ascending
    for (int64_t base = 0; base < k && rep == k; base += 32) {
      const int64_t kp = base + lane;
      unsigned cand = __ballot_sync(0xffffffffu, kp < k && a.part_hash[kp] == key);
      while (cand && rep == k) {
        const int64_t kc = base + (__ffs(cand) - 1);
        cand &= cand - 1u;
        if (words_equal(m, a, k, kc)) rep = kc;
      }
    }
  }
  if (lane == 0) {
    a.part_rep[k] = (int32_t)rep;
    if (rep == k && k < kGridWarpScanMaxPartials) atomicOr(a.sync + 2 + (k >> 5), 1u << (k & 31));
  }
}

__device__ __forceinline__ uint64_t build_clock_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Grid-wide barrier with a bounded wait; returns false (to every thread of
// the CTA) when it gave up.  One arrival counter that only grows during the
// launch (cleared before it): barrier number n of the launch completes when
// the counter reaches n * gridDim.x.  Thread 0 arrives with a release
// reduction after the CTA's barrier (so the CTA's writes before it are
// released) and polls with acquire loads (so every write released before the
// last arrival is visible to the CTA after it).
__device__ __forceinline__ void grid_arrive_release(unsigned int *counter) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
}
__device__ __forceinline__ unsigned int grid_load_acquire(const unsigned int *counter) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
  return v;
}

__device__ bool grid_barrier(unsigned int *sync, uint32_t *err, unsigned int &nbar) {
  __shared__ int s_ok;
  ++nbar;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int target = nbar * gridDim.x;
    grid_arrive_release(sync);
    bool ok = true;
    const uint64_t t0 = build_clock_ns();
    while (grid_load_acquire(sync) < target) {
      if (build_clock_ns() - t0 > kGridBarrierNs) {
        ok = false;
        atomicOr(err, SPLASH_DEV_TIMEOUT_BUILD);
        break;
      }
    }
    s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  return s_ok != 0;
}

__global__ void __launch_bounds__(kGridThreads, 2) build_grid_kernel(DevMask m, GridArgs a) {
  const int64_t bid = blockIdx.x, nb = gridDim.x;
  const int64_t R = (int64_t)m.nbm * m.nq;
  // warp index for the per-warp loops, CTA-minor: consecutive work units go
  // to different CTAs (so to every SM) before a CTA's second warp takes one
  const int64_t warps = nb * (kGridThreads / 32), gw = (int64_t)(threadIdx.x >> 5) * nb + bid;
  const bool seg = m.qseg != nullptr;
  unsigned int nbar = 0;  // grid barriers passed
  // K1: totals and row counters cleared; segment summaries
  if (bid == 0 && threadIdx.x < 8) a.counters[threadIdx.x] = 0ull;
  if (seg) {
    for (int64_t w = gw; w < (m.nq + m.nk) * m.nbm; w += warps)
      seg_summary_warp(m, w % (m.nq + m.nk), (int32_t)(w / (m.nq + m.nk)), a.qsum, a.kvsum, a.row_cnt, a.row_pcnt);
  } else {
    for (int64_t x = bid * kGridThreads + threadIdx.x; x < R; x += nb * kGridThreads) {
      a.row_cnt[x] = 0;
      a.row_pcnt[x] = 0;
    }
  }
  for (int64_t x = bid * kGridThreads + threadIdx.x; x <= a.ht_mask; x += nb * kGridThreads) {
    a.ht_key[x] = 0ull;
    a.ht_val[x] = INT_MAX;
  }
  if (!grid_barrier(a.sync, a.err, nbar)) return;
  // K2: classes, row counts, allowed pairs; undecided blocks to the deferred list
  {
    const int64_t xcs = (m.nk + kGridThreads - 1) / kGridThreads;
    for (int64_t v = bid; v < xcs * R; v += nb) {
      const int64_t row = v / xcs, xc = v - row * xcs;
      classify_body(m, xc, row % m.nq, (int32_t)(row / m.nq), a.qsum, a.kvsum, a.block_mask, a.row_cnt, a.row_pcnt,
                    a.counters, seg ? a.rep_list : nullptr, a.NB);
    }
  }
  if (!grid_barrier(a.sync, a.err, nbar)) return;
  if (seg) {
    // the deferred list lives in rep_list, which the last phase fills later
    count_deferred_body(m, a.rep_list, a.NB, a.block_mask, a.row_cnt, a.row_pcnt, a.counters, bid, nb);
    if (!grid_barrier(a.sync, a.err, nbar)) return;
  }
  // K3: row_ptr, partial offsets, row order and the active lists
  {
    __shared__ int32_t s_kv[kGridThreads / 32][128];  // a warp's key segment IDs (bk <= 128)
    int32_t *kv = s_kv[threadIdx.x >> 5];
    if (R <= kGridRowwiseMaxRows) {
      // one warp per row: its offsets are the sums over the rows before it,
      // its place in the row order the number of rows with more active
      // blocks or as many and a smaller index (a stable sort by count)
      const int lane = threadIdx.x & 31;
      for (int64_t row = gw; row < R; row += warps) {
        const int32_t my = a.row_cnt[row], myp = a.row_pcnt[row];
        int32_t ga = 0, gp = 0, ahead = 0;
        for (int64_t x = lane; x < R; x += 32) {
          const int32_t cx = a.row_cnt[x];
          if (x < row) {
            ga += cx;
            gp += a.row_pcnt[x];
          }
          ahead += (cx > my || (cx == my && x < row)) ? 1 : 0;
        }
        for (int off = 16; off; off >>= 1) {
          ga += __shfl_xor_sync(0xffffffffu, ga, off);
          gp += __shfl_xor_sync(0xffffffffu, gp, off);
          ahead += __shfl_xor_sync(0xffffffffu, ahead, off);
        }
        if (lane == 0) {
          a.row_ptr[row] = ga;
          a.prow_ptr[row] = gp;
          a.row_order[ahead] = (int32_t)row;
          if (my > 0) atomicMax(&a.counters[4], (unsigned long long)my);
          if (row == R - 1) {
            a.row_ptr[R] = ga + my;
            a.prow_ptr[R] = gp + myp;
            a.counters[0] = (unsigned long long)(ga + my);
            a.counters[1] = (unsigned long long)(gp + myp);
          }
        }
        compact_warp(m, row, ga, ga + my, gp, a.block_mask, a.active_rows, a.active_cols, a.mask_next,
                     a.bounds_start, a.bounds_end, a.part_row, a.part_col, a.part_g);
      }
    } else {
      if (bid == 0) {
        scan_rows_body(R, a.row_cnt, a.row_pcnt, a.row_ptr, a.prow_ptr, a.counters);
        __syncthreads();
        row_order_body(R, m.nk, a.row_cnt, a.row_hist, a.row_order);
      }
      if (!grid_barrier(a.sync, a.err, nbar)) return;
      for (int64_t row = gw; row < R; row += warps)
        compact_warp(m, row, a.row_ptr[row], a.row_ptr[row + 1], a.prow_ptr[row], a.block_mask, a.active_rows,
                     a.active_cols, a.mask_next, a.bounds_start, a.bounds_end, a.part_row, a.part_col, a.part_g);
    }
    if (!grid_barrier(a.sync, a.err, nbar)) return;
    // words and hashes (one warp per partial block)
    for (int64_t k = gw; k < (int64_t)a.counters[1]; k += warps) hash_warp(m, a, k, kv);
    if (!grid_barrier(a.sync, a.err, nbar)) return;
    // first occurrences (one warp per partial block)
    const int64_t Ap = (int64_t)a.counters[1];
    for (int64_t k = gw; k < Ap; k += warps) dedup_warp(m, a, k);
  }
  if (!grid_barrier(a.sync, a.err, nbar)) return;
  // Pattern indices: the number of first occurrences before each one, and
  // their total P.  Up to kGridWarpScanMaxPartials partial blocks every warp
  // counts them in the bitmap itself (two words per lane), so neither a
  // single-CTA scan nor a grid barrier comes before the last phase.
  const int64_t Ap = (int64_t)a.counters[1];
  const bool bitmap = Ap <= kGridWarpScanMaxPartials;
  const unsigned int *first = a.sync + 2;
  const int lane = threadIdx.x & 31;
  if (!bitmap) {
    if (bid == 0) scan_reps_body(a.counters, a.part_rep, a.part_pidx);
    if (!grid_barrier(a.sync, a.err, nbar)) return;
    if (bid == 0 && threadIdx.x == 0 && (int64_t)a.counters[2] > a.cap_patterns)
      atomicOr(a.err, SPLASH_DEV_BAD_TABLE);
  } else if (gw == 0) {
    const int tot = __reduce_add_sync(0xffffffffu, __popc(first[lane]) + __popc(first[lane + 32]));
    if (lane == 0) {
      a.counters[2] = (unsigned long long)tot;
      if (tot > a.cap_patterns) atomicOr(a.err, SPLASH_DEV_BAD_TABLE);
    }
  }
  {
    // one warp per partial block: its mask_next entry, and for a first
    // occurrence its place in the pattern list and its pattern
    const int32_t words = m.bk / 32;
    const int64_t n = (int64_t)m.bq * words;
    const bool by_offset = m.qseg == nullptr && !m.ragged;
    for (int64_t k = gw; k < Ap; k += warps) {
      const int32_t rep = a.part_rep[k];
      int64_t u;
      if (bitmap) {
        // bits below rep: whole words before word rep / 32, then that word's low bits
        const int wr = rep >> 5;
        const unsigned int lo = first[lane], hi = first[lane + 32];
        const unsigned int below = (1u << (rep & 31)) - 1u;
        const int cnt = (lane < wr ? __popc(lo) : (lane == wr ? __popc(lo & below) : 0)) +
                        (lane + 32 < wr ? __popc(hi) : (lane + 32 == wr ? __popc(hi & below) : 0));
        u = __reduce_add_sync(0xffffffffu, cnt);
      } else {
        u = a.part_pidx[rep];
      }
      if ((threadIdx.x & 31) == 0) {
        a.mask_next[a.part_g[k]] = (int32_t)u;
        if (rep == k) a.rep_list[u] = (int32_t)k;
      }
      if (rep != k || u >= a.cap_patterns) continue;
      uint32_t *dst = a.pattern_bits + u * n;
      if (by_offset) {  // band only: the words in closed form
        const int64_t row = a.part_row[k], c = a.part_col[k];
        const int64_t r = row % m.nq;
        for (int64_t x = threadIdx.x & 31; x < n; x += 32)
          dst[x] = row_word(m, 0, r * m.bq + x / words, 0, c * m.bk + (x % words) * 32);
      } else {
        const uint32_t *src = a.part_bits + k * n;
        for (int64_t x = threadIdx.x & 31; x < n; x += 32) dst[x] = src[x];
      }
    }
  }
}

// ---------------------------------------------------------------- fused build
// The whole pipeline above in one CTA, for band-only masks (no segment IDs)
// with a small table.  Every phase is a loop over the CTA's 1024 threads with
// __syncthreads between phases; the block classes come from the closed form,
// and every intermediate (row counts and offsets, row-order bins, the partial
// blocks' coordinates and diagonal offsets, their representatives, the
// first-occurrence bitmap and the pattern list) stays in shared memory
// (global memory is only written: the table itself).  Partial
// blocks are deduplicated by their diagonal offset d = c*bk - r*bq: under a
// band mask the pattern of a block is {(i', j'): L <= j' - i' <= U} with L, U
// shifted by -d, and for partial blocks (neither empty nor full) the clipped
// interval of diagonals is strictly monotone in d, so equal content <=> equal
// d — the content comparison of the general pipeline is not needed.
constexpr int kSmallThreads = 1024;
constexpr int64_t kSmallMaxRows = 2048;      // R
constexpr int64_t kSmallMaxCols = 2048;      // nk
constexpr int64_t kSmallMaxBlocks = 65536;   // R * nk
constexpr int64_t kSmallMaxPartials = 2048;  // bound on the partial blocks

struct SmallOut {
  int8_t *block_mask;
  int32_t *row_ptr, *row_order;
  int32_t *active_rows, *active_cols, *mask_next;
  uint8_t *bounds_start, *bounds_end;
  unsigned long long *counters;
  uint32_t *pattern_bits;
  int64_t cap_patterns;
  uint32_t *err;
  int32_t max_partials;  // capacity of the shared partial arrays
};

// Dynamic shared memory of build_small_kernel for R rows, nk columns and up to
// max_partials partial blocks.
inline size_t small_smem_bytes(int64_t R, int64_t nk, int64_t max_partials) {
  return sizeof(int32_t) * (size_t)(2 * R + 2 * (R + 1) + (nk + 1)) +
         (sizeof(int64_t) + 5 * sizeof(int32_t)) * (size_t)max_partials + 64;
}

__global__ void __launch_bounds__(kSmallThreads) build_small_kernel(DevMask m, SmallOut o) {
  extern __shared__ __align__(16) uint8_t s_dyn[];
  const int64_t R = m.nq, nk = m.nk, PM = o.max_partials;
  int64_t *s_pd = reinterpret_cast<int64_t *>(s_dyn);                      // [PM] diagonal offsets
  int32_t *s_cnt = reinterpret_cast<int32_t *>(s_pd + PM);                // [R]
  int32_t *s_pcnt = s_cnt + R;                                             // [R]
  int32_t *s_rp = s_pcnt + R;                                              // [R+1]
  int32_t *s_prp = s_rp + R + 1;                                           // [R+1]
  int32_t *s_hist = s_prp + R + 1;                                         // [nk+1]
  int32_t *s_prow = s_hist + nk + 1;                                       // [PM]
  int32_t *s_pcol = s_prow + PM;                                           // [PM]
  int32_t *s_pg = s_pcol + PM;                                             // [PM]
  int32_t *s_prep = s_pg + PM;                                             // [PM]
  int32_t *s_ppidx = s_prep + PM;                                          // [PM] pattern list
  __shared__ int buf_a[33], s_mx[32];
  __shared__ unsigned long long buf_ap[33];
  __shared__ unsigned long long s_allow[32];  // allowed pairs, per warp
  __shared__ unsigned int s_first[kSmallMaxPartials / 32];  // bit k: partial k is a first occurrence
  __shared__ int64_t s_tot[3];  // A, A_p, P
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int64_t A, W;
  band_limits(m, A, W);

  // classes and per-row counts (one warp per row: ballots, no shared-memory
  // atomics on a row's counters), allowed pairs (per warp, summed below)
  for (int x = tid; x < (int)(kSmallMaxPartials / 32); x += kSmallThreads) s_first[x] = 0u;
  for (int64_t r = warp; r < R; r += kSmallThreads / 32) {
    int na = 0, np = 0;
    for (int64_t cb = 0; cb < nk; cb += 32) {
      const int64_t c = cb + lane;
      const int cls = c < nk ? band_block_class(m, A, W, r, c) : 0;
      if (c < nk) o.block_mask[r * nk + c] = (int8_t)cls;
      na += __popc(__ballot_sync(0xffffffffu, cls != 0));
      np += __popc(__ballot_sync(0xffffffffu, cls == 1));
    }
    if (lane == 0) {
      s_cnt[r] = na;
      s_pcnt[r] = np;
    }
  }
  unsigned long long allowed = 0;
  for (int64_t i = tid; i < m.Lq; i += kSmallThreads) allowed += (unsigned long long)band_row_count(m, A, W, i);
  for (int off = 16; off; off >>= 1) allowed += __shfl_xor_sync(0xffffffffu, allowed, off);
  if (lane == 0) s_allow[warp] = allowed;
  __syncthreads();

  // row_ptr (CSR), partial offsets and the longest row: one scan of the two
  // counts packed in 64 bits (each total is at most R * nk <= 2^16)
  int carry_a = 0, carry_p = 0, mx = 0;
  for (int64_t base = 0; base < R; base += kSmallThreads) {
    const int64_t x = base + tid;
    const int a = x < R ? s_cnt[x] : 0, pc = x < R ? s_pcnt[x] : 0;
    mx = max(mx, a);
    unsigned long long tot;
    const unsigned long long ex =
        block_excl_scan64((unsigned long long)a | ((unsigned long long)pc << 32), tot, buf_ap);
    if (x < R) {
      s_rp[x] = carry_a + (int)(ex & 0xffffffffull);
      s_prp[x] = carry_p + (int)(ex >> 32);
      o.row_ptr[x] = s_rp[x];
    }
    carry_a += (int)(tot & 0xffffffffull);
    carry_p += (int)(tot >> 32);
  }
  for (int off = 16; off; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) s_mx[warp] = mx;
  for (int64_t b = tid; b <= nk; b += kSmallThreads) s_hist[b] = 0;
  __syncthreads();
  if (tid == 0) {
    int t = 0;
    unsigned long long allowed_all = 0;
    for (int x = 0; x < kSmallThreads / 32; ++x) {
      t = max(t, s_mx[x]);
      allowed_all += s_allow[x];
    }
    s_rp[R] = carry_a;
    s_prp[R] = carry_p;
    o.row_ptr[R] = carry_a;
    o.counters[0] = (unsigned long long)carry_a;
    o.counters[1] = (unsigned long long)carry_p;
    o.counters[3] = allowed_all;
    o.counters[4] = (unsigned long long)t;
    s_tot[0] = carry_a;
    s_tot[1] = carry_p;
  }
  // row order: bins of a stable counting sort, descending counts first
  for (int64_t x = tid; x < R; x += kSmallThreads) atomicAdd(&s_hist[s_cnt[x]], 1);
  __syncthreads();
  int carry = 0;
  for (int64_t base = 0; base <= nk; base += kSmallThreads) {
    const int64_t x = base + tid;
    const int64_t bin = nk - x;
    const int h = x <= nk ? s_hist[bin] : 0;
    int tot;
    const int ex = block_excl_scan(h, tot, buf_a);
    if (x <= nk) s_hist[bin] = carry + ex;
    carry += tot;
  }
  __syncthreads();
  const int64_t Ap = s_tot[1];
  if (Ap > PM) {
    // cannot happen (the host bounds the partial blocks); report, do nothing
    if (tid == 0 && o.err) atomicOr(o.err, SPLASH_DEV_BAD_TABLE);
    return;
  }
  if (warp == 0) {
    // placement in row order (ties in ascending row order)
    const unsigned lt = (1u << lane) - 1u;
    for (int64_t base = 0; base < R; base += 32) {
      const int64_t x = base + lane;
      const bool valid = x < R;
      const int c = valid ? s_cnt[x] : -1 - lane;
      const unsigned peers = __match_any_sync(0xffffffffu, c);
      const int pos = valid ? s_hist[c] + __popc(peers & lt) : 0;
      __syncwarp();
      if (valid) {
        o.row_order[pos] = (int32_t)x;
        if ((peers & lt) == 0) s_hist[c] += __popc(peers);
      }
      __syncwarp();
    }
  } else {
    // active lists (warps 1..31, one row at a time); classes recomputed
    const unsigned lt = (1u << lane) - 1u;
    for (int64_t row = warp - 1; row < R; row += kSmallThreads / 32 - 1) {
      const int32_t g0 = s_rp[row], gend = s_rp[row + 1];
      int32_t g = g0, k = s_prp[row];
      for (int64_t cb = 0; cb < nk; cb += 32) {
        const int64_t c = cb + lane;
        const int cls = c < nk ? band_block_class(m, A, W, row, c) : 0;
        const unsigned act = __ballot_sync(0xffffffffu, cls != 0);
        const unsigned par = __ballot_sync(0xffffffffu, cls == 1);
        if (cls != 0) {
          const int32_t pos = g + __popc(act & lt);
          o.active_rows[pos] = (int32_t)row;
          o.active_cols[pos] = (int32_t)c;
          o.bounds_start[pos] = (uint8_t)(pos == g0);
          o.bounds_end[pos] = (uint8_t)(pos == gend - 1);
          if (cls == 1) {
            const int32_t kk = k + __popc(par & lt);
            s_prow[kk] = (int32_t)row;
            s_pcol[kk] = (int32_t)c;
            s_pg[kk] = pos;
            s_pd[kk] = c * m.bk - row * m.bq;
          } else {
            o.mask_next[pos] = -1;
          }
        }
        g += __popc(act);
        k += __popc(par);
      }
    }
  }
  __syncthreads();

  // first partial with the same diagonal offset (one warp per partial)
  for (int32_t k = warp; k < (int32_t)Ap; k += kSmallThreads / 32) {
    const int64_t d = s_pd[k];
    int32_t rep = k;
    for (int32_t base = 0; base < k; base += 32) {
      const int32_t kp = base + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, kp < k && s_pd[kp] == d);
      if (hit) {
        rep = base + __ffs(hit) - 1;
        break;
      }
    }
    if (lane == 0) {
      s_prep[k] = rep;
      if (rep == k) atomicOr(&s_first[k >> 5], 1u << (k & 31));
    }
  }
  __syncthreads();
  // pattern index of partial k's content: the first occurrences before its
  // representative, counted in the bitmap; the mask_next entry, and for a
  // first occurrence its place in the pattern list (s_ppidx: partial index
  // of pattern u)
  for (int64_t k = tid; k < Ap; k += kSmallThreads) {
    const int32_t rep = s_prep[k];
    int32_t u = __popc(s_first[rep >> 5] & ((1u << (rep & 31)) - 1u));
    for (int32_t w = 0; w < (rep >> 5); ++w) u += __popc(s_first[w]);
    o.mask_next[s_pg[k]] = u;
    if (rep == k) s_ppidx[u] = (int32_t)k;
  }
  if (tid == 0) {
    int32_t P = 0;
    for (int32_t w = 0; w < (int32_t)((Ap + 31) >> 5); ++w) P += __popc(s_first[w]);
    o.counters[2] = (unsigned long long)P;
    s_tot[2] = P;
  }
  __syncthreads();
  // the patterns, bit-packed (word w of row di of pattern u holds keys
  // 32w .. 32w+31): one word per thread, consecutive threads on consecutive words
  int64_t P = s_tot[2];
  if (P > o.cap_patterns) {
    if (tid == 0 && o.err) atomicOr(o.err, SPLASH_DEV_BAD_TABLE);
    P = o.cap_patterns;
  }
  const int32_t words = m.bk / 32, per_pattern = m.bq * words;
  for (int64_t x = tid; x < P * per_pattern; x += kSmallThreads) {
    const int64_t u = x / per_pattern;
    const int32_t rem = (int32_t)(x - u * per_pattern), di = rem / words, w = rem - di * words;
    const int64_t k = s_ppidx[u];
    o.pattern_bits[x] = row_word(m, 0, (int64_t)s_prow[k] * m.bq + di, 0, (int64_t)s_pcol[k] * m.bk + w * 32);
  }
}

// ---------------------------------------------------------------- host side
template <typename T>
cudaError_t grow(T *&p, int64_t have, int64_t need) {
  if (p != nullptr && have >= need) return cudaSuccess;
  if (p) cudaFree(p);
  p = nullptr;
  return cudaMalloc(&p, sizeof(T) * (size_t)std::max<int64_t>(need, 1));
}

template <typename T>
cudaError_t grow_host(T *&p, int64_t have, int64_t need) {
  if (p != nullptr && have >= need) return cudaSuccess;
  if (p) cudaFreeHost(p);
  p = nullptr;
  return cudaMallocHost(&p, sizeof(T) * (size_t)std::max<int64_t>(need, 1));
}

// Largest pattern buffer the build reserves from a bound instead of waiting
// for the exact pattern count.
constexpr int64_t kPatternBudgetBytes = (int64_t)256 << 20;

// Blocks of one table batch row that the band part of the mask (causal and
// window bounds, and the padding of a ragged grid) leaves non-empty; the
// same closed form as band_block_class, one row at a time: for the rows
// r0 .. r1 (clipped to Lq) the non-empty key blocks are those with
// c0 <= r1 + A and c1 >= r0 - W, a contiguous range.
int64_t band_active_blocks(const splash_mask_spec *spec, int64_t Lq, int64_t Lk, int32_t bq, int32_t bk, int64_t nq,
                           int64_t nk) {
  const int64_t kInf = (int64_t)1 << 60;
  int64_t A = kInf, W = spec->window_left >= 0 ? spec->window_left : kInf;
  if (spec->causal) A = 0;
  if (spec->window_right >= 0) A = std::min(A, spec->window_right);
  int64_t total = 0;
  for (int64_t r = 0; r < nq; ++r) {
    const int64_t r0 = r * bq, r1 = std::min(r0 + bq - 1, Lq - 1);
    // c * bk <= r1 + A  and  min(c * bk + bk - 1, Lk - 1) >= r0 - W
    const int64_t hi = A >= kInf ? nk - 1 : std::min(nk - 1, (r1 + A) / bk);
    int64_t lo = 0;
    if (W < kInf && r0 - W > 0) lo = (r0 - W) / bk;  // block c holds key r0 - W when c = floor((r0 - W) / bk)
    if (r0 - W > Lk - 1 && W < kInf) lo = nk;         // every key is left of the window
    if (hi >= lo) total += hi - lo + 1;
  }
  return std::max<int64_t>(total, 1);
}

splash_status map_alloc(cudaError_t e) {
  if (e == cudaSuccess) return SPLASH_OK;
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? SPLASH_ERR_OOM : SPLASH_ERR_CUDA;
}

}  // namespace

void splash_mask_info_free_transposed(splash_mask_info *mi) {
  void *dev[] = {mi->t_col_cnt, mi->t_col_ptr, mi->t_col_rows, mi->t_col_next, mi->t_pattern_bits};
  for (void *p : dev)
    if (p) cudaFree(p);
  mi->t_col_cnt = mi->t_col_ptr = mi->t_col_rows = mi->t_col_next = nullptr;
  mi->t_pattern_bits = nullptr;
  mi->t_cap_cols = mi->t_cap_active = mi->t_cap_patterns = 0;
  mi->t_gen = 0;
}

void splash_mask_info_free_buffers(splash_mask_info *mi) {
  splash_mask_info_free_transposed(mi);
  void *dev[] = {mi->block_mask, mi->row_ptr, mi->active_rows, mi->active_cols, mi->mask_next,
                 mi->bounds_start, mi->bounds_end, mi->pattern_bits, mi->row_order,
                 mi->row_cnt, mi->row_pcnt, mi->prow_ptr, mi->seg_summary, mi->part_row,
                 mi->part_col, mi->part_g, mi->part_hash, mi->part_rep, mi->part_pidx,
                 mi->rep_list, mi->counters, mi->row_hist, mi->grid_sync, mi->part_bits,
                 mi->ht_key, mi->ht_val};
  for (void *p : dev)
    if (p) cudaFree(p);
  void *host[] = {mi->h_counters};
  for (void *p : host)
    if (p) cudaFreeHost(p);
  if (mi->counts_ready) cudaEventDestroy(mi->counts_ready);
  if (mi->t_ready) cudaEventDestroy(mi->t_ready);
  const int device = mi->device;
  *mi = splash_mask_info();
  mi->device = device;
}

splash_status splash_mask_info_build_into(splash_mask_info *mi, const splash_mask_spec *spec,
                                          int64_t Lq, int64_t Lk, int32_t bq, int32_t bk,
                                          cudaStream_t stream) {
  const bool seg = spec->q_segment_ids != nullptr;
  const int32_t nbm = seg ? spec->batch : 1;
  const int64_t nq = (Lq + bq - 1) / bq, nk = (Lk + bk - 1) / bk, R = (int64_t)nbm * nq, NB = R * nk;
  const bool ragged = (Lq % bq) != 0 || (Lk % bk) != 0;
  ++mi->build_gen;  // any column-major copy of the previous table is stale

  // -- buffers (reused when large enough) --
  splash_status st;
  if ((st = map_alloc(grow(mi->block_mask, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->active_rows, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->active_cols, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->mask_next, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->bounds_start, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->bounds_end, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->part_row, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->part_col, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->part_g, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->part_hash, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->part_rep, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->part_pidx, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->rep_list, mi->cap_blocks, NB))) != SPLASH_OK) return st;
  mi->cap_blocks = std::max(mi->cap_blocks, NB);
  if ((st = map_alloc(grow(mi->row_ptr, mi->cap_rows, R + 1))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->prow_ptr, mi->cap_rows, R + 1))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->row_cnt, mi->cap_rows, R + 1))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->row_pcnt, mi->cap_rows, R + 1))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow(mi->row_order, mi->cap_rows, R + 1))) != SPLASH_OK) return st;
  mi->cap_rows = std::max(mi->cap_rows, R + 1);
  if ((st = map_alloc(grow(mi->row_hist, mi->cap_hist, nk + 1))) != SPLASH_OK) return st;
  mi->cap_hist = std::max(mi->cap_hist, nk + 1);
  const int64_t nseg = seg ? 2 * (R + (int64_t)nbm * nk) : 2;
  if ((st = map_alloc(grow(mi->seg_summary, mi->cap_seg, nseg))) != SPLASH_OK) return st;
  mi->cap_seg = std::max(mi->cap_seg, nseg);
  if ((st = map_alloc(grow(mi->counters, mi->counters ? 8 : 0, 8))) != SPLASH_OK) return st;
  if ((st = map_alloc(grow_host(mi->h_counters, mi->h_counters ? 8 : 0, 8))) != SPLASH_OK) return st;

  mi->batch_rows = nbm;
  mi->Lq = Lq;
  mi->Lk = Lk;
  mi->nq = nq;
  mi->nk = nk;
  mi->bq = bq;
  mi->bk = bk;
  mi->causal = spec->causal;
  mi->window_left = spec->window_left;
  mi->window_right = spec->window_right;
  mi->has_segments = seg;
  mi->num_active = mi->num_partial = mi->num_patterns = mi->allowed_pairs = 0;

  DevMask m;
  m.causal = spec->causal;
  m.wl = spec->window_left;
  m.wr = spec->window_right;
  m.qseg = spec->q_segment_ids;
  m.kvseg = seg ? (spec->kv_segment_ids ? spec->kv_segment_ids : spec->q_segment_ids) : nullptr;
  m.Lq = Lq;
  m.Lk = Lk;
  m.nq = nq;
  m.nk = nk;
  m.bq = bq;
  m.bk = bk;
  m.nbm = nbm;
  m.ragged = ragged ? 1 : 0;

  int dev = 0, sms = 148;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  SPLASH_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));

  // a previous asynchronous build, possibly on another stream, may still be
  // running on the same buffers: keep it ordered before this one
  // (not while the stream is being captured: a graph cannot wait on work
  // outside it, and its own nodes already order a captured rebuild)
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  SPLASH_CUDA_TRY(cudaStreamIsCapturing(stream, &capturing));
  if (capturing == cudaStreamCaptureStatusNone && mi->counts_pending && !mi->counts_captured && mi->counts_ready)
    SPLASH_CUDA_TRY(cudaStreamWaitEvent(stream, mi->counts_ready, 0));

  uint32_t *err = splash_device_error_word(mi->device);
  // -- pattern buffer (bit-packed patterns, bq * bk / 8 bytes each).  Without
  // segment IDs a q-block row has at most 2 * (ceil((bq-1)/bk) + 1) partial
  // blocks (a block is partial only if one of the two band edges sweeps
  // through it); a ragged grid adds at most the last column's block of every
  // row and the whole last row.  With segment IDs every pattern belongs to an
  // active block, and segments only remove pairs, so P is at most the number
  // of blocks the band alone leaves non-empty (counted here in closed form).
  // When that bound fits the budget the build runs without a host wait and
  // the totals are read when asked for; otherwise it waits once for P.
  const int64_t per_row = 2 * ((bq - 1 + bk - 1) / bk + 1);
  const int64_t p_bound =
      seg ? (int64_t)nbm * band_active_blocks(spec, Lq, Lk, bq, bk, nq, nk)
          : std::min<int64_t>(R * per_row + (ragged ? R + nk : 0), NB);
  const int64_t pattern_bytes = (int64_t)bq * bk / 8;
  const bool async = p_bound * pattern_bytes <= kPatternBudgetBytes;
  auto reserve_patterns = [&](int64_t P_cap) -> splash_status {
    if (P_cap <= 0 || mi->cap_patterns >= P_cap) return SPLASH_OK;
    if (mi->pattern_bits) cudaFree(mi->pattern_bits);
    mi->pattern_bits = nullptr;
    mi->cap_patterns = 0;
    splash_status s2;
    if ((s2 = map_alloc(cudaMalloc(&mi->pattern_bits, (size_t)P_cap * pattern_bytes))) != SPLASH_OK) return s2;
    mi->cap_patterns = P_cap;
    return SPLASH_OK;
  };
  // the totals stay on the device; splash_mask_info_sync_counts copies them
  // once this event has completed
  auto finish_async = [&]() -> splash_status {
    mi->counts_pending = true;
    mi->counts_captured = capturing != cudaStreamCaptureStatusNone;
    if (mi->counts_captured) return SPLASH_OK;  // replays are ordered by the caller
    if (mi->counts_ready == nullptr)
      SPLASH_CUDA_TRY(cudaEventCreateWithFlags(&mi->counts_ready, cudaEventDisableTiming));
    SPLASH_CUDA_TRY(cudaEventRecord(mi->counts_ready, stream));
    return SPLASH_OK;
  };

  if (async && !seg && !ragged && R <= kSmallMaxRows && nk <= kSmallMaxCols && NB <= kSmallMaxBlocks &&
      p_bound <= kSmallMaxPartials) {
    // small band-only table on whole blocks: the whole build is one
    // single-CTA kernel (its diagonal-offset dedup needs whole blocks)
    if ((st = reserve_patterns(p_bound)) != SPLASH_OK) return st;
    SmallOut o;
    o.block_mask = mi->block_mask;
    o.row_ptr = mi->row_ptr;
    o.row_order = mi->row_order;
    o.active_rows = mi->active_rows;
    o.active_cols = mi->active_cols;
    o.mask_next = mi->mask_next;
    o.bounds_start = mi->bounds_start;
    o.bounds_end = mi->bounds_end;
    o.counters = mi->counters;
    o.pattern_bits = mi->pattern_bits;
    o.cap_patterns = mi->cap_patterns;
    o.err = err;
    o.max_partials = (int32_t)p_bound;
    const size_t smem = small_smem_bytes(R, nk, p_bound);
    if (smem > 48 * 1024)
      SPLASH_CUDA_TRY(cudaFuncSetAttribute(build_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)small_smem_bytes(kSmallMaxRows, kSmallMaxCols, kSmallMaxPartials)));
    build_small_kernel<<<1, kSmallThreads, smem, stream>>>(m, o);
    SPLASH_CUDA_TRY(cudaGetLastError());
    splash_count_launches(1);
    return finish_async();
  }

  int32_t *qsum = mi->seg_summary, *kvsum = mi->seg_summary + 2 * R;
  if (async && NB <= kGridMaxBlocks && p_bound <= kGridMaxPartials) {
    // the whole pipeline as one persistent kernel (cooperative launch: every
    // CTA resident; its grid barrier state starts cleared)
    if ((st = reserve_patterns(p_bound)) != SPLASH_OK) return st;
    if (mi->grid_sync == nullptr &&
        (st = map_alloc(cudaMalloc(&mi->grid_sync, kGridSyncWords * sizeof(unsigned int)))) != SPLASH_OK)
      return st;
    // per-partial words (p_bound bounds the partial blocks too) and the hash
    // table, at least twice as large
    const int64_t words_per = (int64_t)bq * (bk / 32);
    if ((st = map_alloc(grow(mi->part_bits, mi->cap_part_bits, p_bound * words_per))) != SPLASH_OK) return st;
    mi->cap_part_bits = std::max(mi->cap_part_bits, p_bound * words_per);
    int64_t ht = 64;
    while (ht < 2 * p_bound) ht <<= 1;
    if ((st = map_alloc(grow(mi->ht_key, mi->cap_ht, ht))) != SPLASH_OK) return st;
    if ((st = map_alloc(grow(mi->ht_val, mi->cap_ht, ht))) != SPLASH_OK) return st;
    mi->cap_ht = std::max(mi->cap_ht, ht);
    // CTAs per SM (at most 2), asked once per device; concurrent first
    // builds on several host threads store the same value
    static std::atomic<int> per_sm[64] = {};
    int cps = dev < 64 ? per_sm[dev].load(std::memory_order_relaxed) : 0;
    if (cps == 0) {
      int n = 0;
      SPLASH_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, build_grid_kernel, kGridThreads, 0));
      cps = std::max(1, std::min(n, 2));
      if (dev < 64) per_sm[dev].store(cps, std::memory_order_relaxed);
    }
    const unsigned grid = (unsigned)(sms * cps);
    GridArgs a;
    a.qsum = qsum;
    a.kvsum = kvsum;
    a.block_mask = mi->block_mask;
    a.row_cnt = mi->row_cnt;
    a.row_pcnt = mi->row_pcnt;
    a.row_ptr = mi->row_ptr;
    a.prow_ptr = mi->prow_ptr;
    a.row_hist = mi->row_hist;
    a.row_order = mi->row_order;
    a.active_rows = mi->active_rows;
    a.active_cols = mi->active_cols;
    a.mask_next = mi->mask_next;
    a.bounds_start = mi->bounds_start;
    a.bounds_end = mi->bounds_end;
    a.part_row = mi->part_row;
    a.part_col = mi->part_col;
    a.part_g = mi->part_g;
    a.part_rep = mi->part_rep;
    a.part_pidx = mi->part_pidx;
    a.rep_list = mi->rep_list;
    a.part_hash = mi->part_hash;
    a.counters = mi->counters;
    a.pattern_bits = mi->pattern_bits;
    a.cap_patterns = mi->cap_patterns;
    a.NB = NB;
    a.part_bits = mi->part_bits;
    a.ht_key = mi->ht_key;
    a.ht_val = mi->ht_val;
    a.ht_mask = ht - 1;
    a.sync = mi->grid_sync;
    a.err = err;
    SPLASH_CUDA_TRY(cudaMemsetAsync(mi->grid_sync, 0, kGridSyncWords * sizeof(unsigned int), stream));
    void *args[] = {&m, &a};
    SPLASH_CUDA_TRY(cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(build_grid_kernel), dim3(grid),
                                                dim3(kGridThreads), args, 0, stream));
    splash_count_launches(1);
    return finish_async();
  }
  if (seg) {
    // (the summary kernel also clears the row counters and the totals)
    dim3 grid((unsigned)((nq + nk + 7) / 8), (unsigned)nbm);
    seg_summary_kernel<<<grid, 256, 0, stream>>>(m, qsum, kvsum, mi->row_cnt, mi->row_pcnt, mi->counters);
  } else {
    SPLASH_CUDA_TRY(cudaMemsetAsync(mi->row_cnt, 0, sizeof(int32_t) * R, stream));
    SPLASH_CUDA_TRY(cudaMemsetAsync(mi->row_pcnt, 0, sizeof(int32_t) * R, stream));
    SPLASH_CUDA_TRY(cudaMemsetAsync(mi->counters, 0, sizeof(unsigned long long) * 8, stream));
  }
  {
    dim3 grid((unsigned)((nk + kClassifyThreads - 1) / kClassifyThreads), (unsigned)nq, (unsigned)nbm);
    classify_kernel<<<grid, kClassifyThreads, 0, stream>>>(m, qsum, kvsum, mi->block_mask, mi->row_cnt,
                                                          mi->row_pcnt, mi->counters, seg ? mi->rep_list : nullptr,
                                                          NB);
  }
  if (seg) {
    // the deferred list lives in rep_list, which scan_finalize_kernel fills later
    count_deferred_kernel<<<sms * 8, kClassifyThreads, 0, stream>>>(m, mi->rep_list, NB, mi->block_mask,
                                                                   mi->row_cnt, mi->row_pcnt, mi->counters);
  }
  scan_order_kernel<<<1, 1024, 0, stream>>>(R, nk, mi->row_cnt, mi->row_pcnt, mi->row_ptr, mi->prow_ptr, mi->counters,
                                            mi->row_hist, mi->row_order);
  compact_kernel<<<(unsigned)((R + 7) / 8), 256, 0, stream>>>(
      m, R, mi->block_mask, mi->row_ptr, mi->prow_ptr, mi->active_rows, mi->active_cols,
      mi->mask_next, mi->bounds_start, mi->bounds_end, mi->part_row, mi->part_col, mi->part_g);
  // one CTA per partial block up to eight per SM (the partial count is a
  // device value; p_bound bounds it from the host)
  const unsigned pgrid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(p_bound, (int64_t)sms * 8));
  partial_hash_kernel<<<pgrid, bq, 0, stream>>>(m, mi->counters, mi->part_row, mi->part_col, mi->part_hash);
  dedup_kernel<<<pgrid, kDedupThreads, 0, stream>>>(m, mi->counters, mi->part_row, mi->part_col, mi->part_hash,
                                                    mi->part_rep);
  scan_finalize_kernel<<<1, 1024, 0, stream>>>(mi->counters, mi->part_g, mi->part_rep, mi->part_pidx, mi->mask_next,
                                               mi->rep_list);
  SPLASH_CUDA_TRY(cudaGetLastError());
  splash_count_launches(seg ? 8 : 6);

  int64_t P_cap;
  if (async) {
    P_cap = p_bound;
  } else {
    SPLASH_CUDA_TRY(cudaMemcpyAsync(mi->h_counters, mi->counters, sizeof(unsigned long long) * 8,
                                    cudaMemcpyDeviceToHost, stream));
    SPLASH_CUDA_TRY(cudaStreamSynchronize(stream));
    P_cap = (int64_t)mi->h_counters[2];
  }
  if ((st = reserve_patterns(P_cap)) != SPLASH_OK) return st;
  if (P_cap > 0) {
    const unsigned grid = (unsigned)std::min<int64_t>(P_cap, async ? sms * 8 : 65535);
    materialize_kernel<<<grid, bq, 0, stream>>>(m, mi->counters, mi->cap_patterns, mi->rep_list, mi->part_row,
                                                mi->part_col, mi->pattern_bits, err);
    SPLASH_CUDA_TRY(cudaGetLastError());
    splash_count_launches(1);
  }
  if (async) {
    if ((st = finish_async()) != SPLASH_OK) return st;
  } else {
    mi->counts_pending = false;
    mi->num_active = (int64_t)mi->h_counters[0];
    mi->num_partial = (int64_t)mi->h_counters[1];
    mi->num_patterns = (int64_t)mi->h_counters[2];
    mi->allowed_pairs = (int64_t)mi->h_counters[3];
    mi->max_row_blocks = (int32_t)mi->h_counters[4];
  }
  return SPLASH_OK;
}

splash_status splash_mask_info_sync_counts(splash_mask_info *mi) {
  if (!mi->counts_pending) return SPLASH_OK;
  // a rebuild captured into a graph recorded no event: wait for the device
  if (mi->counts_captured)
    SPLASH_CUDA_TRY(cudaDeviceSynchronize());
  else
    SPLASH_CUDA_TRY(cudaEventSynchronize(mi->counts_ready));
  SPLASH_CUDA_TRY(cudaMemcpy(mi->h_counters, mi->counters, sizeof(unsigned long long) * 8, cudaMemcpyDeviceToHost));
  mi->num_active = (int64_t)mi->h_counters[0];
  mi->num_partial = (int64_t)mi->h_counters[1];
  mi->num_patterns = (int64_t)mi->h_counters[2];
  mi->allowed_pairs = (int64_t)mi->h_counters[3];
  mi->max_row_blocks = (int32_t)mi->h_counters[4];
  mi->counts_pending = false;
  return SPLASH_OK;
}

// ---------------------------------------------------------------- no-allocation variant
// Block classification (the classify step above, with its per-row counters
// and segment summaries) for callers that must not allocate device memory --
// for example a serving process whose device memory is owned by its own pool
// allocator under a fixed budget, where a cudaMalloc behind the pool's back
// can fail or break its accounting.  The scratch lives in the fixed array
// below instead: it is part of the module image, so every GPU that loads the
// library holds it until the process exits.
//
// Limits: B_mask * nq <= kNoAllocMaxRows and B_mask * nk <= kNoAllocMaxCols.
// Blocks that the segment summaries cannot decide are counted one CTA per
// block while the fixed list has room (kNoAllocMaxDeferred), the rest one
// thread per block.  All calls share the array (it keeps the last call's contents; the counters
// are cleared at the start of every call), so calls that overlap on the GPU
// -- on different streams, or from different host threads -- race.
namespace {
constexpr int64_t kNoAllocMaxRows = 16384;
constexpr int64_t kNoAllocMaxCols = 16384;
constexpr int64_t kNoAllocMaxDeferred = 65536;  // undecided blocks counted one CTA each
struct NoAllocScratch {
  int32_t row_cnt[kNoAllocMaxRows];
  int32_t row_pcnt[kNoAllocMaxRows];
  int32_t qsum[2 * kNoAllocMaxRows];
  int32_t kvsum[2 * kNoAllocMaxCols];
  int32_t deferred[kNoAllocMaxDeferred];
  unsigned long long counters[8];
  unsigned long long totals[4];
};
}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[sizeof(NoAllocScratch)];

namespace {

constexpr int kMaxNoAllocDevices = 64;
NoAllocScratch *g_noalloc_addr[kMaxNoAllocDevices];
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device; resolved once
// per device (the first call on a device does it), under a lock so that
// host threads making their first calls at the same time are safe.
splash_status noalloc_scratch(NoAllocScratch **out) {
  int dev = 0;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxNoAllocDevices) return SPLASH_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return SPLASH_ERR_CUDA;
    }
    g_noalloc_addr[dev] = static_cast<NoAllocScratch *>(ptr);
  }
  *out = g_noalloc_addr[dev];
  return SPLASH_OK;
}

// Sums the per-row counters: totals = {active, partial, allowed pairs, max row}.
__global__ void __launch_bounds__(256) noalloc_totals_kernel(int64_t R, NoAllocScratch *s) {
  unsigned long long a = 0, p = 0, mx = 0;
  for (int64_t x = threadIdx.x; x < R; x += blockDim.x) {
    a += (unsigned long long)s->row_cnt[x];
    p += (unsigned long long)s->row_pcnt[x];
    mx = max(mx, (unsigned long long)s->row_cnt[x]);
  }
  for (int off = 16; off; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    p += __shfl_xor_sync(0xffffffffu, p, off);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  __shared__ unsigned long long sa[8], sp[8], sm[8];
  if ((threadIdx.x & 31) == 0) {
    sa[threadIdx.x >> 5] = a;
    sp[threadIdx.x >> 5] = p;
    sm[threadIdx.x >> 5] = mx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long ta = 0, tp = 0, tm = 0;
    for (int w = 0; w < 8; ++w) {
      ta += sa[w];
      tp += sp[w];
      tm = max(tm, sm[w]);
    }
    s->totals[0] = ta;
    s->totals[1] = tp;
    s->totals[2] = s->counters[3];
    s->totals[3] = tm;
  }
}

}  // namespace

splash_status splash_classify_blocks_noalloc_impl(const splash_mask_spec *spec, int64_t Lq, int64_t Lk,
                                                  int32_t bq, int32_t bk, int8_t *block_mask,
                                                  int64_t *totals, cudaStream_t stream) {
  const bool seg = spec->q_segment_ids != nullptr;
  const int32_t nbm = seg ? spec->batch : 1;
  const int64_t nq = (Lq + bq - 1) / bq, nk = (Lk + bk - 1) / bk, R = (int64_t)nbm * nq;
  if (R > kNoAllocMaxRows || (int64_t)nbm * nk > kNoAllocMaxCols) return SPLASH_ERR_UNSUPPORTED;
  NoAllocScratch *s = nullptr;
  splash_status st = noalloc_scratch(&s);
  if (st != SPLASH_OK) return st;

  DevMask m;
  m.causal = spec->causal;
  m.wl = spec->window_left;
  m.wr = spec->window_right;
  m.qseg = spec->q_segment_ids;
  m.kvseg = seg ? (spec->kv_segment_ids ? spec->kv_segment_ids : spec->q_segment_ids) : nullptr;
  m.Lq = Lq;
  m.Lk = Lk;
  m.nq = nq;
  m.nk = nk;
  m.bq = bq;
  m.bk = bk;
  m.nbm = nbm;
  m.ragged = (Lq % bq) != 0 || (Lk % bk) != 0;

  // the counters must start at zero: the array keeps the previous call's values
  SPLASH_CUDA_TRY(cudaMemsetAsync(s->row_cnt, 0, sizeof(int32_t) * R, stream));
  SPLASH_CUDA_TRY(cudaMemsetAsync(s->row_pcnt, 0, sizeof(int32_t) * R, stream));
  SPLASH_CUDA_TRY(cudaMemsetAsync(s->counters, 0, sizeof(s->counters), stream));
  if (seg) {
    dim3 grid((unsigned)((nq + nk + 7) / 8), (unsigned)nbm);
    seg_summary_kernel<<<grid, 256, 0, stream>>>(m, s->qsum, s->kvsum, s->row_cnt, s->row_pcnt, s->counters);
  }
  {
    dim3 grid((unsigned)((nk + kClassifyThreads - 1) / kClassifyThreads), (unsigned)nq, (unsigned)nbm);
    classify_kernel<<<grid, kClassifyThreads, 0, stream>>>(m, s->qsum, s->kvsum, block_mask, s->row_cnt,
                                                          s->row_pcnt, s->counters, seg ? s->deferred : nullptr,
                                                          kNoAllocMaxDeferred);
  }
  if (seg) {
    int dev = 0, sms = 148;
    SPLASH_CUDA_TRY(cudaGetDevice(&dev));
    SPLASH_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    count_deferred_kernel<<<sms * 4, kClassifyThreads, 0, stream>>>(m, s->deferred, kNoAllocMaxDeferred, block_mask,
                                                                   s->row_cnt, s->row_pcnt, s->counters);
  }
  noalloc_totals_kernel<<<1, 256, 0, stream>>>(R, s);
  SPLASH_CUDA_TRY(cudaGetLastError());
  splash_count_launches(seg ? 4 : 2);
  unsigned long long t[4];
  SPLASH_CUDA_TRY(cudaMemcpyAsync(t, s->totals, sizeof t, cudaMemcpyDeviceToHost, stream));
  SPLASH_CUDA_TRY(cudaStreamSynchronize(stream));
  for (int x = 0; x < 4; ++x) totals[x] = (int64_t)t[x];
  return SPLASH_OK;
}
