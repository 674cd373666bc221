// attention_bwd.cu -- block-sparse (Splash) masked attention, backward pass,
// for sm_103a: tcgen05 MMAs with TMEM accumulators, TMA-staged tiles,
// warp-specialised elementwise work.
//
// What it computes: the gradients of the forward
//   out_i = sum_j P_ij v_j,   P_ij = exp(s_ij - LSE_i)   (keys j the mask allows)
// for an upstream gradient dout.  P is not stored by the forward: it is
// rebuilt on chip from the scores and the residual LSE the forward wrote
// ("Pallas Kernels and Splash Attention" §6.3, the residual outputs kept for
// the backward; "The maths and infra behind core LLM operations" (joto.ai),
// "LSE and Online Softmax": recomputing the probabilities from LSE instead of
// reading an L x L matrix).  With dP_ij = dout_i . v_j and
// D_i = dout_i . out_i (= sum_j P_ij dP_ij):
//   dS_ij = P_ij (dP_ij - D_i)        (times 1 - t_ij^2 under the soft cap
//                                      s = cap tanh(t), t = scale q.k / cap)
//   dv_j = sum_i P_ij dout_i,  dk_j = scale sum_i dS_ij q_i,
//   dq_i = scale sum_j dS_ij k_j.
// Only active blocks are visited, through the MaskInfo's column-major
// (transposed) form: one work item is (batch, kv head, kv block); it loops
// over the query heads of its GQA group and the active q-blocks of its column,
// so dk and dv of the item are complete when it ends.
//
// GB300 design:
//   * kernels per call: the transposed table (column counts, scan, fill,
//     pattern transpose; only on the first call after each build of the
//     MaskInfo, which keeps it), a prep kernel (D, dq accumulator cleared),
//     the main kernel and a conversion of the fp32 dq accumulator to bf16;
//   * main kernel: one persistent CTA per SM, items dealt longest column
//     first in serpentine order; 384 threads; warps 0-7 (two
//     warpgroups) do the elementwise work: a thread owns one key (TMEM lane)
//     and half of the block's 128 queries; warp 8 issues TMA loads; warp 9
//     issues the MMAs from one elected lane of the converged warp; warps
//     10-11 only hand their registers to the elementwise warpgroups;
//   * five MMAs per (query head, q-block) iteration, M = 128:
//       S^T  = K Q^T    dP^T = V dO^T           (TMEM, 128 columns each)
//       dV  += P^T dO   (A = P^T from TMEM)
//       dK  += dS^T Q   (A = dS^T from shared memory, K-major)
//       dQ   = dS K     (A = the same shared buffer read MN-major)
//     dQ reuses the dP^T columns once dS is formed; it is added to an fp32
//     accumulator in global memory by asynchronous TMA tile reductions staged
//     in shared memory, so the columns are free again as soon as they are read.
//     dK and dV stay in TMEM for the whole item;
//   * Q is double-buffered, dO single-buffered (it is first needed by dP one
//     MMA group after Q);
//   * every wait is bounded: on timeout the CTA raises an error bit, stops,
//     drains its copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace splash {
namespace {

constexpr int kBwdThreads = 384;
constexpr int kBwdProducerWarp = 8;
constexpr int kBwdMmaWarp = 9;
// setmaxnreg split: 384 x 168 at launch; elementwise warpgroups 208 each,
// control warpgroup 88: 2*128*208 + 128*88 = 64512 = 384*168.
constexpr int kBwdWorkRegs = 208;
constexpr int kBwdControlRegs = 88;
constexpr int kBwdTmemCols = 512;
constexpr float kBwdLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int CH = D / 64;            // 64-column chunks of a D-wide tile
  static constexpr int CHUNK = 128 * 128;      // bytes of a 128-row x 64-column bf16 box
  static constexpr int TILE = CH * CHUNK;      // a 128-row x D tile
  static constexpr int DS_BYTES = 2 * CHUNK;   // dS^T: 128 keys x 128 queries
  // shared memory: K, V, Q[2], dO, dS, LSE/D[2], second dQ staging, barriers,
  // TMEM holder, abort flag
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;
  static constexpr int OFF_DO = 4 * TILE;
  static constexpr int OFF_DS = 5 * TILE;
  static constexpr int OFF_LD = 5 * TILE + DS_BYTES;  // [2][LSE 128 floats, D 128 floats]
  // dQ readout: a warp reduces D / 64 pieces of 32 x 32 fp32 per iteration;
  // the first is staged in the warp's own rows of the dS^T buffer, the second
  // (D = 128) in a 4 KB slot of its own, so that the two reductions overlap
  static constexpr int NPIECE = D / 64;
  static constexpr int OFF_ST2 = OFF_LD + 2 * 1024;
  static constexpr int ST2_BYTES = NPIECE > 1 ? 8 * 4096 : 0;
  static constexpr int OFF_BAR = OFF_ST2 + ST2_BYTES;
  static constexpr int NBAR = 15;
  // no alignment slack: the dynamic shared memory starts 1024-byte aligned on
  // this GPU (checked by the kernel, which does nothing and reports
  // SPLASH_DEV_SMEM_ALIGN otherwise)
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(OFF_ST2 % 1024 == 0, "128B-swizzled staging needs 1024-byte alignment");
  // TMEM columns: S^T / P^T, dP^T / dQ, dV, dK
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
  // instruction descriptors (bits: 4-5 D f32, 7-9 A bf16, 10-12 B bf16,
  // 15 A MN-major, 16 B MN-major, 17-22 N/8, 24-28 M/16)
  static constexpr uint32_t idesc(int n, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
  }
  static constexpr uint32_t ID_S = idesc(128, false, false);  // S^T, dP^T
  static constexpr uint32_t ID_DV = idesc(D, false, true);    // dV (A from TMEM)
  static constexpr uint32_t ID_DK = idesc(D, false, true);    // dK
  static constexpr uint32_t ID_DQ = idesc(D, true, true);     // dQ
};

struct BwdParams {
  int32_t B, Hq, Hkv, G;
  int64_t Lq, Lk;
  int64_t Lq_pad;               // nq * bq: row stride of the padded workspace arrays
  int32_t nq, nk, nbm;
  // q-blocks of 128 or 256 rows; an iteration takes 128 query rows (one half
  // of a 256-row q-block), so a block's active entry is visited `halves` times
  int32_t bq, halves;
  int64_t num_items;            // B * Hkv * nk
  const int32_t *col_ptr;       // [nbm*nk + 1]
  const int32_t *col_rows;      // q-block of each active block, column-major
  const int32_t *col_next;      // its pattern index, -1 for full blocks
  const uint32_t *pattern_t;    // [P][128 keys][bq/32 words]: bit i%32 of word i/32 = (query i, key) allowed
  const unsigned long long *counters;  // device totals of the MaskInfo build ([2] = patterns)
  int64_t cap_patterns;
  const float *lse;             // [B*Hq*Lq_pad] (copied from the forward's, padding rows 0)
  const float *delta;           // [B*Hq*Lq_pad]
  float *dq_acc;                // [B*Hq*Lq_pad][D] fp32
  __nv_bfloat16 *dk, *dv;       // [B*Hkv*Lk][D]
  float scale, scale_log2, cap_inner, cap_log2;
  uint32_t *err;
  uint64_t timeout_ns;
};

struct BwdItem {
  int32_t b, kvh, j;
  int32_t e0, cnt;  // the column's range of the transposed list
};

__device__ __forceinline__ BwdItem bwd_item(const BwdParams &p, int64_t w) {
  BwdItem it;
  const int64_t bh = (int64_t)p.B * p.Hkv;
  it.j = (int32_t)(w / bh);
  const int32_t r = (int32_t)(w % bh);
  it.b = r / p.Hkv;
  it.kvh = r % p.Hkv;
  const int64_t c = (p.nbm > 1 ? (int64_t)it.b * p.nk : 0) + it.j;
  it.e0 = p.col_ptr[c];
  it.cnt = p.col_ptr[c + 1] - it.e0;
  return it;
}

// Work item of this CTA's round k: items are ordered longest column first
// (kv block ascending) and dealt in serpentine order (CTA c takes item
// k*G + c on even rounds, k*G + G-1-c on odd ones); -1 past the end, -2 for
// a slot of the last round that has no item.
__device__ __forceinline__ int64_t bwd_item_of_round(const BwdParams &p, int64_t k) {
  const int64_t g = gridDim.x;
  if (k * g >= p.num_items) return -1;
  const int64_t w = k * g + ((k & 1) ? g - 1 - blockIdx.x : blockIdx.x);
  return w < p.num_items ? w : -2;
}

// (query head, q-block, its 128-row half, pattern) of the item's iteration t:
// heads outermost, halves innermost
__device__ __forceinline__ void bwd_step(const BwdParams &p, const BwdItem &it, int32_t t, int32_t &h,
                                         int32_t &i, int32_t &half, int32_t &mn) {
  const int32_t u = t / p.halves;
  half = t - u * p.halves;
  const int32_t hh = u / it.cnt, e = it.e0 + u % it.cnt;
  h = it.kvh * p.G + hh;
  i = p.col_rows[e];
  mn = p.col_next[e];
  const int64_t np = (int64_t)p.counters[2];
  if (i < 0 || i >= p.nq || mn >= np || mn >= p.cap_patterns) {
    atomicOr(p.err, SPLASH_DEV_BAD_TABLE);
    i = 0;
    mn = -1;
  }
}

// first query row (within the head) of iteration (q-block i, half)
__device__ __forceinline__ int64_t bwd_q0(const BwdParams &p, int32_t i, int32_t half) {
  return (int64_t)i * p.bq + (int64_t)half * 128;
}

struct BwdBars {
  uint32_t base;
  __device__ uint32_t kv_full() const { return base; }
  __device__ uint32_t kv_empty() const { return base + 8; }
  __device__ uint32_t q_full(int s) const { return base + 16 + 8 * s; }
  __device__ uint32_t q_empty(int s) const { return base + 32 + 8 * s; }
  __device__ uint32_t do_full() const { return base + 48; }
  __device__ uint32_t do_empty() const { return base + 56; }
  __device__ uint32_t s_full() const { return base + 64; }
  __device__ uint32_t dp_full() const { return base + 72; }
  __device__ uint32_t dq_full() const { return base + 80; }
  __device__ uint32_t p_ready() const { return base + 88; }
  __device__ uint32_t ds_ready() const { return base + 96; }
  __device__ uint32_t dq_empty() const { return base + 104; }
  __device__ uint32_t drain() const { return base + 112; }
};

__device__ __forceinline__ void bwd_raise(const BwdParams &p, volatile int *abort, uint32_t bits) {
  atomicOr(p.err, bits);
  *abort = 1;
}

// 1-D bulk copy global -> shared completing `bytes` on the mbarrier (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Tiled TMA reduction: the box at (x, y) of the tensor map += the shared
// memory tile at src (fp32 add, bulk-group completion).
__device__ __forceinline__ void tma_reduce_add_2d(const void *tmap, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// tanh(t) = 1 - 2 / (e^(2t) + 1), odd-symmetric, |t| clamped where fp32
// tanh is 1.
__device__ __forceinline__ float tanh_exp(float t) {
  const float a = fminf(fabsf(t), 16.f);
  const float e = ex2_approx(2.8853900817779268f * a);  // e^(2a)
  return copysignf(1.f - __fdividef(2.f, e + 1.f), t);
}

// ------------------------------------------------------------ producer
template <int D>
__device__ void bwd_producer(const BwdParams &p, const CUtensorMap *tmQ, const CUtensorMap *tmK,
                             const CUtensorMap *tmV, const CUtensorMap *tmDO, uint32_t s0, const BwdBars &bar,
                             volatile int *abort) {
  using C = BwdCfg<D>;
  uint32_t n = 0, kv = 0;
  bool ok = true;
  for (int64_t k = 0; ok; ++k) {
    const int64_t w = bwd_item_of_round(p, k);
    if (w == -1) break;
    if (w < 0) continue;
    const BwdItem it = bwd_item(p, w);
    const int32_t N = p.G * it.cnt * p.halves;
    if (N == 0) continue;
    if (kv > 0 && !(ok = mbar_wait(bar.kv_empty(), (kv - 1) & 1u, abort, p.timeout_ns))) break;
    const int32_t ykv = (int32_t)(((int64_t)it.b * p.Hkv + it.kvh) * p.Lk + (int64_t)it.j * 128);
    mbar_arrive_expect_tx(bar.kv_full(), 2 * C::TILE);
    for (int ch = 0; ch < C::CH; ++ch) {
      tma_load_2d(s0 + C::OFF_K + ch * C::CHUNK, tmK, ch * 64, ykv, bar.kv_full());
      tma_load_2d(s0 + C::OFF_V + ch * C::CHUNK, tmV, ch * 64, ykv, bar.kv_full());
    }
    ++kv;
    for (int32_t t = 0; t < N; ++t, ++n) {
      int32_t h, i, half, mn;
      bwd_step(p, it, t, h, i, half, mn);
      const int st = n & 1;
      if (n >= 2 && !(ok = mbar_wait(bar.q_empty(st), ((n >> 1) - 1) & 1u, abort, p.timeout_ns))) break;
      // tiles from the caller's tensors (rows past a ragged Lq read the next
      // head's rows or the zero fill, all masked); LSE and D from the padded
      // workspace (whole blocks, always in bounds)
      const int64_t row = ((int64_t)it.b * p.Hq + h) * p.Lq + bwd_q0(p, i, half);
      const int64_t prow = ((int64_t)it.b * p.Hq + h) * p.Lq_pad + bwd_q0(p, i, half);
      mbar_arrive_expect_tx(bar.q_full(st), C::TILE + 1024);
      for (int ch = 0; ch < C::CH; ++ch)
        tma_load_2d(s0 + C::OFF_Q + st * C::TILE + ch * C::CHUNK, tmQ, ch * 64, (int32_t)row, bar.q_full(st));
      bulk_load(s0 + C::OFF_LD + st * 1024, p.lse + prow, 512, bar.q_full(st));
      bulk_load(s0 + C::OFF_LD + st * 1024 + 512, p.delta + prow, 512, bar.q_full(st));
      if (n >= 1 && !(ok = mbar_wait(bar.do_empty(), (n - 1) & 1u, abort, p.timeout_ns))) break;
      mbar_arrive_expect_tx(bar.do_full(), C::TILE);
      for (int ch = 0; ch < C::CH; ++ch)
        tma_load_2d(s0 + C::OFF_DO + ch * C::CHUNK, tmDO, ch * 64, (int32_t)row, bar.do_full());
    }
  }
  if (!ok) bwd_raise(p, abort, SPLASH_DEV_TIMEOUT_PRODUCER);
  // drain: every load issued has landed
  bool drained = true;
  if (kv > 0) drained &= mbar_wait_drain(bar.kv_full(), (kv - 1) & 1u, p.timeout_ns);
  for (uint32_t m = n > 2 ? n - 2 : 0; m < n; ++m)
    drained &= mbar_wait_drain(bar.q_full(m & 1), (m >> 1) & 1u, p.timeout_ns);
  if (n > 0) drained &= mbar_wait_drain(bar.do_full(), (n - 1) & 1u, p.timeout_ns);
  if (!drained) atomicOr(p.err, SPLASH_DEV_TIMEOUT_DRAIN);
}

// ------------------------------------------------------------ MMA issuer
// K-major x K-major, 128 x 128 output: A rows (keys) and B rows (queries) of
// D columns, 64-column chunks CHUNK bytes apart, k-step = 32 bytes inside the
// 128-byte swizzle atom.
template <int D>
__device__ __forceinline__ void issue_kk(uint32_t leader, uint32_t d_tmem, uint32_t a, uint32_t b) {
  using C = BwdCfg<D>;
  constexpr uint32_t HI = sdesc_hi_sw128(1024);
  const uint32_t ad = sdesc_lo(a, 16), bd = sdesc_lo(b, 16);
#pragma unroll
  for (int ch = 0; ch < C::CH; ++ch)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lhp(leader, d_tmem, ad + (uint32_t)((ch * C::CHUNK + kk * 32) >> 4), HI,
                 bd + (uint32_t)((ch * C::CHUNK + kk * 32) >> 4), HI, C::ID_S, (ch | kk) != 0);
}

// dV (+)= P^T dO: A = P^T in TMEM (bf16 pairs; queries 0-63 at columns 0-31,
// queries 64-127 at columns 64-95 of the S^T region), B = dO MN-major
// (k-step = 16 query rows = 2048 bytes, D chunks CHUNK bytes apart).
template <int D>
__device__ __forceinline__ void issue_dv(uint32_t leader, uint32_t d_tmem, uint32_t p_tmem, uint32_t b,
                                         bool first) {
  using C = BwdCfg<D>;
  constexpr uint32_t HI = sdesc_hi_sw128(1024);
  const uint32_t bd = sdesc_lo(b, C::CHUNK);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    mma_ts_lhp(leader, d_tmem, p_tmem + (j < 4 ? 8u * j : 64u + 8u * (j - 4)), bd + (uint32_t)((j * 2048) >> 4),
               HI, C::ID_DV, (!first || j > 0) ? 1u : 0u);
}

// dK (+)= dS^T Q: A = dS^T K-major (rows = keys, queries in two 64-wide
// halves CHUNK bytes apart), B = Q MN-major.
template <int D>
__device__ __forceinline__ void issue_dk(uint32_t leader, uint32_t d_tmem, uint32_t ds, uint32_t q, bool first) {
  using C = BwdCfg<D>;
  constexpr uint32_t HI = sdesc_hi_sw128(1024);
  const uint32_t ad = sdesc_lo(ds, 16), bd = sdesc_lo(q, C::CHUNK);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    mma_ss_lhp(leader, d_tmem, ad + (uint32_t)(((j >> 2) * C::CHUNK + (j & 3) * 32) >> 4), HI,
               bd + (uint32_t)((j * 2048) >> 4), HI, C::ID_DK, (!first || j > 0) ? 1u : 0u);
}

// dQ = dS K: A = dS MN-major (the dS^T buffer: queries contiguous within a
// key row, two 64-query chunks CHUNK bytes apart; k-step = 16 key rows), B = K
// MN-major.
template <int D>
__device__ __forceinline__ void issue_dq(uint32_t leader, uint32_t d_tmem, uint32_t ds, uint32_t k) {
  using C = BwdCfg<D>;
  constexpr uint32_t HI = sdesc_hi_sw128(1024);
  const uint32_t ad = sdesc_lo(ds, C::CHUNK), bd = sdesc_lo(k, C::CHUNK);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    mma_ss_lhp(leader, d_tmem, ad + (uint32_t)((j * 2048) >> 4), HI, bd + (uint32_t)((j * 2048) >> 4), HI,
               C::ID_DQ, j > 0 ? 1u : 0u);
}

template <int D>
__device__ void bwd_mma(const BwdParams &p, uint32_t tmem, uint32_t s0, const BwdBars &bar, volatile int *abort,
                        uint32_t leader) {
  using C = BwdCfg<D>;
  const uint32_t tS = tmem + C::T_S, tDP = tmem + C::T_DP, tDV = tmem + C::T_DV, tDK = tmem + C::T_DK;
  uint32_t n = 0, kv = 0;
  bool ok = true;
  for (int64_t k = 0; ok; ++k) {
    const int64_t w = bwd_item_of_round(p, k);
    if (w == -1) break;
    if (w < 0) continue;
    const BwdItem it = bwd_item(p, w);
    const int32_t N = p.G * it.cnt * p.halves;
    if (N == 0) continue;
    if (!(ok = mbar_wait(bar.kv_full(), kv & 1u, abort, p.timeout_ns))) break;
    ++kv;
    if (!(ok = mbar_wait(bar.q_full(n & 1), (n >> 1) & 1u, abort, p.timeout_ns))) break;
    tc_fence_after();
    issue_kk<D>(leader, tS, s0 + C::OFF_K, s0 + C::OFF_Q + (n & 1) * C::TILE);
    tc_commit_p(leader, bar.s_full());
    for (int32_t t = 0; t < N && ok; ++t, ++n) {
      const int st = n & 1;
      // dP^T(n): dO(n) landed and dQ(n-1) read out of the same columns
      if (!(ok = mbar_wait(bar.do_full(), n & 1u, abort, p.timeout_ns))) break;
      if (n > 0 && !(ok = mbar_wait(bar.dq_empty(), (n - 1) & 1u, abort, p.timeout_ns))) break;
      tc_fence_after();
      issue_kk<D>(leader, tDP, s0 + C::OFF_V, s0 + C::OFF_DO);
      tc_commit_p(leader, bar.dp_full());
      // dV(n) once P^T(n) is in TMEM
      if (!(ok = mbar_wait(bar.p_ready(), n & 1u, abort, p.timeout_ns))) break;
      tc_fence_after();
      issue_dv<D>(leader, tDV, tS, s0 + C::OFF_DO, t == 0);
      tc_commit_p(leader, bar.do_empty());
      // S^T(n+1) into the S^T columns (after dV(n) read P^T(n) from them)
      if (t + 1 < N) {
        if (!(ok = mbar_wait(bar.q_full((n + 1) & 1), ((n + 1) >> 1) & 1u, abort, p.timeout_ns))) break;
        tc_fence_after();
        issue_kk<D>(leader, tS, s0 + C::OFF_K, s0 + C::OFF_Q + ((n + 1) & 1) * C::TILE);
        tc_commit_p(leader, bar.s_full());
      }
      // dK(n), dQ(n) once dS(n) is in shared memory
      if (!(ok = mbar_wait(bar.ds_ready(), n & 1u, abort, p.timeout_ns))) break;
      tc_fence_after();
      issue_dk<D>(leader, tDK, s0 + C::OFF_DS, s0 + C::OFF_Q + st * C::TILE, t == 0);
      issue_dq<D>(leader, tDP, s0 + C::OFF_DS, s0 + C::OFF_K);
      tc_commit_p(leader, bar.dq_full());
      tc_commit_p(leader, bar.q_empty(st));
      if (t + 1 == N) tc_commit_p(leader, bar.kv_empty());
    }
  }
  if (!ok && leader) bwd_raise(p, abort, SPLASH_DEV_TIMEOUT_MMA);
  tc_commit_p(leader, bar.drain());
  if (!mbar_wait_drain(bar.drain(), 0, p.timeout_ns) && leader) atomicOr(p.err, SPLASH_DEV_TIMEOUT_DRAIN);
}

// ------------------------------------------------------------ elementwise warps
// dQ(m) from TMEM (lane = query, this warpgroup's half of the D columns)
// added to the fp32 accumulator by TMA tile reductions: each 32 x 32 piece
// is staged in this warp's own 4 KB of the dS^T buffer (its dS^T rows, free
// once the MMAs of iteration m have completed; 128B-swizzled, as the tensor
// map expects) and reduced into global memory asynchronously.  TMEM is
// released as soon as the pieces are in registers; a later staging (or dS
// store) into the same 4 KB first waits until the reduction has read it.
// row0: accumulator row of the warp's first query.
// The warp's bulk groups are committed in order piece 0 (slot A, the dS^T
// rows), piece 1 (slot B, D = 128 only), and the dS^T rows are written
// between readouts.  So before writing slot A (piece 0 or dS^T) only the
// most recent group may still be reading when it is piece 1's (slot B), and
// before writing slot B only the just-committed piece 0: bwd_wait_slot
// waits for all groups but the latest one when D = 128, for all of them
// when there is a single piece per readout.
// all but this thread's most recent bulk group have finished reading their
// shared-memory source
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

template <int D>
__device__ __forceinline__ void bwd_wait_slot() {
  if constexpr (D / 64 > 1)
    bulk_wait_read_1();
  else
    bulk_wait_read_all();
}

template <int D>
__device__ __forceinline__ bool bwd_readout(const BwdParams &p, const CUtensorMap *tmDQ, uint32_t tDQ, uint32_t m,
                                            int32_t row0, int32_t col0, uint32_t stage, uint32_t stage2,
                                            volatile int *abort, uint32_t bars_dq_full, uint32_t bars_dq_empty,
                                            int lane) {
  if (!__all_sync(0xffffffffu, mbar_wait(bars_dq_full, m & 1u, abort, p.timeout_ns))) return false;
  tc_fence_after();
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    const uint32_t slot = c == 0 ? stage : stage2;
    const uint32_t wrow = slot + (uint32_t)lane * 128u;
    uint32_t r[32];
    tmem_ld32(tDQ + 32u * c, r);
    tmem_wait_ld();
    reg_fence32(r);
    if (c + 1 == D / 64) {  // TMEM fully read: the columns may take the next dP^T
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars_dq_empty);
    }
    if (lane == 0) bwd_wait_slot<D>();  // the slot's previous reduction has read it
    __syncwarp();
#pragma unroll
    for (int y = 0; y < 8; ++y)
      st_shared_v4(wrow + (uint32_t)(((y ^ (lane & 7)) << 4)), r[4 * y], r[4 * y + 1], r[4 * y + 2], r[4 * y + 3]);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_reduce_add_2d(tmDQ, slot, col0 + 32 * c, row0);
      bulk_commit_group();
    }
  }
  return true;
}

template <int D, bool CAP>
__device__ void bwd_work(const BwdParams &p, const CUtensorMap *tmDQ, uint32_t tmem, uint32_t s0, const BwdBars &bar,
                         volatile int *abort, int warp, int lane) {
  using C = BwdCfg<D>;
  const int wg = warp >> 2;   // which 64 queries of the block
  const int wq = warp & 3;    // TMEM lane quarter
  const int jj = wq * 32 + lane;  // key within the block (S^T / dP^T / dK / dV lane) or query (dQ lane)
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = tmem + C::T_S + lane_off + 64u * wg;
  const uint32_t tDP = tmem + C::T_DP + lane_off + 64u * wg;
  const uint32_t tDQ = tmem + C::T_DP + lane_off + (uint32_t)(wg * (D / 2));
  const uint32_t tDV = tmem + C::T_DV + lane_off + (uint32_t)(wg * (D / 2));
  const uint32_t tDK = tmem + C::T_DK + lane_off + (uint32_t)(wg * (D / 2));
  const float mul = CAP ? p.cap_log2 : p.scale_log2;
  uint32_t n = 0;
  bool ok = true;
  int32_t prev_row = 0;  // dq accumulator row of the previous iteration's first query of this warp
  const int32_t col0 = wg * (D / 2);
  // this warp's 32 rows of its half of the dS^T buffer (staging for the dQ readout)
  const uint32_t stage = s0 + C::OFF_DS + wg * C::CHUNK + (uint32_t)(wq * 32) * 128u;
  const uint32_t stage2 = s0 + C::OFF_ST2 + (uint32_t)warp * 4096u;  // D = 128 only
  for (int64_t k = 0; ok; ++k) {
    const int64_t w = bwd_item_of_round(p, k);
    if (w == -1) break;
    if (w < 0) continue;
    const BwdItem it = bwd_item(p, w);
    const int32_t N = p.G * it.cnt * p.halves;
    const int64_t krow = ((int64_t)it.b * p.Hkv + it.kvh) * p.Lk + (int64_t)it.j * 128 + jj;
    __nv_bfloat16 *dk_row = p.dk + krow * D + wg * (D / 2);
    __nv_bfloat16 *dv_row = p.dv + krow * D + wg * (D / 2);
    const bool key_out = (int64_t)it.j * 128 + jj < p.Lk;  // padding keys of a ragged Lk are never stored
    if (N == 0) {  // no query sees this key block: zero gradients
      if (!key_out) continue;
      for (int x = 0; x < D / 2; x += 8) {
        *reinterpret_cast<uint4 *>(dk_row + x) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(dv_row + x) = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    for (int32_t t = 0; t < N && ok; ++t, ++n) {
      int32_t h, i, half, mn;
      bwd_step(p, it, t, h, i, half, mn);
      const int st = n & 1;
      const uint32_t ld = s0 + C::OFF_LD + st * 1024 + 256u * wg;  // this half's LSE; D at +512
      // ---- P^T(n) = exp(S^T - LSE): S^T lane = key jj, columns = queries 64wg + x
      ok = __all_sync(0xffffffffu, mbar_wait(bar.s_full(), n & 1u, abort, p.timeout_ns) &&
                                       mbar_wait(bar.q_full(st), (n >> 1) & 1u, abort, p.timeout_ns));
      if (!ok) break;
      tc_fence_after();
      float P[64];
      float G[CAP ? 64 : 1];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tS, r0);
        tmem_ld32(tS + 32u, r1);
        uint32_t bits0 = 0xffffffffu, bits1 = 0xffffffffu;
        if (mn >= 0) {
          const uint32_t *src = p.pattern_t + ((int64_t)mn * 128 + jj) * (p.bq / 32) + 4 * half + 2 * wg;
          bits0 = __ldg(src);
          bits1 = __ldg(src + 1);
        }
        tmem_wait_ld();
        reg_fence32(r0);
        reg_fence32(r1);
#pragma unroll
        for (int x = 0; x < 64; x += 4) {
          const float4 l4 = ld_shared_f4(ld + 4u * x);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            const int q = x + y;
            float s = __uint_as_float(q < 32 ? r0[q] : r1[q - 32]);
            if (CAP) {
              s = tanh_exp(s * p.cap_inner);
              G[q] = 1.f - s * s;
            }
            const bool allowed = ((q < 32 ? bits0 : bits1) >> (q & 31)) & 1u;
            P[q] = allowed ? ex2_approx(fmaf(s, mul, -lv[y] * kBwdLog2e)) : 0.f;
          }
        }
        uint32_t pk[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) pk[x] = pack_bf16x2(P[2 * x], P[2 * x + 1]);
        tmem_st32(tS, pk);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.p_ready());
      // ---- dQ(n-1) out of TMEM (its MMAs ran while P(n) was formed)
      if (t > 0 && !(ok = bwd_readout<D>(p, tmDQ, tDQ, n - 1, prev_row, col0, stage, stage2, abort,
                                         bar.dq_full(), bar.dq_empty(), lane)))
        break;
      // ---- dS^T(n) = P^T (dP^T - D) [(1 - t^2)], bf16 into the swizzled dS^T buffer
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar.dp_full(), n & 1u, abort, p.timeout_ns)))) break;
      tc_fence_after();
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tDP, r0);
        tmem_ld32(tDP + 32u, r1);
        tmem_wait_ld();
        reg_fence32(r0);
        reg_fence32(r1);
        if (lane == 0) bwd_wait_slot<D>();  // dQ staging in these rows has been read
        __syncwarp();
        const uint32_t row = s0 + C::OFF_DS + wg * C::CHUNK + jj * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 8 queries = one 16-byte chunk
          const float4 d0 = ld_shared_f4(ld + 512u + 32u * c);
          const float4 d1 = ld_shared_f4(ld + 512u + 32u * c + 16u);
          const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
          uint32_t pk[4];
#pragma unroll
          for (int y = 0; y < 8; y += 2) {
            float g2[2];
#pragma unroll
            for (int z = 0; z < 2; ++z) {
              const int q = 8 * c + y + z;
              const float dp = __uint_as_float(q < 32 ? r0[q] : r1[q - 32]);
              float g = P[q] * (dp - dd[y + z]);
              if (CAP) g *= G[q];
              g2[z] = g;
            }
            pk[y >> 1] = pack_bf16x2(g2[0], g2[1]);
          }
          st_shared_v4(row + (uint32_t)((c ^ (jj & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar.ds_ready());
      prev_row = (int32_t)(((int64_t)it.b * p.Hq + h) * p.Lq_pad + bwd_q0(p, i, half) + wq * 32);
    }
    if (!ok) break;
    // ---- the item's last dQ, then dK, dV (complete once that dQ has landed)
    if (!(ok = bwd_readout<D>(p, tmDQ, tDQ, n - 1, prev_row, col0, stage, stage2, abort, bar.dq_full(),
                              bar.dq_empty(), lane)))
      break;
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      uint32_t rk[32], rv[32];
      tmem_ld32(tDK + 32u * c, rk);
      tmem_ld32(tDV + 32u * c, rv);
      tmem_wait_ld();
      reg_fence32(rk);
      reg_fence32(rv);
#pragma unroll
      for (int x = 0; x < 32; x += 8) {
        uint4 a, b;
        a.x = pack_bf16x2(__uint_as_float(rk[x]) * p.scale, __uint_as_float(rk[x + 1]) * p.scale);
        a.y = pack_bf16x2(__uint_as_float(rk[x + 2]) * p.scale, __uint_as_float(rk[x + 3]) * p.scale);
        a.z = pack_bf16x2(__uint_as_float(rk[x + 4]) * p.scale, __uint_as_float(rk[x + 5]) * p.scale);
        a.w = pack_bf16x2(__uint_as_float(rk[x + 6]) * p.scale, __uint_as_float(rk[x + 7]) * p.scale);
        b.x = pack_bf16x2(__uint_as_float(rv[x]), __uint_as_float(rv[x + 1]));
        b.y = pack_bf16x2(__uint_as_float(rv[x + 2]), __uint_as_float(rv[x + 3]));
        b.z = pack_bf16x2(__uint_as_float(rv[x + 4]), __uint_as_float(rv[x + 5]));
        b.w = pack_bf16x2(__uint_as_float(rv[x + 6]), __uint_as_float(rv[x + 7]));
        if (key_out) {
          *reinterpret_cast<uint4 *>(dk_row + 32 * c + x) = a;
          *reinterpret_cast<uint4 *>(dv_row + 32 * c + x) = b;
        }
      }
    }
    tc_fence_before();
  }
  if (!ok && lane == 0) bwd_raise(p, abort, SPLASH_DEV_TIMEOUT_SOFTMAX);
  if (lane == 0) bulk_wait_all();  // this warp's dq reductions have completed
}

template <int D, bool CAP>
__global__ void __launch_bounds__(kBwdThreads, 1)
splash_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // uniform over the CTA: nothing has started yet
    if (threadIdx.x == 0) atomicOr(p.err, SPLASH_DEV_SMEM_ALIGN);
    return;
  }
  uint8_t *smem = smem_raw;
  const uint32_t s0 = smem_u32(smem);
  const BwdBars bar{s0 + C::OFF_BAR};
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_holder), kBwdTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    mbar_init(bar.kv_full(), 1);
    mbar_init(bar.kv_empty(), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar.q_full(s), 1);
      mbar_init(bar.q_empty(s), 1);
    }
    mbar_init(bar.do_full(), 1);
    mbar_init(bar.do_empty(), 1);
    mbar_init(bar.s_full(), 1);
    mbar_init(bar.dp_full(), 1);
    mbar_init(bar.dq_full(), 1);
    mbar_init(bar.p_ready(), 8);   // the eight elementwise warps
    mbar_init(bar.ds_ready(), 8);
    mbar_init(bar.dq_empty(), 8);
    mbar_init(bar.drain(), 1);
    *abort = 0;
    mbar_fence_init();
  }
  if (threadIdx.x == kBwdProducerWarp * 32) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmDQ);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp >= 8) {
    regs_decrease<kBwdControlRegs>();
    if (warp == kBwdProducerWarp) {
      if (lane == 0) bwd_producer<D>(p, &tmQ, &tmK, &tmV, &tmDO, s0, bar, abort);
    } else if (warp == kBwdMmaWarp) {
      bwd_mma<D>(p, tmem, s0, bar, abort, elect_one_sync());
    }
  } else {
    regs_increase<kBwdWorkRegs>();
    bwd_work<D, CAP>(p, &tmDQ, tmem, s0, bar, abort, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

// ------------------------------------------------------------ small kernels
// Padded workspace rows r = bh * Lq_pad + i (whole q-blocks per head):
// D_r = sum_x dout[bh*Lq + i][x] * out[...][x] (fp32) and a copy of the
// forward's LSE for i < Lq, 0 on padding rows; the dq accumulator rows are
// cleared.  One 16-lane half-warp per row (a warp takes two consecutive rows,
// so its shuffles always see all 32 lanes).
template <int D>
__global__ void bwd_prep_kernel(const __nv_bfloat16 *out, const __nv_bfloat16 *dout, const float *lse_in,
                                float *delta, float *lse_pad, float *dq_acc, int64_t rows_pad, int64_t Lq,
                                int64_t Lq_pad) {
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int half = (threadIdx.x >> 4) & 1, sub = threadIdx.x & 15;
  for (int64_t base = 2 * warp; base < rows_pad; base += 2 * nwarps) {
    const int64_t r = base + half;
    const bool valid = r < rows_pad;
    const int64_t bh = r / Lq_pad, i = r - bh * Lq_pad;
    const bool real = valid && i < Lq;
    const int64_t src = bh * Lq + i;
    float acc = 0.f;
    if (real) {
#pragma unroll
      for (int x = sub * 8; x < D; x += 128) {
        const uint4 a = *reinterpret_cast<const uint4 *>(out + src * D + x);
        const uint4 b = *reinterpret_cast<const uint4 *>(dout + src * D + x);
        const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
        const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const float2 fa = __bfloat1622float2(pa[y]), fb = __bfloat1622float2(pb[y]);
          acc = fmaf(fa.x, fb.x, acc);
          acc = fmaf(fa.y, fb.y, acc);
        }
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (valid) {
      if (sub == 0) {
        delta[r] = acc;
        lse_pad[r] = real ? lse_in[src] : 0.f;
      }
#pragma unroll
      for (int x = sub * 4; x < D; x += 64)
        *reinterpret_cast<float4 *>(dq_acc + r * D + x) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// dq[bh][i] = bf16(dq_acc[bh * Lq_pad + i] * scale) for the real rows i < Lq
// (x counts groups of 4 columns of dq).
__global__ void bwd_dq_convert_kernel(const float *dq_acc, __nv_bfloat16 *dq, int64_t n4, int32_t d4, int64_t Lq,
                                      int64_t Lq_pad, float scale) {
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n4; x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = x / d4, c = x - row * d4;
    const int64_t bh = row / Lq, i = row - bh * Lq;
    const float4 v = reinterpret_cast<const float4 *>(dq_acc)[(bh * Lq_pad + i) * d4 + c];
    uint2 o;
    o.x = pack_bf16x2(v.x * scale, v.y * scale);
    o.y = pack_bf16x2(v.z * scale, v.w * scale);
    reinterpret_cast<uint2 *>(dq)[x] = o;
  }
}

// Column counts of the block mask: cnt[c] = #{i : block_mask[bm][i][j] != 0},
// c = bm*nk + j; one warp per column.
__global__ void col_count_kernel(const int8_t *block_mask, int32_t nq, int32_t nk, int64_t ncols, int32_t *cnt) {
  const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (c >= ncols) return;
  const int64_t bm = c / nk, j = c % nk;
  int32_t k = 0;
  for (int32_t i = lane; i < nq; i += 32) k += block_mask[(bm * nq + i) * nk + j] != 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k += __shfl_xor_sync(0xffffffffu, k, o);
  if (lane == 0) cnt[c] = k;
}

// Exclusive scan of the column counts (one CTA of 1024 threads; each thread
// sums a contiguous run, then a block scan of the run totals).
__global__ void col_scan_kernel(const int32_t *cnt, int64_t ncols, int32_t *col_ptr) {
  __shared__ int32_t part[1024];
  const int tid = threadIdx.x;
  const int64_t per = (ncols + 1023) / 1024;
  const int64_t lo = min(ncols, (int64_t)tid * per), hi = min(ncols, lo + per);
  int32_t s = 0;
  for (int64_t c = lo; c < hi; ++c) s += cnt[c];
  part[tid] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int32_t v = tid >= o ? part[tid - o] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int32_t run = part[tid] - s;
  for (int64_t c = lo; c < hi; ++c) {
    col_ptr[c] = run;
    run += cnt[c];
  }
  if (tid == 1023) col_ptr[ncols] = part[1023];
}

// Column-major list of the active blocks: for column c, its q-blocks in
// ascending order and their pattern index (mask_next of the row-major entry,
// found by binary search in the row's ascending active columns).
__global__ void col_fill_kernel(const int8_t *block_mask, const int32_t *row_ptr, const int32_t *active_cols,
                                const int32_t *mask_next, int32_t nq, int32_t nk, int64_t ncols,
                                const int32_t *col_ptr, int32_t *col_rows, int32_t *col_next) {
  const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (c >= ncols) return;
  const int64_t bm = c / nk;
  const int32_t j = (int32_t)(c % nk);
  int32_t base = col_ptr[c];
  for (int32_t i0 = 0; i0 < nq; i0 += 32) {
    const int32_t i = i0 + lane;
    const bool act = i < nq && block_mask[(bm * nq + i) * nk + j] != 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, act);
    if (act) {
      const int32_t pos = base + __popc(bal & ((1u << lane) - 1u));
      const int64_t r = bm * nq + i;
      int32_t lo = row_ptr[r], hi = row_ptr[r + 1] - 1;
      while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (active_cols[mid] < j) lo = mid + 1; else hi = mid;
      }
      col_rows[pos] = i;
      col_next[pos] = mask_next[lo];
    }
    base += __popc(bal);
  }
}

// Transposed pattern bits: word (p, key j, w) holds, at bit b, whether query
// 32w + b may see key j (bq / 32 words per key).  Source: pattern_bits
// [p][query][4 words over the 128 keys].
__global__ void pattern_transpose_kernel(const uint32_t *pattern_bits, const unsigned long long *counters,
                                         int64_t cap_patterns, int32_t bq, uint32_t *pattern_t) {
  const int64_t np = min((int64_t)counters[2], cap_patterns);
  const int32_t qw = bq / 32;
  const int64_t total = np * 128 * qw;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pidx = x / (128 * qw);
    const int32_t j = (int32_t)((x / qw) % 128), w = (int32_t)(x % qw);
    const uint32_t *src = pattern_bits + pidx * bq * 4;
    uint32_t v = 0;
#pragma unroll 8
    for (int b = 0; b < 32; ++b) v |= ((src[(32 * w + b) * 4 + (j >> 5)] >> (j & 31)) & 1u) << b;
    pattern_t[x] = v;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 bwd_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// bf16 [rows][cols] tiles of 128 rows x 64 columns (128B swizzle)
bool make_bwd_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows) {
  auto fn = bwd_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows][cols] tiles of 32 rows x 32 columns (128B swizzle), for the dq
// accumulator's reductions
bool make_bwd_map_f32(CUtensorMap *map, void *base, uint64_t cols, uint64_t rows) {
  auto fn = bwd_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool CAP>
splash_status launch_bwd(const void *q, const void *k, const void *v, const void *dout, const BwdParams &prm,
                         int sms, cudaStream_t stream) {
  using C = BwdCfg<D>;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_bwd_map(&tq, q, D, (uint64_t)prm.B * prm.Hq * prm.Lq) ||
      !make_bwd_map(&tk, k, D, (uint64_t)prm.B * prm.Hkv * prm.Lk) ||
      !make_bwd_map(&tv, v, D, (uint64_t)prm.B * prm.Hkv * prm.Lk) ||
      !make_bwd_map(&tdo, dout, D, (uint64_t)prm.B * prm.Hq * prm.Lq) ||
      !make_bwd_map_f32(&tdq, prm.dq_acc, D, (uint64_t)prm.B * prm.Hq * prm.Lq_pad))
    return SPLASH_ERR_CUDA;
  static int configured_device = -1;
  int dev = 0;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  if (configured_device != dev) {
    SPLASH_CUDA_TRY(cudaFuncSetAttribute(splash_bwd_kernel<D, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM));
    configured_device = dev;
  }
  const int64_t grid = prm.num_items < sms ? prm.num_items : sms;
  if (grid <= 0) return SPLASH_OK;
  splash_bwd_kernel<D, CAP><<<(unsigned)grid, kBwdThreads, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, prm);
  SPLASH_CUDA_TRY(cudaGetLastError());
  splash_count_launches(1);
  return SPLASH_OK;
}

}  // namespace
}  // namespace splash

using namespace splash;

// fp32 dq accumulator, D and a copy of LSE, each over whole q-blocks per
// head (rows past a ragged Lq are padding); sized for 256-row blocks, which
// covers 128-row ones
size_t splash_attention_bwd_workspace_bytes(int32_t B, int32_t Hq, int64_t Lq, int32_t dqk) {
  const size_t rows = (size_t)B * Hq * (size_t)((Lq + 255) / 256 * 256);
  return ((rows * dqk * 4 + 255) & ~(size_t)255) + 2 * ((rows * 4 + 255) & ~(size_t)255);
}

splash_status splash_attention_bwd_launch(const void *q, const void *k, const void *v, const void *out,
                                          const float *lse, const void *dout, int32_t B, int32_t Hq, int32_t Hkv,
                                          int64_t Lq, int64_t Lk, int32_t d, splash_mask_info *mi, float scale,
                                          float softcap, void *dq, void *dk, void *dv, void *workspace,
                                          cudaStream_t stream, uint32_t *err_word) {
  // the transposed table, owned by the MaskInfo (allocated on first use),
  // made once per build of the table and reused by later calls
  const int64_t ncols = (int64_t)mi->batch_rows * mi->nk;
  const bool fresh = mi->t_gen != 0 && mi->t_gen == mi->build_gen && mi->t_ready != nullptr;
  const int64_t pwords = 128 * (mi->bq / 32);  // transposed words per pattern
  if (!fresh && (mi->t_cap_cols < ncols || mi->t_cap_active < mi->cap_blocks ||
                 mi->t_cap_patterns < mi->cap_patterns * pwords)) {
    splash_mask_info_free_transposed(mi);
    if (cudaMalloc(&mi->t_col_cnt, sizeof(int32_t) * ncols) != cudaSuccess ||
        cudaMalloc(&mi->t_col_ptr, sizeof(int32_t) * (ncols + 1)) != cudaSuccess ||
        cudaMalloc(&mi->t_col_rows, sizeof(int32_t) * std::max<int64_t>(mi->cap_blocks, 1)) != cudaSuccess ||
        cudaMalloc(&mi->t_col_next, sizeof(int32_t) * std::max<int64_t>(mi->cap_blocks, 1)) != cudaSuccess ||
        cudaMalloc(&mi->t_pattern_bits, sizeof(uint32_t) * pwords * std::max<int64_t>(mi->cap_patterns, 1)) !=
            cudaSuccess) {
      splash_mask_info_free_transposed(mi);
      cudaGetLastError();
      return SPLASH_ERR_OOM;
    }
    mi->t_cap_cols = ncols;
    mi->t_cap_active = mi->cap_blocks;
    mi->t_cap_patterns = mi->cap_patterns * pwords;
  }
  int dev = 0;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  int sms = 148;
  SPLASH_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (fresh) {
    // made by an earlier call, possibly on another stream
    SPLASH_CUDA_TRY(cudaStreamWaitEvent(stream, mi->t_ready, 0));
  } else {
  const unsigned cgrid = (unsigned)((ncols * 32 + 255) / 256);
  col_count_kernel<<<cgrid, 256, 0, stream>>>(mi->block_mask, (int32_t)mi->nq, (int32_t)mi->nk, ncols,
                                              mi->t_col_cnt);
  col_scan_kernel<<<1, 1024, 0, stream>>>(mi->t_col_cnt, ncols, mi->t_col_ptr);
  col_fill_kernel<<<cgrid, 256, 0, stream>>>(mi->block_mask, mi->row_ptr, mi->active_cols, mi->mask_next,
                                             (int32_t)mi->nq, (int32_t)mi->nk, ncols, mi->t_col_ptr,
                                             mi->t_col_rows, mi->t_col_next);
  pattern_transpose_kernel<<<(unsigned)std::max<int64_t>(1, std::min<int64_t>(
                                 (pwords * std::max<int64_t>(mi->cap_patterns, 1) + 255) / 256, sms * 8)),
                             256, 0, stream>>>(mi->pattern_bits, mi->counters, mi->cap_patterns, mi->bq,
                                               mi->t_pattern_bits);
  SPLASH_CUDA_TRY(cudaGetLastError());
  splash_count_launches(4);
  if (mi->t_ready == nullptr) SPLASH_CUDA_TRY(cudaEventCreateWithFlags(&mi->t_ready, cudaEventDisableTiming));
  SPLASH_CUDA_TRY(cudaEventRecord(mi->t_ready, stream));
  mi->t_gen = mi->build_gen;
  }

  const int64_t rows = (int64_t)B * Hq * Lq;
  const int64_t Lq_pad = mi->nq * mi->bq, rows_pad = (int64_t)B * Hq * Lq_pad;
  float *dq_acc = static_cast<float *>(workspace);
  float *delta = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                           ((rows_pad * d * 4 + 255) & ~(int64_t)255));
  float *lse_pad = reinterpret_cast<float *>(reinterpret_cast<char *>(delta) + ((rows_pad * 4 + 255) & ~(int64_t)255));
  const unsigned pgrid = (unsigned)std::max<int64_t>(1, std::min<int64_t>((rows_pad * 16 + 255) / 256, sms * 16));
  if (d == 128)
    bwd_prep_kernel<128><<<pgrid, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(out),
                                                     static_cast<const __nv_bfloat16 *>(dout), lse, delta, lse_pad,
                                                     dq_acc, rows_pad, Lq, Lq_pad);
  else
    bwd_prep_kernel<64><<<pgrid, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(out),
                                                    static_cast<const __nv_bfloat16 *>(dout), lse, delta, lse_pad,
                                                    dq_acc, rows_pad, Lq, Lq_pad);
  SPLASH_CUDA_TRY(cudaGetLastError());
  splash_count_launches(1);

  BwdParams prm;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = Hq / Hkv;
  prm.Lq = Lq;
  prm.Lq_pad = Lq_pad;
  prm.Lk = Lk;
  prm.nq = (int32_t)mi->nq;
  prm.nk = (int32_t)mi->nk;
  prm.nbm = mi->batch_rows;
  prm.bq = mi->bq;
  prm.halves = mi->bq / 128;
  prm.num_items = (int64_t)B * Hkv * mi->nk;
  prm.col_ptr = mi->t_col_ptr;
  prm.col_rows = mi->t_col_rows;
  prm.col_next = mi->t_col_next;
  prm.pattern_t = mi->t_pattern_bits;
  prm.counters = mi->counters;
  prm.cap_patterns = mi->cap_patterns;
  prm.lse = lse_pad;
  prm.delta = delta;
  prm.dq_acc = dq_acc;
  prm.dk = static_cast<__nv_bfloat16 *>(dk);
  prm.dv = static_cast<__nv_bfloat16 *>(dv);
  prm.scale = scale;
  prm.scale_log2 = scale * kBwdLog2e;
  prm.cap_inner = softcap > 0.f ? scale / softcap : 0.f;
  prm.cap_log2 = softcap > 0.f ? softcap * kBwdLog2e : 0.f;
  prm.err = err_word;
  prm.timeout_ns = 1000000000ull;
  splash_status st;
  if (d == 128)
    st = softcap > 0.f ? launch_bwd<128, true>(q, k, v, dout, prm, sms, stream)
                       : launch_bwd<128, false>(q, k, v, dout, prm, sms, stream);
  else
    st = softcap > 0.f ? launch_bwd<64, true>(q, k, v, dout, prm, sms, stream)
                       : launch_bwd<64, false>(q, k, v, dout, prm, sms, stream);
  if (st != SPLASH_OK) return st;

  const int64_t n4 = rows * d / 4;
  const unsigned vgrid = (unsigned)std::max<int64_t>(1, std::min<int64_t>((n4 + 255) / 256, sms * 16));
  bwd_dq_convert_kernel<<<vgrid, 256, 0, stream>>>(dq_acc, static_cast<__nv_bfloat16 *>(dq), n4, d / 4, Lq, Lq_pad,
                                                   scale);
  SPLASH_CUDA_TRY(cudaGetLastError());
  splash_count_launches(1);
  return SPLASH_OK;
}
