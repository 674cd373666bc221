// attention_fwd.cu -- block-sparse (Splash) masked attention, forward pass,
// for sm_103a: TMA-staged Q/K/V tiles, QK^T and PV on tcgen05 tensor cores
// with TMEM accumulators, warp-specialised online softmax.
//
// What it computes ("Pallas Kernels and Splash Attention", CMU 11-868
// Lecture 13 notes):
//   §5.1  online softmax: running max m and sum l, alpha = exp(m_old - m_new);
//   §5.2  the Flash body per (head, q-block, kv-block): scores, mask + soft
//         cap, m_next, exp, alpha, l and o updates, o / l once at the end
//         (deferred normalisation); heads independent, GQA heads share K/V;
//   §5.4  soft cap cap * tanh(x / cap);
//   §6.3  only active blocks of a q-block row are visited (the row's range of
//         the MaskInfo active list), partial blocks are masked from their
//         pattern, and the residual LSE is written next to O.
// "The maths and infra behind core LLM operations" (joto.ai), "Causal Mask":
// empty blocks are neither loaded nor multiplied; "LSE and Online Softmax":
// LSE = m + log l.
//
// GB300 design (differs from the TPU kernel on the pages):
//   * one persistent CTA per SM; each work item is (batch, two query heads,
//     one q-block row); the two heads are two 128-row query tiles that share
//     the row's active list, and share K/V tiles when they are in the same
//     GQA group.  With 256-row q-blocks an item is (batch, one head, one
//     q-block row) and its tiles are the block's two halves, which share
//     every K/V tile (the MHA analogue of the GQA pairing);
//   * items are sorted longest row first and dealt to the CTAs in serpentine
//     order; when rows span all keys and all heads' K/V exceeds what L2 can
//     keep, the items are first grouped by heads whose K/V fits
//     (splash_choose_head_group, csrc/api.cu);
//   * K/V staging: rings of whole K and V tiles; at dqk = 192 with 256-row
//     q-blocks one ring of 64-column chunks shared by K and V, released
//     chunk by chunk;
//   * warp roles (384 threads): warps 0-3 / 4-7 run the softmax of tile 0 /
//     tile 1 (one thread per query row = one TMEM lane), warp 8 issues TMA
//     loads; warp 9 (as a whole warp, one elected lane issuing) issues the
//     tcgen05 MMAs of both tiles when they share K/V (GQA), or lane 0 of
//     warps 9 / 10 issues those of tile 0 / tile 1 (MHA);
//     warp 11 decodes the CTA's work items ahead into a ring in shared
//     memory (an item start costs the other roles a shared-memory read);
//   * TMEM (512 columns): S_t / P_t at column 128t (P, bf16 pairs, overwrites
//     the first half of S after it is read), O_t at 256 + 128t;
//   * the exponent is base 2 (log2 e folded into the scale); a row's
//     reference moves only to its first allowed keys' maximum and when a
//     block's sum of exponentials would reach 2^64 (so the steady state takes
//     no running maximum and the accumulator is rarely rescaled; l and O use
//     the same reference, and O / l does not depend on it);
//   * ragged lengths: the last q-block / kv-block may extend past Lq / Lk;
//     its padding is masked by the block's pattern and padding rows are
//     never stored;
//   * every wait is bounded (mbar_wait): on timeout the CTA raises an error
//     bit, stops all roles, drains its copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstddef>
#include <cmath>
#include <mutex>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace splash {
namespace {

constexpr int kThreads = 384;       // 12 warps = 3 warpgroups
// Register split (setmaxnreg): the launch gives 384 x 168; the two softmax
// warpgroups take 192 each and the producer / MMA warpgroup keeps 120:
// 2*128*192 + 128*120 = 64512 = 384*168.
constexpr int kSoftmaxRegs = 192;
constexpr int kControlRegs = 120;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Upper bound on a block row's sum of exponentials (2^64): reaching it moves
// the row's reference (no overflow in P, l or O).
constexpr float kPMax = 1.8446744e19f;
// Decoded work items handed from the decoder warp to the other roles through
// a ring in shared memory (slots, and bytes per slot).
constexpr int kItemRing = 8;
constexpr int kItemBytes = 48;
constexpr int kDecoderWarp = 11;

template <int DQK, int DV, int BK>
struct Cfg {
  static constexpr int BM = 128;                      // MMA M (rows of a query tile)
  static constexpr int QCH = DQK / 64;                // 64-column chunks of Q / K
  static constexpr int VCH = DV / 64;                 // 64-column chunks of V
  static constexpr int Q_CHUNK = BM * 128;            // bytes of a 128-row x 64-col bf16 box
  static constexpr int KV_CHUNK = BK * 128;           // bytes of a BK-row x 64-col bf16 box
  static constexpr int Q_BYTES = QCH * Q_CHUNK;
  static constexpr int K_BYTES = QCH * KV_CHUNK;
  static constexpr int V_BYTES = VCH * KV_CHUNK;
  static constexpr int TILE_BUDGET = 227 * 1024 - 2048;
  static constexpr int NK = (DQK >= 192) ? 2 : ((DQK >= 128) ? 2 : 4);
  static constexpr int NV = (DQK >= 192) ? 1 : ((DQK >= 128) ? 2 : 4);
  static constexpr int TILES = 2 * Q_BYTES + NK * K_BYTES + NV * V_BYTES;
  static_assert(TILES <= TILE_BUDGET, "shared memory budget");
  // O staging for the epilogue's TMA stores: per softmax warp, 32 rows x 64
  // columns of bf16 (128B-swizzled), when it fits next to the tiles
  static constexpr int STAGE_WARP = 32 * 128;
  static constexpr bool STAGE = TILES + 8 * STAGE_WARP <= TILE_BUDGET;
  static constexpr int STAGE_BYTES = STAGE ? 8 * STAGE_WARP : 0;
  // At dqk = 192 (one 32 KB V slot next to two 48 KB K slots) the items of
  // 256-row q-blocks stream K and V instead through a ring of NCH chunk
  // slots of one 64-column box each (the same bytes), so that V tiles are no
  // longer limited to one slot.
  static constexpr int NCH = (DQK >= 192 && BK == 128) ? (NK * K_BYTES + NV * V_BYTES) / KV_CHUNK : 0;
  static_assert(NCH == 0 || NCH * KV_CHUNK == NK * K_BYTES + NV * V_BYTES, "chunk ring covers the K/V region");
  static_assert(NCH <= 32, "chunk-slot bit masks");
  static_assert(NCH == 0 || (QCH <= 3 && VCH <= 3), "release_chunks covers at most three chunks per tile");
  // barriers: q_full[2] q_empty[2] k_full[NK] k_empty[NK] v_full[NV] v_empty[NV]
  //           s_full[2] p_full[2] o_done[2] drain ch_full[NCH] ch_empty[NCH]
  //           item_full[kItemRing] item_empty[kItemRing]
  static constexpr int NBAR = 2 + 2 + 2 * NK + 2 * NV + 2 + 2 + 2 + 1 + 2 * NCH + 2 * kItemRing;
  // tiles, O staging, barriers, TMEM address + abort flag (16), item ring
  static constexpr int SMEM = 1024 + TILES + STAGE_BYTES + NBAR * 8 + 16 + kItemRing * kItemBytes;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, BK, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, DV, true);
};

struct FwdParams {
  int32_t B, Hq, Hkv, G;
  int64_t Lq, Lk;
  int32_t bq, nq, nk, nbm;
  // an item's two 128-row query tiles: two heads of one q-block (t1_off = 0,
  // bq <= 128), or the two halves of one 256-row q-block of one head
  // (t1_off = 128; the tiles then share every K / V tile)
  int32_t t1_off;
  int32_t npairs;  // head pairs (t1_off = 0) or heads (t1_off = 128) per row
  int32_t head_group;  // items are ordered by groups of this many pairs / heads
  int32_t dense_rows;  // the mask has neither a window nor segments: rows reach across the keys
  int64_t num_items;
  const int32_t *row_ptr;
  const int32_t *active_cols;
  const int32_t *mask_next;
  const uint32_t *pattern_bits;
  const int32_t *row_order;
  // partial blocks' element masks computed from positions instead of read
  // from pattern_bits: causal / window bounds, and with segment IDs the
  // arrays [nbm][Lq] and [nbm][Lk] the table was built from
  int32_t band_bits, band_causal;
  int64_t band_wl, band_wr;
  const int32_t *seg_q, *seg_kv;
  int64_t num_patterns;
  float scale_log2;   // scale * log2(e)             (no soft cap)
  float cap_inner;    // scale / cap                 (soft cap)
  float cap_log2;     // cap * log2(e)               (soft cap)
  // cap*log2(e) * tanh(s*scale/cap) by the series, as an odd polynomial in
  // the raw score s: s * (scale_log2 + u (cap_c1 + u cap_c2)), u = s^2
  float cap_c1;       // kTanhC1 * scale^3 * log2(e) / cap^2
  float cap_c2;       // kTanhC2 * scale^5 * log2(e) / cap^4
  int32_t use_softcap;
  // Max Logit Estimate: every row's reference starts at this constant (log2
  // units, c * log2(e)) instead of its first allowed keys' maximum
  int32_t use_mle;
  float mle_ref;
  int32_t dual_issuer;  // one MMA issuer per tile (pairs with different KV heads)
  __nv_bfloat16 *out;
  float *lse;
  // split-KV: each q-block row's active list is cut into nsplit consecutive
  // ranges (separate work items); split s writes its normalized partial O
  // (fp32) and LSE at o_part / lse_part + s * part_rows rows (out / lse unused)
  int32_t nsplit;
  float *o_part;
  float *lse_part;
  int64_t part_rows;  // B * Hq * Lq
  uint32_t *err;
  uint64_t timeout_ns;
};

struct Item {
  int32_t b, h0, h1, kvh0, kvh1, qrow;
  int32_t g0, nb;  // this item's range of the row's active list
  int32_t split;
  bool act1, shared;
};
static_assert(sizeof(Item) <= kItemBytes, "item ring slot");
// nb of the item after the CTA's last one
constexpr int32_t kItemEnd = INT_MIN;

// Work item w: rows in longest-first order; for a table shared by the batch,
// each row expands into B batches; each (row, batch) into npairs head pairs;
// each of those into nsplit consecutive ranges of the row's active blocks
// (split s of nb blocks: [nb*s/nsplit, nb*(s+1)/nsplit)).
// TALL: 256-row q-blocks (p.t1_off = 128), a compile-time flag so that the
// head-pair items of the other instantiations carry no extra branch.
template <bool TALL>
__device__ __forceinline__ Item decode_item(const FwdParams &p, int64_t w) {
  Item it;
  int64_t k;
  int32_t pair;
  it.split = 0;
  if (p.nsplit > 1) {
    const int64_t base = w / p.nsplit;
    it.split = (int32_t)(w - base * p.nsplit);
    w = base;
  }
  // head groups: the items are ordered by group of head_group heads (or
  // head pairs) first, so that the CTAs running at the same time work on few
  // heads and share their K / V through L2; within a group as above
  const int64_t rows = (int64_t)p.nbm * p.nq;
  const int64_t per_b = p.nbm == 1 ? p.B : 1;
  const int64_t gsize = rows * per_b * p.head_group;
  const int64_t gi = w / gsize;
  w -= gi * gsize;
  const int32_t hbase = (int32_t)gi * p.head_group;
  const int32_t hg = min(p.head_group, p.npairs - hbase);
  {
    const int64_t per = per_b * hg;
    k = w / per;
    const int64_t rem = w - k * per;
    it.b = p.nbm == 1 ? (int32_t)(rem / hg) : -1;
    pair = hbase + (int32_t)(rem - (p.nbm == 1 ? (int64_t)it.b * hg : 0));
  }
  const int32_t mrow = p.row_order[k];
  if (p.nbm != 1) it.b = mrow / p.nq;
  it.qrow = mrow % p.nq;
  it.g0 = p.row_ptr[mrow];
  it.nb = p.row_ptr[mrow + 1] - it.g0;
  if (p.nsplit > 1) {
    const int32_t lo = (int32_t)((int64_t)it.nb * it.split / p.nsplit);
    const int32_t hi = (int32_t)((int64_t)it.nb * (it.split + 1) / p.nsplit);
    it.g0 += lo;
    it.nb = hi - lo;
  }
  if constexpr (TALL) {
    it.h0 = it.h1 = pair;
    it.act1 = (int64_t)it.qrow * p.bq + p.t1_off < p.Lq;  // the lower half holds a real row
  } else {
    it.h0 = 2 * pair;
    it.h1 = 2 * pair + 1;
    it.act1 = it.h1 < p.Hq;
  }
  it.kvh0 = it.h0 / p.G;
  it.kvh1 = it.act1 ? it.h1 / p.G : it.kvh0;
  it.shared = (it.kvh0 == it.kvh1);
  return it;
}

// Serpentine static schedule: round k of the CTA's items visits the CTAs in
// alternating directions, so that the rows (sorted longest first) spread
// evenly over the grid.  Returns the item index of round k, or -1 when done.
__device__ __forceinline__ int64_t item_of_round(const FwdParams &p, int64_t k) {
  const int64_t G = gridDim.x;
  const int64_t c = (k & 1) ? (G - 1 - blockIdx.x) : blockIdx.x;
  const int64_t w = k * G + c;
  return w < p.num_items ? w : -1;
}

__device__ __forceinline__ void raise_error(const FwdParams &p, volatile int *abort, uint32_t bits) {
  atomicOr(p.err, bits);
  *abort = 1;
}

// Maximum of N values: four independent chains of three-input maxima.
template <int N>
__device__ __forceinline__ float max_tree(const float (&v)[N]) {
  float m[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) m[x] = fmaxf(v[2 * x], v[2 * x + 1]);
#pragma unroll
  for (int j = 8; j < N; j += 2) m[(j >> 1) & 3] = fmax3(m[(j >> 1) & 3], v[j], v[j + 1]);
  return fmax3(m[0], m[1], fmaxf(m[2], m[3]));
}

// tanh for the soft cap, two ways, both from the mathematics of tanh (not
// from any library implementation):
//  * |t| <= 0.25: t * (1 + u (c1 + c2 u)), u = t^2, with c1, c2 a minimax fit
//    of tanh(t)/t on [0, 0.25] (Lawson-weighted least squares, q(0) = 1 held
//    fixed); max relative error 4.8e-7, like the Maclaurin series to t^7
//    (3.3e-7) with one multiply-add less;
//  * otherwise the identity tanh|t| = 1 - 2 / (1 + e^(2|t|)) with the sign
//    restored (absolute error ~1e-7 from ex2 / division rounding).
constexpr float kTanhC1 = -0.33324610f;
constexpr float kTanhC2 = 0.12877172f;
constexpr float kTanhSeriesLimit = 0.25f;

__device__ __forceinline__ float tanh_identity(float t) {
  const float a = fminf(fabsf(t), 16.f);  // tanh(16) rounds to 1 in fp32
  const float e = ex2_approx(2.8853900817779268f * a);  // e^(2a)
  return copysignf(1.f - __fdividef(2.f, e + 1.f), t);
}

// Shared-memory addresses of the CTA's mbarriers:
//   q_full[2] q_empty[2] k_full[NK] k_empty[NK] v_full[NV] v_empty[NV]
//   s_full[2] p_full[2] o_done[2] drain ch_full[NCH] ch_empty[NCH]
template <class C>
struct Bars {
  uint32_t base;
  __device__ __forceinline__ uint32_t q_full(int t) const { return base + 8u * t; }
  __device__ __forceinline__ uint32_t q_empty(int t) const { return base + 8u * (2 + t); }
  __device__ __forceinline__ uint32_t k_full(int s) const { return base + 8u * (4 + s); }
  __device__ __forceinline__ uint32_t k_empty(int s) const { return base + 8u * (4 + C::NK + s); }
  __device__ __forceinline__ uint32_t v_full(int s) const { return base + 8u * (4 + 2 * C::NK + s); }
  __device__ __forceinline__ uint32_t v_empty(int s) const { return base + 8u * (4 + 2 * C::NK + C::NV + s); }
  __device__ __forceinline__ uint32_t s_full(int t) const { return base + 8u * (4 + 2 * C::NK + 2 * C::NV + t); }
  __device__ __forceinline__ uint32_t p_full(int t) const { return base + 8u * (6 + 2 * C::NK + 2 * C::NV + t); }
  __device__ __forceinline__ uint32_t o_done(int t) const { return base + 8u * (8 + 2 * C::NK + 2 * C::NV + t); }
  __device__ __forceinline__ uint32_t drain() const { return base + 8u * (10 + 2 * C::NK + 2 * C::NV); }
  __device__ __forceinline__ uint32_t ch_full(uint32_t s) const { return base + 8u * (11 + 2 * C::NK + 2 * C::NV + s); }
  __device__ __forceinline__ uint32_t ch_empty(uint32_t s) const {
    return base + 8u * (11 + 2 * C::NK + 2 * C::NV + C::NCH + s);
  }
  __device__ __forceinline__ uint32_t item_full(uint32_t s) const {
    return base + 8u * (11 + 2 * C::NK + 2 * C::NV + 2 * C::NCH + s);
  }
  __device__ __forceinline__ uint32_t item_empty(uint32_t s) const {
    return base + 8u * (11 + 2 * C::NK + 2 * C::NV + 2 * C::NCH + kItemRing + s);
  }
};

// The decoded work items of this CTA, in shared memory: an array of
// kItemRing Item slots after the barriers (and the TMEM address / abort
// words).  The decoder warp (one thread) writes item k into slot
// k % kItemRing once every role has released the slot's previous item
// (item_empty), then arrives on item_full; each role waits for item k, reads
// the fields it uses (item_i32: volatile shared loads, so that only those stay
// in registers) and releases the slot.
template <class C>
__device__ __forceinline__ uint32_t item_slot(const Bars<C> &bar, int64_t k) {
  return bar.base + (uint32_t)(C::NBAR * 8 + 16) + (uint32_t)(k % kItemRing) * (uint32_t)sizeof(Item);
}

// A 32-bit field of an item slot (offsetof(Item, field)).
__device__ __forceinline__ int32_t item_i32(uint32_t addr, size_t offset) {
  int32_t v;
  asm volatile("ld.volatile.shared.s32 %0, [%1];" : "=r"(v) : "r"(addr + (uint32_t)offset));
  return v;
}

// The two flag bytes of an item (act1, shared), from one 32-bit load.
__device__ __forceinline__ void item_flags(uint32_t addr, bool &act1, bool &shared) {
  static_assert(offsetof(Item, shared) == offsetof(Item, act1) + 1 && offsetof(Item, act1) % 4 == 0, "flag bytes");
  const int32_t w = item_i32(addr, offsetof(Item, act1));
  act1 = (w & 0xff) != 0;
  shared = ((w >> 8) & 0xff) != 0;
}

// Waits for item k (one thread).  Returns its slot address, or 0 after the
// CTA's last item (the slot is then released) or with ok = false; the caller
// releases the slot with release_item once it has read the fields.
template <class C>
__device__ __forceinline__ uint32_t hold_item(const Bars<C> &bar, int64_t k, bool &ok, volatile int *abort,
                                              uint64_t timeout_ns) {
  const uint32_t s = (uint32_t)(k % kItemRing);
  ok = mbar_wait(bar.item_full(s), (uint32_t)(k / kItemRing) & 1u, abort, timeout_ns);
  if (!ok) return 0u;
  const uint32_t addr = item_slot(bar, k);
  if (item_i32(addr, offsetof(Item, nb)) == kItemEnd) {
    mbar_arrive(bar.item_empty(s));
    return 0u;
  }
  return addr;
}

template <class C>
__device__ __forceinline__ void release_item(const Bars<C> &bar, int64_t k) {
  mbar_arrive(bar.item_empty((uint32_t)(k % kItemRing)));
}

// The same for a whole, converged warp (one arrival per warp).
template <class C>
__device__ __forceinline__ uint32_t hold_item_warp(const Bars<C> &bar, int64_t k, bool &ok, volatile int *abort,
                                                   uint64_t timeout_ns) {
  const uint32_t s = (uint32_t)(k % kItemRing);
  ok = __all_sync(0xffffffffu, mbar_wait(bar.item_full(s), (uint32_t)(k / kItemRing) & 1u, abort, timeout_ns));
  if (!ok) return 0u;
  const uint32_t addr = item_slot(bar, k);
  if (item_i32(addr, offsetof(Item, nb)) == kItemEnd) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar.item_empty(s));
    return 0u;
  }
  return addr;
}

template <class C>
__device__ __forceinline__ void release_item_warp(const Bars<C> &bar, int64_t k) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar.item_empty((uint32_t)(k % kItemRing)));
}

// The decoder (one thread of warp kDecoderWarp): decodes this CTA's items
// ahead of the roles that use them, so that an item start costs them a few
// shared-memory reads instead of the table loads and index arithmetic.
template <class C, bool TALL>
__device__ __noinline__ void run_decoder(const FwdParams &p, const Bars<C> bar, Item *items, volatile int *abort) {
  bool ok = true;
  for (int64_t k = 0;; ++k) {
    const uint32_t s = (uint32_t)(k % kItemRing);
    if (k >= kItemRing &&
        !(ok = mbar_wait(bar.item_empty(s), (uint32_t)((k / kItemRing) - 1) & 1u, abort, p.timeout_ns)))
      break;
    const int64_t w = item_of_round(p, k);
    Item it;
    if (w < 0) {
      it = Item{};
      it.nb = kItemEnd;
    } else {
      it = decode_item<TALL>(p, w);
    }
    items[s] = it;
    mbar_arrive(bar.item_full(s));  // release: the item's stores come first
    if (w < 0) break;
  }
  if (!ok) raise_error(p, abort, SPLASH_DEV_TIMEOUT_PRODUCER);
}

// Loads one K or V tile (CH boxes of 64 columns x BK rows) into the next slot
// of a ring of NS slots of BYTES bytes; waits (bounded) for the slot to be
// released by the MMAs that read its previous contents.
template <int NS, int BYTES, int CH, int CHUNK>
__device__ __forceinline__ bool produce_tile(const FwdParams &p, const CUtensorMap *tm, uint32_t ring,
                                             uint32_t full0, uint32_t empty0, uint32_t &cnt, int32_t y,
                                             volatile int *abort) {
  const uint32_t s = cnt % NS;
  if (cnt >= (uint32_t)NS && !mbar_wait(empty0 + 8u * s, ((cnt / NS) - 1u) & 1u, abort, p.timeout_ns))
    return false;
  mbar_arrive_expect_tx(full0 + 8u * s, BYTES);
#pragma unroll
  for (int ch = 0; ch < CH; ++ch) tma_load_2d(ring + s * BYTES + ch * CHUNK, tm, ch * 64, y, full0 + 8u * s);
  ++cnt;
  return true;
}

__device__ __forceinline__ int32_t checked_col(const FwdParams &p, int32_t g) {
  int32_t c = p.active_cols[g];
  if (c < 0 || c >= p.nk) {
    atomicOr(p.err, SPLASH_DEV_BAD_TABLE);
    c = 0;
  }
  return c;
}

// The TMA producer (one thread): per work item the two Q tiles, then K and V
// tiles in exactly the order the MMA issuer consumes them:
//   K0(0) [K1(0)], then per block g: V0(g) K0(g+1) [V1(g) K1(g+1)]
// (the bracketed loads only when the two query heads use different KV heads).
template <class C, int BK, bool TALL>
__device__ __noinline__ void run_producer(const FwdParams &p, const CUtensorMap *tmQ, const CUtensorMap *tmK,
                                          const CUtensorMap *tmV, uint32_t sQ, uint32_t sK, uint32_t sV,
                                          const Bars<C> bar, volatile int *abort) {
  uint32_t kcnt = 0, vcnt = 0, q0 = 0, q1 = 0;
  bool ok = true;
  for (int64_t k = 0; ok; ++k) {
    const uint32_t ia = hold_item(bar, k, ok, abort, p.timeout_ns);
    if (ia == 0u) break;
    Item it;
    it.nb = item_i32(ia, offsetof(Item, nb));
    it.g0 = item_i32(ia, offsetof(Item, g0));
    it.b = item_i32(ia, offsetof(Item, b));
    it.h0 = item_i32(ia, offsetof(Item, h0));
    it.h1 = item_i32(ia, offsetof(Item, h1));
    it.kvh0 = item_i32(ia, offsetof(Item, kvh0));
    it.kvh1 = item_i32(ia, offsetof(Item, kvh1));
    it.qrow = item_i32(ia, offsetof(Item, qrow));
    item_flags(ia, it.act1, it.shared);
    release_item(bar, k);
    if (it.nb <= 0) continue;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (t == 1 && !it.act1) break;
      uint32_t &qc = t ? q1 : q0;
      if (qc > 0 && !mbar_wait(bar.q_empty(t), (qc - 1) & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(bar.q_full(t), C::Q_BYTES);
      const int32_t y = (int32_t)(((int64_t)it.b * p.Hq + (t ? it.h1 : it.h0)) * p.Lq + (int64_t)it.qrow * p.bq +
                                  ((TALL && t) ? 128 : 0));
#pragma unroll
      for (int ch = 0; ch < C::QCH; ++ch)
        tma_load_2d(sQ + t * C::Q_BYTES + ch * C::Q_CHUNK, tmQ, ch * 64, y, bar.q_full(t));
      ++qc;
    }
    if (!ok) break;
    const bool two_kv = it.act1 && !it.shared;
    const int64_t kv0 = ((int64_t)it.b * p.Hkv + it.kvh0) * p.Lk;
    const int64_t kv1 = ((int64_t)it.b * p.Hkv + it.kvh1) * p.Lk;
    int32_t c = checked_col(p, it.g0);
    ok = produce_tile<C::NK, C::K_BYTES, C::QCH, C::KV_CHUNK>(p, tmK, sK, bar.k_full(0), bar.k_empty(0), kcnt,
                                                              (int32_t)(kv0 + (int64_t)c * BK), abort);
    if (ok && two_kv)
      ok = produce_tile<C::NK, C::K_BYTES, C::QCH, C::KV_CHUNK>(p, tmK, sK, bar.k_full(0), bar.k_empty(0), kcnt,
                                                                (int32_t)(kv1 + (int64_t)c * BK), abort);
    for (int32_t g = 0; g < it.nb && ok; ++g) {
      const bool more = g + 1 < it.nb;
      const int32_t cn = more ? checked_col(p, it.g0 + g + 1) : 0;
      ok = produce_tile<C::NV, C::V_BYTES, C::VCH, C::KV_CHUNK>(p, tmV, sV, bar.v_full(0), bar.v_empty(0), vcnt,
                                                                (int32_t)(kv0 + (int64_t)c * BK), abort);
      if (ok && more)
        ok = produce_tile<C::NK, C::K_BYTES, C::QCH, C::KV_CHUNK>(p, tmK, sK, bar.k_full(0), bar.k_empty(0), kcnt,
                                                                  (int32_t)(kv0 + (int64_t)cn * BK), abort);
      if (ok && two_kv)
        ok = produce_tile<C::NV, C::V_BYTES, C::VCH, C::KV_CHUNK>(p, tmV, sV, bar.v_full(0), bar.v_empty(0),
                                                                  vcnt, (int32_t)(kv1 + (int64_t)c * BK), abort);
      if (ok && two_kv && more)
        ok = produce_tile<C::NK, C::K_BYTES, C::QCH, C::KV_CHUNK>(p, tmK, sK, bar.k_full(0), bar.k_empty(0),
                                                                  kcnt, (int32_t)(kv1 + (int64_t)cn * BK), abort);
      c = cn;
    }
  }
  if (!ok) raise_error(p, abort, SPLASH_DEV_TIMEOUT_PRODUCER);
  // drain: the last load issued into every slot has landed
  bool drained = true;
  for (int s = 0; s < C::NK; ++s)
    if (kcnt > (uint32_t)s) drained &= mbar_wait_drain(bar.k_full(s), ((kcnt - 1 - s) / C::NK) & 1, p.timeout_ns);
  for (int s = 0; s < C::NV; ++s)
    if (vcnt > (uint32_t)s) drained &= mbar_wait_drain(bar.v_full(s), ((vcnt - 1 - s) / C::NV) & 1, p.timeout_ns);
  if (q0 > 0) drained &= mbar_wait_drain(bar.q_full(0), (q0 - 1) & 1, p.timeout_ns);
  if (q1 > 0) drained &= mbar_wait_drain(bar.q_full(1), (q1 - 1) & 1, p.timeout_ns);
  if (!drained) atomicOr(p.err, SPLASH_DEV_TIMEOUT_DRAIN);
}

// S_t = Q_t K^T: QCH chunks x 4 MMAs of K = 16 (K-major A and B, 128B swizzle;
// the k-step advances the start address by 32 bytes inside the swizzle atom).
// Descriptors are passed as their low halves; the high halves are constants.
// Only the lane with `leader` != 0 issues (mma_ss_lhp / mma_ts_lhp).
template <class C>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr, uint32_t leader) {
  constexpr uint32_t HI = sdesc_hi_sw128(1024);
  const uint32_t qd = sdesc_lo(q_addr, 16), kd = sdesc_lo(k_addr, 16);
#pragma unroll
  for (int ch = 0; ch < C::QCH; ++ch)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lhp(leader, d_tmem, qd + (uint32_t)((ch * C::Q_CHUNK + kk * 32) >> 4), HI,
                 kd + (uint32_t)((ch * C::KV_CHUNK + kk * 32) >> 4), HI, C::IDESC_QK, (ch | kk) != 0);
}

// O_t (+)= P_t V: P read from TMEM (bf16 pairs, 8 columns per K = 16 step),
// V MN-major with 128B swizzle (K step = 16 rows = 2048 bytes; the 64-column
// chunks of V are KV_CHUNK bytes apart).
template <class C, int BK>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr, bool first_block,
                                         uint32_t leader) {
  constexpr uint32_t HI = sdesc_hi_sw128(1024);
  const uint32_t vd = sdesc_lo(v_addr, C::KV_CHUNK);
#pragma unroll
  for (int j = 0; j < BK / 16; ++j)
    mma_ts_lhp(leader, d_tmem, p_tmem + 8u * j, vd + (uint32_t)((j * 2048) >> 4), HI, C::IDESC_PV,
               (!first_block || j > 0) ? 1u : 0u);
}

__device__ __forceinline__ bool wait_ring(uint32_t full0, uint32_t cnt, int ns, volatile int *abort,
                                          uint64_t timeout_ns, uint32_t &slot) {
  slot = cnt % (uint32_t)ns;
  if (!mbar_wait(full0 + 8u * slot, (cnt / (uint32_t)ns) & 1u, abort, timeout_ns)) return false;
  tc_fence_after();
  return true;
}

// Per-ring bookkeeping of one MMA issuer.  Uses of the ring are numbered in
// the producer's order; the empty barrier of a slot counts two releases per
// use, one from each issuer: a commit from the issuer whose MMAs read the slot
// (it arrives when they complete), a plain arrive from the other one, given
// only after the use's data has landed.  An issuer never waits on a use while
// an earlier use of the same ring is unreleased by it; issuer 0 defers its
// release of tile 1's use (always the later of a pair) to its next step.
struct RingState {
  uint32_t cnt;      // next use
  uint32_t pending;  // a deferred plain release, valid when has_pending
  bool has_pending;
};

__device__ __forceinline__ bool plain_release(uint32_t full0, uint32_t empty0, uint32_t use, int ns,
                                              volatile int *abort, uint64_t timeout_ns) {
  const uint32_t slot = use % (uint32_t)ns;
  if (!mbar_wait(full0 + 8u * slot, (use / (uint32_t)ns) & 1u, abort, timeout_ns)) return false;
  mbar_arrive(empty0 + 8u * slot);
  return true;
}

__device__ __forceinline__ bool flush_pending(RingState &r, uint32_t full0, uint32_t empty0, int ns,
                                              volatile int *abort, uint64_t timeout_ns) {
  if (!r.has_pending) return true;
  r.has_pending = false;
  return plain_release(full0, empty0, r.pending, ns, abort, timeout_ns);
}

// One step of a ring: the tile-0 and tile-1 uses of one K or V tile (one use
// when both tiles share it).  Waits for this issuer's use, and returns its
// slot in `slot` (use_it = false when this issuer has no MMA on it).
__device__ __forceinline__ bool ring_step_acquire(RingState &r, uint32_t full0, uint32_t empty0, int ns, int t,
                                                  bool two_kv, bool mine, volatile int *abort, uint64_t timeout_ns,
                                                  uint32_t &slot, uint32_t &use) {
  if (!flush_pending(r, full0, empty0, ns, abort, timeout_ns)) return false;
  if (two_kv && t == 1) {
    // tile 0's use comes first in the ring: release it before waiting on ours
    if (!plain_release(full0, empty0, r.cnt, ns, abort, timeout_ns)) return false;
  }
  use = (two_kv && t == 1) ? r.cnt + 1 : r.cnt;
  slot = use % (uint32_t)ns;
  if (!mine) return plain_release(full0, empty0, use, ns, abort, timeout_ns);
  if (!mbar_wait(full0 + 8u * slot, (use / (uint32_t)ns) & 1u, abort, timeout_ns)) return false;
  tc_fence_after();
  return true;
}

// After this issuer's MMAs on the step's slot: commit its release, defer or
// skip the other tile's, advance the ring.
__device__ __forceinline__ void ring_step_release(RingState &r, uint32_t empty0, int ns, int t, bool two_kv,
                                                  bool mine, uint32_t use) {
  if (mine) tc_commit(empty0 + 8u * (use % (uint32_t)ns));
  if (two_kv && t == 0) {
    r.pending = r.cnt + 1;
    r.has_pending = true;
  }
  r.cnt += two_kv ? 2u : 1u;
}

// An MMA issuer (one thread per query tile t).  Per item: S_t(0) = Q_t K(0)^T;
// then per block g: wait P_t(g): O_t += P_t V(g); S_t(g+1) = Q_t K(g+1)^T.
// Both issuers walk the same K / V ring sequence (the producer's order:
// K0(0) [K1(0)], then per block V0(g) K0(g+1) [V1(g) K1(g+1)]).  Commits:
// s_full after each S, o_done after the last PV, q_empty after the tile's
// last S.  Two issuers keep one tile's MMA burst from waiting behind the
// other's in the tensor pipe's queue.
template <class C, int BK, bool TALL>
__device__ __noinline__ void run_mma(const FwdParams &p, uint32_t tmem, uint32_t sQ, uint32_t sK, uint32_t sV,
                                     const Bars<C> bar, volatile int *abort, const int t) {
  RingState kr{0u, 0u, false}, vr{0u, 0u, false};
  uint32_t qc = 0, pc = 0;
  bool ok = true;
  const uint32_t tS = tmem + 128u * t, tO = tmem + 256u + 128u * t;
  const uint32_t sQt = sQ + t * C::Q_BYTES;
  for (int64_t k = 0; ok; ++k) {
    const uint32_t ia = hold_item(bar, k, ok, abort, p.timeout_ns);
    if (ia == 0u) break;
    Item it;
    it.nb = item_i32(ia, offsetof(Item, nb));
    item_flags(ia, it.act1, it.shared);
    release_item(bar, k);
    if (it.nb <= 0) continue;
    const bool mine = (t == 0) || it.act1;
    const bool two_kv = it.act1 && !it.shared;
    if (mine) {
      if (!(ok = mbar_wait(bar.q_full(t), qc & 1, abort, p.timeout_ns))) break;
      ++qc;
      tc_fence_after();
    }
    uint32_t slot, use;
    // S_t(0)
    if (!(ok = ring_step_acquire(kr, bar.k_full(0), bar.k_empty(0), C::NK, t, two_kv, mine, abort, p.timeout_ns,
                                 slot, use)))
      break;
    if (mine) {
      issue_qk<C>(tS, sQt, sK + slot * C::K_BYTES, 1u);
      tc_commit(bar.s_full(t));
      if (it.nb == 1) tc_commit(bar.q_empty(t));
    }
    ring_step_release(kr, bar.k_empty(0), C::NK, t, two_kv, mine, use);
    for (int32_t g = 0; g < it.nb && ok; ++g) {
      const bool more = g + 1 < it.nb;
      // O_t += P_t V(g)
      if (mine) {
        if (!(ok = mbar_wait(bar.p_full(t), pc & 1, abort, p.timeout_ns))) break;
        ++pc;
        tc_fence_after();
      }
      if (!(ok = ring_step_acquire(vr, bar.v_full(0), bar.v_empty(0), C::NV, t, two_kv, mine, abort,
                                   p.timeout_ns, slot, use)))
        break;
      if (mine) {
        issue_pv<C, BK>(tO, tS, sV + slot * C::V_BYTES, g == 0, 1u);
        if (!more) tc_commit(bar.o_done(t));
      }
      ring_step_release(vr, bar.v_empty(0), C::NV, t, two_kv, mine, use);
      if (!more) break;
      // S_t(g+1) = Q_t K(g+1)^T
      if (!(ok = ring_step_acquire(kr, bar.k_full(0), bar.k_empty(0), C::NK, t, two_kv, mine, abort,
                                   p.timeout_ns, slot, use)))
        break;
      if (mine) {
        issue_qk<C>(tS, sQt, sK + slot * C::K_BYTES, 1u);
        tc_commit(bar.s_full(t));
        if (g + 2 == it.nb) tc_commit(bar.q_empty(t));
      }
      ring_step_release(kr, bar.k_empty(0), C::NK, t, two_kv, mine, use);
    }
  }
  if (ok) ok = flush_pending(kr, bar.k_full(0), bar.k_empty(0), C::NK, abort, p.timeout_ns) &&
               flush_pending(vr, bar.v_full(0), bar.v_empty(0), C::NV, abort, p.timeout_ns);
  if (!ok) raise_error(p, abort, SPLASH_DEV_TIMEOUT_MMA);
  // drain: every MMA issued by this thread has completed (the barrier counts
  // both issuers)
  tc_commit(bar.drain());
  if (!mbar_wait_drain(bar.drain(), 0, p.timeout_ns)) atomicOr(p.err, SPLASH_DEV_TIMEOUT_DRAIN);
}

// Waits for the phase `pph` of barrier `pb` and, when needed, for the ring
// tiles (V slot, K slot) the MMAs after it read.  The barriers are first
// polled together, so that one poll's latency covers all of them; the bounded
// waits one by one are the fallback.
__device__ __forceinline__ bool wait_ready(uint32_t pb, uint32_t pph, bool need_v, uint32_t vb, uint32_t vph,
                                           bool need_k, uint32_t kb, uint32_t kph, volatile int *abort,
                                           uint64_t timeout_ns) {
  bool r;
  if (need_v && need_k)
    r = mbar_try_wait3(pb, pph, vb, vph, kb, kph);
  else if (need_v)
    r = mbar_try_wait2(pb, pph, vb, vph);
  else if (need_k)
    r = mbar_try_wait2(pb, pph, kb, kph);
  else
    r = mbar_try_wait(pb, pph);
  if (r) return true;
  return mbar_wait(pb, pph, abort, timeout_ns) && (!need_v || mbar_wait(vb, vph, abort, timeout_ns)) &&
         (!need_k || mbar_wait(kb, kph, abort, timeout_ns));
}

// The single MMA issuer for both tiles, used when the tiles share their K / V
// tiles (GQA heads of one group).  It runs as a whole, converged warp: every
// lane waits and computes the same (warp-uniform) ring state and descriptors,
// and the elected lane `leader` issues the MMAs and commits.  (Measured on
// GB300: a burst of MMAs issued this way costs ~17 cycles per MMA, against
// ~50 from one lane of a diverged warp and ~68 when softmax warps share the
// sub-partition; a 128x128x16 MMA executes in ~64.)
// Per item: S_0(0), S_1(0); then per block g:
//   wait P_0(g): O_0 += P_0 V(g); S_0(g+1) = Q_0 K(g+1)^T;
//   wait P_1(g): O_1 += P_1 V(g); S_1(g+1) = Q_1 K(g+1)^T.
// Commits: s_full after each S, o_done after the last PV, slot releases
// after the last MMA that reads a slot, q_empty after a tile's last S.
template <class C, int BK, bool TALL>
__device__ __forceinline__ void run_mma_pair(const FwdParams &p, uint32_t tmem, uint32_t sQ, uint32_t sK, uint32_t sV,
                                     const Bars<C> bar, volatile int *abort, const uint32_t leader) {
  const uint64_t tmo = p.timeout_ns;
  uint32_t kcnt = 0, vcnt = 0, q0 = 0, q1 = 0, p0 = 0, p1 = 0;
  bool ok = true;
  const uint32_t tS0 = tmem, tS1 = tmem + 128u, tO0 = tmem + 256u, tO1 = tmem + 384u;
  for (int64_t k = 0; ok; ++k) {
    const uint32_t ia = hold_item_warp(bar, k, ok, abort, p.timeout_ns);
    if (ia == 0u) break;
    Item it;
    it.nb = item_i32(ia, offsetof(Item, nb));
    item_flags(ia, it.act1, it.shared);
    release_item_warp(bar, k);
    if (it.nb <= 0) continue;
    const bool two = it.act1;
    const bool two_kv = it.act1 && !it.shared;
    // S_0(0) [and S_1(0)]: Q tiles and the first K tile
    uint32_t ks = kcnt % C::NK;
    if (!(ok = wait_ready(bar.q_full(0), q0 & 1u, two, bar.q_full(1), q1 & 1u, true, bar.k_full(ks),
                          (kcnt / C::NK) & 1u, abort, tmo)))
      break;
    ++q0;
    if (two) ++q1;
    tc_fence_after();
    issue_qk<C>(tS0, sQ, sK + ks * C::K_BYTES, leader);
    tc_commit_p(leader, bar.s_full(0));
    if (two_kv) {
      tc_commit_p(leader, bar.k_empty(ks));
      ++kcnt;
      if (!(ok = wait_ring(bar.k_full(0), kcnt, C::NK, abort, tmo, ks))) break;
    }
    if (two) {
      issue_qk<C>(tS1, sQ + C::Q_BYTES, sK + ks * C::K_BYTES, leader);
      tc_commit_p(leader, bar.s_full(1));
    }
    tc_commit_p(leader, bar.k_empty(ks));
    ++kcnt;
    if (it.nb == 1) {
      tc_commit_p(leader, bar.q_empty(0));
      if (two) tc_commit_p(leader, bar.q_empty(1));
    }
    for (int32_t g = 0; g < it.nb && ok; ++g) {
      const bool more = g + 1 < it.nb;
      // ---- tile 0: P_0(g), V(g) and K(g+1)
      const uint32_t vs0 = vcnt % C::NV, ks0 = kcnt % C::NK;
      if (!(ok = wait_ready(bar.p_full(0), p0 & 1u, true, bar.v_full(vs0), (vcnt / C::NV) & 1u, more,
                            bar.k_full(ks0), (kcnt / C::NK) & 1u, abort, tmo)))
        break;
      ++p0;
      tc_fence_after();
      issue_pv<C, BK>(tO0, tS0, sV + vs0 * C::V_BYTES, g == 0, leader);
      if (!more) tc_commit_p(leader, bar.o_done(0));
      if (!two || two_kv) {
        tc_commit_p(leader, bar.v_empty(vs0));
        ++vcnt;
      }
      if (more) {
        issue_qk<C>(tS0, sQ, sK + ks0 * C::K_BYTES, leader);
        tc_commit_p(leader, bar.s_full(0));
        if (!two || two_kv) {
          tc_commit_p(leader, bar.k_empty(ks0));
          ++kcnt;
        }
        if (g + 2 == it.nb) tc_commit_p(leader, bar.q_empty(0));
      }
      if (!two) continue;
      // ---- tile 1: P_1(g) [and its own V(g), K(g+1)]
      const uint32_t vs1 = two_kv ? vcnt % C::NV : vs0, ks1 = two_kv ? kcnt % C::NK : ks0;
      if (!(ok = wait_ready(bar.p_full(1), p1 & 1u, two_kv, bar.v_full(vs1), (vcnt / C::NV) & 1u,
                            two_kv && more, bar.k_full(ks1), (kcnt / C::NK) & 1u, abort, tmo)))
        break;
      ++p1;
      tc_fence_after();
      issue_pv<C, BK>(tO1, tS1, sV + vs1 * C::V_BYTES, g == 0, leader);
      if (!more) tc_commit_p(leader, bar.o_done(1));
      tc_commit_p(leader, bar.v_empty(vs1));
      ++vcnt;
      if (more) {
        issue_qk<C>(tS1, sQ + C::Q_BYTES, sK + ks1 * C::K_BYTES, leader);
        tc_commit_p(leader, bar.s_full(1));
        tc_commit_p(leader, bar.k_empty(ks1));
        ++kcnt;
        if (g + 2 == it.nb) tc_commit_p(leader, bar.q_empty(1));
      }
    }
  }
  if (!ok && leader) raise_error(p, abort, SPLASH_DEV_TIMEOUT_MMA);
  // drain: every MMA issued by this thread has completed
  tc_commit_p(leader, bar.drain());
  if (!mbar_wait_drain(bar.drain(), 0, tmo) && leader) atomicOr(p.err, SPLASH_DEV_TIMEOUT_DRAIN);
}

// ---------------------------------------------------------------- chunk ring
// Items of 256-row q-blocks at dqk = 192: both tiles read every K / V tile,
// and the K / V region is a ring of NCH chunk slots (one 64-column x BK-row
// box each).  Chunk n of the stream goes to slot n % NCH; a K tile is QCH
// consecutive chunks, a V tile VCH, in the issuer's order
//   K(0), then per block g: V(g), K(g+1)
// and a tile's chunks need not be adjacent in shared memory.  Each chunk is
// released on its own barrier (ch_empty, one commit per use) as soon as the
// MMAs that read it have completed, so the loads of the next tiles start
// chunk by chunk instead of waiting for a whole slot.  A tile completes on
// the full barrier of its first chunk's slot (armed with the whole tile's
// bytes), so the issuer waits once per tile; since which slots start a tile
// varies, both sides track those barriers' phases per slot (bit masks).
//
// Phase safety: the producer arms ch_full(s) only after waiting for
// ch_empty(s), i.e. after the issuer has released the chunk that last used
// slot s; the issuer consumes tiles in stream order, so by then it has
// waited for every earlier tile, including the last one armed on ch_full(s).

// One K or V tile of `nch` chunks at global row y, streamed into the ring.
template <class C>
__device__ __forceinline__ bool produce_tile_chunked(const FwdParams &p, const CUtensorMap *tm, uint32_t ring,
                                                     const Bars<C> &bar, uint32_t &n, uint32_t &armed,
                                                     uint32_t &arm_par, int nch, int32_t y, volatile int *abort) {
  const uint32_t first = n % C::NCH;
  for (int ch = 0; ch < nch; ++ch, ++n) {
    const uint32_t s = n % C::NCH;
    if (n >= (uint32_t)C::NCH && !mbar_wait(bar.ch_empty(s), ((n / C::NCH) - 1u) & 1u, abort, p.timeout_ns))
      return false;
    if (ch == 0) {
      mbar_arrive_expect_tx(bar.ch_full(first), (uint32_t)(nch * C::KV_CHUNK));
      armed |= 1u << first;
      arm_par ^= 1u << first;  // bit = number of armings of the slot, mod 2
    }
    tma_load_2d(ring + s * C::KV_CHUNK, tm, ch * 64, y, bar.ch_full(first));
  }
  return true;
}

template <class C, int BK>
__device__ __noinline__ void run_producer_chunked(const FwdParams &p, const CUtensorMap *tmQ, const CUtensorMap *tmK,
                                                  const CUtensorMap *tmV, uint32_t sQ, uint32_t ring,
                                                  const Bars<C> bar, volatile int *abort) {
  uint32_t n = 0, armed = 0, arm_par = 0, q0 = 0, q1 = 0;
  bool ok = true;
  for (int64_t k = 0; ok; ++k) {
    const uint32_t ia = hold_item(bar, k, ok, abort, p.timeout_ns);
    if (ia == 0u) break;
    Item it;
    it.nb = item_i32(ia, offsetof(Item, nb));
    it.g0 = item_i32(ia, offsetof(Item, g0));
    it.b = item_i32(ia, offsetof(Item, b));
    it.h0 = item_i32(ia, offsetof(Item, h0));
    it.h1 = item_i32(ia, offsetof(Item, h1));
    it.kvh0 = item_i32(ia, offsetof(Item, kvh0));
    it.kvh1 = item_i32(ia, offsetof(Item, kvh1));
    it.qrow = item_i32(ia, offsetof(Item, qrow));
    item_flags(ia, it.act1, it.shared);
    release_item(bar, k);
    if (it.nb <= 0) continue;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (t == 1 && !it.act1) break;
      uint32_t &qc = t ? q1 : q0;
      if (qc > 0 && !mbar_wait(bar.q_empty(t), (qc - 1) & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(bar.q_full(t), C::Q_BYTES);
      const int32_t y = (int32_t)(((int64_t)it.b * p.Hq + it.h0) * p.Lq + (int64_t)it.qrow * p.bq + 128 * t);
#pragma unroll
      for (int ch = 0; ch < C::QCH; ++ch)
        tma_load_2d(sQ + t * C::Q_BYTES + ch * C::Q_CHUNK, tmQ, ch * 64, y, bar.q_full(t));
      ++qc;
    }
    if (!ok) break;
    const int64_t kv0 = ((int64_t)it.b * p.Hkv + it.kvh0) * p.Lk;
    int32_t c = checked_col(p, it.g0);
    ok = produce_tile_chunked<C>(p, tmK, ring, bar, n, armed, arm_par, C::QCH, (int32_t)(kv0 + (int64_t)c * BK),
                                 abort);
    for (int32_t g = 0; g < it.nb && ok; ++g) {
      const bool more = g + 1 < it.nb;
      const int32_t cn = more ? checked_col(p, it.g0 + g + 1) : 0;
      ok = produce_tile_chunked<C>(p, tmV, ring, bar, n, armed, arm_par, C::VCH, (int32_t)(kv0 + (int64_t)c * BK),
                                   abort);
      if (ok && more)
        ok = produce_tile_chunked<C>(p, tmK, ring, bar, n, armed, arm_par, C::QCH,
                                     (int32_t)(kv0 + (int64_t)cn * BK), abort);
      c = cn;
    }
  }
  if (!ok) raise_error(p, abort, SPLASH_DEV_TIMEOUT_PRODUCER);
  // drain: the last tile armed on every slot has landed (its phase parity is
  // the number of armings minus one, mod 2)
  bool drained = true;
  for (int s = 0; s < C::NCH; ++s)
    if ((armed >> s) & 1u) drained &= mbar_wait_drain(bar.ch_full(s), ((arm_par >> s) & 1u) ^ 1u, p.timeout_ns);
  if (q0 > 0) drained &= mbar_wait_drain(bar.q_full(0), (q0 - 1) & 1, p.timeout_ns);
  if (q1 > 0) drained &= mbar_wait_drain(bar.q_full(1), (q1 - 1) & 1, p.timeout_ns);
  if (!drained) atomicOr(p.err, SPLASH_DEV_TIMEOUT_DRAIN);
}

// S_t = Q_t K^T with the K tile's chunk ch in ring slot (first + ch) % NCH.
template <class C>
__device__ __forceinline__ void issue_qk_chunked(uint32_t d_tmem, uint32_t q_addr, uint32_t ring, uint32_t first,
                                                 uint32_t leader) {
  constexpr uint32_t HI = sdesc_hi_sw128(1024);
  const uint32_t qd = sdesc_lo(q_addr, 16);
#pragma unroll
  for (int ch = 0; ch < C::QCH; ++ch) {
    const uint32_t kd = sdesc_lo(ring + ((first + ch) % C::NCH) * C::KV_CHUNK, 16);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lhp(leader, d_tmem, qd + (uint32_t)((ch * C::Q_CHUNK + kk * 32) >> 4), HI,
                 kd + (uint32_t)((kk * 32) >> 4), HI, C::IDESC_QK, (ch | kk) != 0);
  }
}

// O_t (+)= P_t V, one N = 64 MMA chain per V chunk (the chunks need not be
// adjacent, so each is its own MN-major operand): output columns 64h..64h+63
// of O_t from chunk h.
template <class C, int BK>
__device__ __forceinline__ void issue_pv_chunked(uint32_t d_tmem, uint32_t p_tmem, uint32_t ring, uint32_t first,
                                                 bool first_block, uint32_t leader) {
  constexpr uint32_t HI = sdesc_hi_sw128(1024);
  constexpr uint32_t IDESC_PV64 = idesc_bf16_f32(128, 64, true);  // N = one 64-column V chunk
#pragma unroll
  for (int h = 0; h < C::VCH; ++h) {
    const uint32_t vd = sdesc_lo(ring + ((first + h) % C::NCH) * C::KV_CHUNK, C::KV_CHUNK);
#pragma unroll
    for (int j = 0; j < BK / 16; ++j)
      mma_ts_lhp(leader, d_tmem + 64u * h, p_tmem + 8u * j, vd + (uint32_t)((j * 2048) >> 4), HI, IDESC_PV64,
                 (!first_block || j > 0) ? 1u : 0u);
  }
}

// Releases chunks first .. first+nch-1 when the MMAs issued so far complete.
template <class C>
__device__ __forceinline__ void release_chunks(const Bars<C> &bar, uint32_t first, int nch, uint32_t leader) {
#pragma unroll
  for (int ch = 0; ch < 3; ++ch)
    if (ch < nch) tc_commit_p(leader, bar.ch_empty((first + ch) % C::NCH));
}

// The single MMA issuer for items of 256-row q-blocks on the chunk ring (the
// run_mma_pair schedule with shared K / V):
//   S_0(0), S_1(0); then per block g:
//   wait P_0(g): O_0 += P_0 V(g); S_0(g+1) = Q_0 K(g+1)^T;
//   wait P_1(g): O_1 += P_1 V(g); S_1(g+1) = Q_1 K(g+1)^T.
// A tile's chunks are released after the last MMA that reads them (tile 1's,
// or tile 0's when the lower half of the block is all padding).
template <class C, int BK>
__device__ __forceinline__ void run_mma_pair_chunked(const FwdParams &p, uint32_t tmem, uint32_t sQ, uint32_t ring,
                                                     const Bars<C> bar, volatile int *abort,
                                                     const uint32_t leader) {
  const uint64_t tmo = p.timeout_ns;
  uint32_t n = 0, fwait = 0, q0 = 0, q1 = 0, p0 = 0, p1 = 0;
  bool ok = true;
  const uint32_t tS0 = tmem, tS1 = tmem + 128u, tO0 = tmem + 256u, tO1 = tmem + 384u;
  for (int64_t k = 0; ok; ++k) {
    const uint32_t ia = hold_item_warp(bar, k, ok, abort, p.timeout_ns);
    if (ia == 0u) break;
    Item it;
    it.nb = item_i32(ia, offsetof(Item, nb));
    item_flags(ia, it.act1, it.shared);
    release_item_warp(bar, k);
    if (it.nb <= 0) continue;
    const bool two = it.act1;
    // S_0(0) [and S_1(0)]: Q tiles and the first K tile
    const uint32_t kf0 = n, ks0 = kf0 % C::NCH;
    if (!(ok = wait_ready(bar.q_full(0), q0 & 1u, two, bar.q_full(1), q1 & 1u, true, bar.ch_full(ks0),
                          (fwait >> ks0) & 1u, abort, tmo)))
      break;
    fwait ^= 1u << ks0;
    n += C::QCH;
    ++q0;
    if (two) ++q1;
    tc_fence_after();
    issue_qk_chunked<C>(tS0, sQ, ring, kf0, leader);
    tc_commit_p(leader, bar.s_full(0));
    if (two) {
      issue_qk_chunked<C>(tS1, sQ + C::Q_BYTES, ring, kf0, leader);
      tc_commit_p(leader, bar.s_full(1));
    }
    release_chunks<C>(bar, kf0, C::QCH, leader);
    if (it.nb == 1) {
      tc_commit_p(leader, bar.q_empty(0));
      if (two) tc_commit_p(leader, bar.q_empty(1));
    }
    for (int32_t g = 0; g < it.nb && ok; ++g) {
      const bool more = g + 1 < it.nb;
      // the stream: V(g), then K(g+1)
      const uint32_t vf = n, vs = vf % C::NCH;
      n += C::VCH;
      const uint32_t kf = n, ks = kf % C::NCH;
      if (more) n += C::QCH;
      // ---- tile 0: P_0(g) and V(g); then K(g+1), which is waited for
      // separately: its chunks reuse the slots of the previous block's V
      // (released last), so it tends to land after V(g)
      if (!(ok = wait_ready(bar.p_full(0), p0 & 1u, true, bar.ch_full(vs), (fwait >> vs) & 1u, false, 0u, 0u,
                            abort, tmo)))
        break;
      fwait ^= 1u << vs;
      ++p0;
      tc_fence_after();
      issue_pv_chunked<C, BK>(tO0, tS0, ring, vf, g == 0, leader);
      if (!more) tc_commit_p(leader, bar.o_done(0));
      if (!two) release_chunks<C>(bar, vf, C::VCH, leader);
      if (more) {
        if (!(ok = mbar_wait(bar.ch_full(ks), (fwait >> ks) & 1u, abort, tmo))) break;
        fwait ^= 1u << ks;
        tc_fence_after();
        issue_qk_chunked<C>(tS0, sQ, ring, kf, leader);
        tc_commit_p(leader, bar.s_full(0));
        if (!two) release_chunks<C>(bar, kf, C::QCH, leader);
        if (g + 2 == it.nb) tc_commit_p(leader, bar.q_empty(0));
      }
      if (!two) continue;
      // ---- tile 1: P_1(g); V(g) and K(g+1) are resident
      if (!(ok = mbar_wait(bar.p_full(1), p1 & 1u, abort, tmo))) break;
      ++p1;
      tc_fence_after();
      issue_pv_chunked<C, BK>(tO1, tS1, ring, vf, g == 0, leader);
      if (!more) tc_commit_p(leader, bar.o_done(1));
      release_chunks<C>(bar, vf, C::VCH, leader);
      if (more) {
        issue_qk_chunked<C>(tS1, sQ + C::Q_BYTES, ring, kf, leader);
        tc_commit_p(leader, bar.s_full(1));
        release_chunks<C>(bar, kf, C::QCH, leader);
        if (g + 2 == it.nb) tc_commit_p(leader, bar.q_empty(1));
      }
    }
  }
  if (!ok && leader) raise_error(p, abort, SPLASH_DEV_TIMEOUT_MMA);
  // drain: every MMA issued by this warp has completed
  tc_commit_p(leader, bar.drain());
  if (!mbar_wait_drain(bar.drain(), 0, tmo) && leader) atomicOr(p.err, SPLASH_DEV_TIMEOUT_DRAIN);
}

// A full soft-capped block's exponentials in one pass when the series holds
// and the row's reference m is known: 2^(cap*log2(e)*tanh(s*scale/cap) - m)
// with the series written as an odd polynomial in s (three packed FMA-pipe
// operations per pair, the last one also subtracting m).  Returns the row
// sum like exp2_block.
template <int N>
__device__ __forceinline__ float exp2_capped_series(float (&s)[N], const FwdParams &p, float m) {
  const f32x2 c2{p.cap_c2, p.cap_c2}, c1{p.cap_c1, p.cap_c1}, ck{p.scale_log2, p.scale_log2}, nm{-m, -m};
  f32x2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const f32x2 x{s[j], s[j + 1]};
    const f32x2 u = fmul2(x, x);
    f32x2 q = ffma2(u, c2, c1);
    q = ffma2(u, q, ck);
    const f32x2 a = ffma2(x, q, nm);
    s[j] = ex2_approx(a.x);
    s[j + 1] = ex2_approx(a.y);
    acc[(j >> 1) & 3] = fadd2(acc[(j >> 1) & 3], f32x2{s[j], s[j + 1]});
  }
  const f32x2 t = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
  return t.x + t.y;
}

// tanh(s*k) for two scores by the series (|s*k| <= 0.25), packed fp32x2:
// a = s*k, then a + a*u*(c1 + c2*u) with u = a*a.
__device__ __forceinline__ f32x2 tanh_series2(f32x2 s, f32x2 k) {
  const f32x2 a = fmul2(s, k);
  const f32x2 u = fmul2(a, a);
  const f32x2 p1 = ffma2(u, f32x2{kTanhC2, kTanhC2}, f32x2{kTanhC1, kTanhC1});
  return ffma2(fmul2(a, u), p1, a);
}

// Element mask of a partial block for query position qpos (row `row` of the
// tile; active block g_idx, pattern mn): read from the stored bit-packed
// pattern, or computed from positions when the table allows it (the band part
// of the mask: causal and window bounds, and the padding of ragged lengths --
// "Pallas Kernels and Splash Attention" §6.6: masks can be computed in the
// kernel from q / kv positions instead of stored patterns).
// Where a partial block's element mask comes from: the stored pattern, or
// positions (the band part), or positions and segment IDs.
constexpr int kPatStored = 0, kPatBand = 1, kPatBandSeg = 2;

template <int BK, int PM>
__device__ __forceinline__ void partial_bits(const FwdParams &p, int32_t mn, int row, int64_t qpos, int32_t g_idx,
                                             uint32_t (&bits)[BK / 32]) {
  if constexpr (PM != kPatStored) {
    const int64_t c0 = (int64_t)__ldg(p.active_cols + g_idx) * BK;
    int64_t lo = c0, hi = min(c0 + BK - 1, p.Lk - 1);
    if (p.band_causal) hi = min(hi, qpos);
    if (p.band_wl >= 0) lo = max(lo, qpos - p.band_wl);
    if (p.band_wr >= 0) hi = min(hi, qpos + p.band_wr);
    if (qpos >= p.Lq) hi = lo - 1;
#pragma unroll
    for (int x = 0; x < BK / 32; ++x) {
      const int64_t w0 = c0 + 32 * x, a = max(lo, w0), b = min(hi, w0 + 31);
      const int32_t n = (int32_t)(b - a + 1);
      bits[x] = n <= 0 ? 0u : ((n >= 32 ? 0xffffffffu : ((1u << n) - 1u)) << (int32_t)(a - w0));
    }
  } else {
    const uint32_t *src = p.pattern_bits + ((int64_t)mn * p.bq + row) * (BK / 32);
#pragma unroll
    for (int x = 0; x < BK / 32; ++x) bits[x] = __ldg(src + x);
  }
}

// Segment part of a partial block's mask ("Pallas Kernels and Splash
// Attention" §6.4, §6.6): key j is allowed for the query only if their
// segment IDs are equal.  Lane l holds kid[x], the ID of key 32x + l of the
// block, so a warp ballot on "ID == the query's ID" is word x of the row's
// mask for every lane that has that query ID.  The usual case, all 32 rows of
// the warp in one segment, takes one ballot per word; a warp whose rows span
// several segments takes one more pass per further query ID.  Warp-collective:
// every lane of the warp calls it with the same control flow.
// The key IDs of active block g_idx (kid) and the query's own ID (returned)
// for batch row b; rows past Lq and keys past Lk read nothing (the band part
// masks them).
template <int BK>
__device__ __forceinline__ int32_t seg_kids(const FwdParams &p, int32_t b, int32_t qpos, int32_t g_idx, int lane,
                                            int32_t (&kid)[BK / 32]) {
  const int64_t sr = p.nbm > 1 ? b : 0;  // segment-array row
  const int64_t c0 = (int64_t)__ldg(p.active_cols + g_idx) * BK;
#pragma unroll
  for (int x = 0; x < BK / 32; ++x) {
    const int64_t kp = c0 + 32 * x + lane;
    kid[x] = kp < p.Lk ? __ldg(p.seg_kv + sr * p.Lk + kp) : 0;
  }
  return qpos < p.Lq ? __ldg(p.seg_q + sr * p.Lq + qpos) : 0;
}

template <int BK>
__device__ __forceinline__ void seg_and(uint32_t (&bits)[BK / 32], const int32_t (&kid)[BK / 32], int32_t qseg) {
  const int32_t q0 = __shfl_sync(0xffffffffu, qseg, 0);
  if (__all_sync(0xffffffffu, qseg == q0)) {
#pragma unroll
    for (int x = 0; x < BK / 32; ++x) bits[x] &= __ballot_sync(0xffffffffu, kid[x] == q0);
    return;
  }
  // rows of several segments (a warp at a segment boundary): one ballot per
  // word for each distinct query ID, lane 0's first
  uint32_t w[BK / 32];
#pragma unroll
  for (int x = 0; x < BK / 32; ++x) w[x] = __ballot_sync(0xffffffffu, kid[x] == q0);
  uint32_t done = __ballot_sync(0xffffffffu, qseg == q0);
  while (done != 0xffffffffu) {  // warp-uniform
    const int32_t qv = __shfl_sync(0xffffffffu, qseg, __ffs(~done) - 1);
#pragma unroll
    for (int x = 0; x < BK / 32; ++x) {
      const uint32_t b = __ballot_sync(0xffffffffu, kid[x] == qv);
      w[x] = qseg == qv ? b : w[x];
    }
    done |= __ballot_sync(0xffffffffu, qseg == qv);
  }
#pragma unroll
  for (int x = 0; x < BK / 32; ++x) bits[x] &= w[x];
}

// s_j <- 2^(s_j * mul - sub) in place (packed argument), returns the row sum
// (eight independent partial sums).
template <int N>
__device__ __forceinline__ float exp2_block(float (&s)[N], float mul, float sub) {
  const f32x2 m2{mul, mul}, n2{-sub, -sub};
  f32x2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const f32x2 a = ffma2(f32x2{s[j], s[j + 1]}, m2, n2);
    s[j] = ex2_approx(a.x);
    s[j + 1] = ex2_approx(a.y);
    acc[(j >> 1) & 3] = fadd2(acc[(j >> 1) & 3], f32x2{s[j], s[j + 1]});
  }
  const f32x2 t = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
  return t.x + t.y;
}

// PM: partial blocks' masks from the stored patterns, or computed from
// positions (and segment IDs) -- separate instantiations, so that the default
// stored-pattern loop is unchanged.
// CAP: the tanh soft cap, a compile-time flag so that the kernels without
// it carry none of its code (the fused cap + exponent loop changes their
// register allocation).
template <int DQK, int DV, int BK, int PM, bool TALL, bool CAP>
__global__ void __launch_bounds__(kThreads, 1)
splash_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p) {
  using C = Cfg<DQK, DV, BK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + 2 * C::Q_BYTES;
  const uint32_t sV = sK + C::NK * C::K_BYTES;
  const uint32_t sStage = sV + C::NV * C::V_BYTES;  // C::STAGE_BYTES of O staging
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::TILES + C::STAGE_BYTES);
  const Bars<C> bar{smem_u32(bars)};
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::TILES + C::STAGE_BYTES + C::NBAR * 8);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + C::TILES + C::STAGE_BYTES + C::NBAR * 8 + 4);
  Item *items = reinterpret_cast<Item *>(smem + C::TILES + C::STAGE_BYTES + C::NBAR * 8 + 16);  // the item ring

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar.q_full(t), 1);
      mbar_init(bar.q_empty(t), 1);
      mbar_init(bar.s_full(t), 1);
      mbar_init(bar.p_full(t), 4);  // the four warps of the tile's softmax
      mbar_init(bar.o_done(t), 1);
    }
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(bar.k_full(s), 1);
      mbar_init(bar.k_empty(s), p.dual_issuer ? 2 : 1);  // one release per MMA issuer
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(bar.v_full(s), 1);
      mbar_init(bar.v_empty(s), p.dual_issuer ? 2 : 1);
    }
    mbar_init(bar.drain(), p.dual_issuer ? 2 : 1);
    for (int s = 0; s < C::NCH; ++s) {
      mbar_init(bar.ch_full(s), 1);   // the producer's arm of the tile whose first chunk is here
      mbar_init(bar.ch_empty(s), 1);  // the (single) issuer's release of the chunk
    }
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(bar.item_full(s), 1);  // the decoder
      // released by the producer, the MMA issuer(s) and the eight softmax warps
      mbar_init(bar.item_empty(s), 1 + (p.dual_issuer ? 2 : 1) + 8);
    }
    *abort = 0;
    mbar_fence_init();
  }
  if (threadIdx.x == kProducerWarp * 32) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if (C::STAGE) tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp >= 8) {
  // ============================================================ warpgroup 2
  regs_decrease<kControlRegs>();
  if (warp == kProducerWarp) {
    if constexpr (TALL && C::NCH > 0) {
      if (lane == 0) run_producer_chunked<C, BK>(p, &tmQ, &tmK, &tmV, sQ, sK, bar, abort);
    } else {
      if (lane == 0) run_producer<C, BK, TALL>(p, &tmQ, &tmK, &tmV, sQ, sK, sV, bar, abort);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    if constexpr (TALL && C::NCH > 0) {
      if (warp == kMmaWarp) run_mma_pair_chunked<C, BK>(p, tmem, sQ, sK, bar, abort, elect_one_sync());
    } else if (p.dual_issuer) {
      if (lane == 0) run_mma<C, BK, TALL>(p, tmem, sQ, sK, sV, bar, abort, warp - kMmaWarp);
    } else if (warp == kMmaWarp) {
      run_mma_pair<C, BK, TALL>(p, tmem, sQ, sK, sV, bar, abort, elect_one_sync());
    }
  } else if (warp == kDecoderWarp) {
    if (lane == 0) run_decoder<C, TALL>(p, bar, items, abort);
  }
  } else {
  // ============================================================ warpgroups 0, 1
  regs_increase<kSoftmaxRegs>();
  {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;          // query tile
    const int wq = warp & 3;          // TMEM lane quarter
    const int row = wq * 32 + lane;   // query row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + 128u * t + lane_off;
    const uint32_t tO = tmem + 256u + 128u * t + lane_off;
    const int prow = (TALL && t) ? 128 + row : row;  // row within the q-block (pattern row)
    const bool row_valid = prow < p.bq;
    uint32_t scnt = 0, ocnt = 0;
    bool ok = true;
    for (int64_t k = 0; ok; ++k) {
      // the fields this warp needs, read from the ring slot, which is then released
      const uint32_t ia = hold_item_warp(bar, k, ok, abort, p.timeout_ns);
      if (ia == 0u) break;
      const bool it_act1 = (item_i32(ia, offsetof(Item, act1) & ~(size_t)3) >> (8 * (offsetof(Item, act1) & 3))) & 0xff;
      const int32_t it_g0 = item_i32(ia, offsetof(Item, g0)), it_nb = item_i32(ia, offsetof(Item, nb));
      const int32_t it_qrow = item_i32(ia, offsetof(Item, qrow)), it_b = item_i32(ia, offsetof(Item, b));
      const int32_t it_h = item_i32(ia, t ? offsetof(Item, h1) : offsetof(Item, h0));
      const int32_t it_split = item_i32(ia, offsetof(Item, split));
      release_item_warp(bar, k);
      if (t == 1 && !it_act1) continue;
      const int32_t qpos = it_qrow * p.bq + prow;  // < 2^31: nq * bq <= 65535 * 256
      float m_ref = p.use_mle ? p.mle_ref : -INFINITY;  // running reference (log2 units)
      float l = 0.f;
      for (int32_t g = 0; g < it_nb && ok; ++g) {
        int32_t mn = p.mask_next[it_g0 + g];
        if (mn >= p.num_patterns) {
          atomicOr(p.err, SPLASH_DEV_BAD_TABLE);
          mn = -1;
        }
        const bool partial = mn >= 0;
        const bool need_mask = partial || !row_valid;
        uint32_t bits[BK / 32];
        if (partial && row_valid) {
          partial_bits<BK, PM>(p, mn, prow, qpos, it_g0 + g, bits);
        } else {
#pragma unroll
          for (int x = 0; x < BK / 32; ++x) bits[x] = row_valid ? 0xffffffffu : 0u;
        }
        // the segment part, before the wait for S (whose latency hides the
        // key IDs' loads); partial is the same for every lane of the warp
        if constexpr (PM == kPatBandSeg) {
          if (partial) {
            int32_t kid[BK / 32];
            const int32_t qseg = seg_kids<BK>(p, it_b, qpos, it_g0 + g, lane, kid);
            seg_and<BK>(bits, kid, qseg);
          }
        }
        // all lanes wait; the outcome is made warp-uniform before the
        // warp-collective TMEM accesses
        ok = __all_sync(0xffffffffu, mbar_wait(bar.s_full(t), scnt & 1, abort, p.timeout_ns));
        if (!ok) break;
        ++scnt;
        tc_fence_after();
        float s[BK];
        {
          uint32_t r[BK / 32][32];
#pragma unroll
          for (int c = 0; c < BK / 32; ++c) tmem_ld32(tS + 32u * c, r[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < BK / 32; ++c) {
            reg_fence32(r[c]);
#pragma unroll
            for (int x = 0; x < 32; ++x) s[c * 32 + x] = __uint_as_float(r[c][x]);
          }
        }
        // Scores in log2 units are s*mul: mul = scale*log2e, or with the soft
        // cap s <- tanh(s*scale/cap) here and mul = cap*log2e (the exponent's
        // FFMA applies it).  Masked entries become -inf.
        const float mul = CAP ? p.cap_log2 : p.scale_log2;
        float alpha = 1.f;
        float sum = 0.f;
        bool fused = false;  // exponentials already taken by exp2_capped_series
        if constexpr (CAP) {
          float am[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) am[x] = fmaxf(fabsf(s[2 * x]), fabsf(s[2 * x + 1]));
#pragma unroll
          for (int j = 8; j < BK; j += 2) am[(j >> 1) & 3] = fmax3(am[(j >> 1) & 3], fabsf(s[j]), fabsf(s[j + 1]));
          const float amax = fmax3(am[0], am[1], fmaxf(am[2], am[3])) * p.cap_inner;
          if (__any_sync(0xffffffffu, amax > kTanhSeriesLimit)) {
#pragma unroll
            for (int j = 0; j < BK; ++j) s[j] = tanh_identity(s[j] * p.cap_inner);
          } else if (!need_mask && !__any_sync(0xffffffffu, m_ref == -INFINITY)) {
            // the steady state of a full block: the cap and the exponent in one pass
            sum = exp2_capped_series<BK>(s, p, m_ref);
            fused = true;
          } else {
            const f32x2 k2{p.cap_inner, p.cap_inner};
#pragma unroll
            for (int j = 0; j < BK; j += 2) {
              const f32x2 r2 = tanh_series2(f32x2{s[j], s[j + 1]}, k2);
              s[j] = r2.x;
              s[j + 1] = r2.y;
            }
          }
        }
        if (!fused) {
          if (need_mask) {
#pragma unroll
            for (int j = 0; j < BK; ++j) s[j] = ((bits[j >> 5] >> (j & 31)) & 1u) ? s[j] : -INFINITY;
          }
          // Exponentials against the row's running reference m_ref, which
          // moves only (i) to the first allowed keys' maximum and (ii) when a
          // block's sum of exponentials would reach 2^64 (then the block is
          // recomputed against its own maximum): between those events the max
          // is not needed at all.  P, l and O stay far from overflow (P < 2^64),
          // and O / l is independent of the reference.
          if (__any_sync(0xffffffffu, m_ref == -INFINITY)) {
            // a row's first block with allowed keys: its reference is their max
            const float mx = max_tree<BK>(s) * mul;  // scale > 0
            if (m_ref == -INFINITY && mx != -INFINITY) {
              alpha = 0.f;
              m_ref = mx;
            }
          }
          sum = exp2_block<BK>(s, mul, m_ref == -INFINITY ? 0.f : m_ref);
        }
        const bool redo = !(sum < kPMax);
        if (__any_sync(0xffffffffu, redo)) {
          // rare: exponentials above 2^64 for some lane.  The warp reloads S
          // (warp-collective; P has not been written yet); those lanes move
          // their reference to the block's maximum, and every lane
          // recomputes its row (for the others this gives the values they
          // already have, up to rounding); nothing from the main path stays
          // live across this branch but the references.  (With segment IDs
          // the row's mask words are formed again first, before S occupies
          // the registers.)
          [[maybe_unused]] uint32_t rs[PM == kPatBandSeg ? BK / 32 : 1];
          if constexpr (PM == kPatBandSeg) {
            if (partial && row_valid) {
              partial_bits<BK, PM>(p, mn, prow, qpos, it_g0 + g, rs);
            } else {
#pragma unroll
              for (int x = 0; x < BK / 32; ++x) rs[x] = row_valid ? 0xffffffffu : 0u;
            }
            if (partial) {
              int32_t kr[BK / 32];
              const int32_t qseg = seg_kids<BK>(p, it_b, qpos, it_g0 + g, lane, kr);
              seg_and<BK>(rs, kr, qseg);
            }
          }
          {
            uint32_t r[BK / 32][32];
#pragma unroll
            for (int c = 0; c < BK / 32; ++c) tmem_ld32(tS + 32u * c, r[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < BK / 32; ++c) {
              reg_fence32(r[c]);
#pragma unroll
              for (int x = 0; x < 32; ++x) s[c * 32 + x] = __uint_as_float(r[c][x]);
            }
          }
          if constexpr (CAP) {
#pragma unroll
            for (int j = 0; j < BK; ++j) s[j] = tanh_identity(s[j] * p.cap_inner);
          }
          if (need_mask) {
            if constexpr (PM == kPatBandSeg) {
#pragma unroll
              for (int x = 0; x < BK / 32; ++x) {
#pragma unroll
                for (int j = 0; j < 32; ++j) s[x * 32 + j] = ((rs[x] >> j) & 1u) ? s[x * 32 + j] : -INFINITY;
              }
            } else if constexpr (PM == kPatBand) {
              uint32_t rb[BK / 32];
              if (partial && row_valid) {
                partial_bits<BK, PM>(p, mn, prow, qpos, it_g0 + g, rb);
              } else {
#pragma unroll
                for (int x = 0; x < BK / 32; ++x) rb[x] = row_valid ? 0xffffffffu : 0u;
              }
#pragma unroll
              for (int x = 0; x < BK / 32; ++x) {
#pragma unroll
                for (int j = 0; j < 32; ++j) s[x * 32 + j] = ((rb[x] >> j) & 1u) ? s[x * 32 + j] : -INFINITY;
              }
            } else {
              const uint32_t *src = p.pattern_bits + ((int64_t)mn * p.bq + prow) * (BK / 32);
#pragma unroll
              for (int x = 0; x < BK / 32; ++x) {
                const uint32_t b = (partial && row_valid) ? __ldg(src + x) : (row_valid ? 0xffffffffu : 0u);
#pragma unroll
                for (int j = 0; j < 32; ++j) s[x * 32 + j] = ((b >> j) & 1u) ? s[x * 32 + j] : -INFINITY;
              }
            }
          }
          if (redo) {
            const float mx = max_tree<BK>(s) * mul;
            alpha *= ex2_approx(m_ref - mx);
            m_ref = mx;
          }
          sum = exp2_block<BK>(s, mul, m_ref == -INFINITY ? 0.f : m_ref);
        }
        // P (bf16 pairs) into the first BK/2 columns of S_t, 32 columns per store
#pragma unroll
        for (int c = 0; c < BK / 64; ++c) {
          uint32_t r[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) r[x] = pack_bf16x2(s[c * 64 + 2 * x], s[c * 64 + 2 * x + 1]);
          tmem_st32(tS + 32u * c, r);
        }
        l = l * alpha + sum;
        // rescale the output accumulator (its previous PV has completed:
        // S_t(g) was committed after it)
        if (g > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            tmem_ld32(tO + 32u * c, r);
            tmem_wait_ld();
            reg_fence32(r);
#pragma unroll
            for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
            tmem_st32(tO + 32u * c, r);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.p_full(t));  // one arrival per warp
      }
      if (!ok) break;
      // ---- epilogue: O / l and the LSE
      const int32_t h = it_h;
      const int64_t orow = ((int64_t)it_b * p.Hq + h) * p.Lq + qpos;
      // rows past a ragged Lq are padding: computed (all masked), never stored
      const bool row_out = row_valid && qpos < p.Lq;
      if (it_nb > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar.o_done(t), ocnt & 1, abort, p.timeout_ns));
        if (!ok) break;
        ++ocnt;
        tc_fence_after();
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (p.o_part != nullptr) {
        // split-KV partial: the split's normalized O in fp32 (32-byte stores)
        float *dst = p.o_part + ((int64_t)it_split * p.part_rows + orow) * DV;
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t r[32];
          if (it_nb > 0) {
            tmem_ld32(tO + 32u * c, r);
            tmem_wait_ld();
            reg_fence32(r);
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) r[x] = 0u;
          }
          if (row_out) {
#pragma unroll
            for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * inv);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              st_global_v8(dst + c * 32 + 8 * x, r[8 * x], r[8 * x + 1], r[8 * x + 2], r[8 * x + 3], r[8 * x + 4],
                           r[8 * x + 5], r[8 * x + 6], r[8 * x + 7]);
          }
        }
      } else if (C::STAGE) {
        // O rows to the warp's 128B-swizzled staging box (32 rows x 64
        // columns), one TMA store per box: whole-line global writes instead
        // of 32 rows' scattered pieces per store instruction
        const uint32_t stage = sStage + (uint32_t)warp * C::STAGE_WARP;
        const int wrow = ((TALL && t) ? 128 : 0) + wq * 32;  // the warp's first row within the q-block
        const bool warp_rows = wrow < p.bq;             // rows beyond bq belong to no output
#pragma unroll
        for (int hh = 0; hh < DV / 64; ++hh) {
          uint32_t r0[32], r1[32];
          if (it_nb > 0) {
            tmem_ld32(tO + 64u * hh, r0);
            tmem_ld32(tO + 64u * hh + 32u, r1);
            tmem_wait_ld();
            reg_fence32(r0);
            reg_fence32(r1);
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) r0[x] = r1[x] = 0u;
          }
          uint32_t o[32];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const f32x2 y0 = fmul2(f32x2{__uint_as_float(r0[2 * x]), __uint_as_float(r0[2 * x + 1])}, f32x2{inv, inv});
            const f32x2 y1 = fmul2(f32x2{__uint_as_float(r1[2 * x]), __uint_as_float(r1[2 * x + 1])}, f32x2{inv, inv});
            o[x] = pack_bf16x2(y0.x, y0.y);
            o[16 + x] = pack_bf16x2(y1.x, y1.y);
          }
          if (warp_rows) {
            if (lane == 0) bulk_wait_read_all();  // the previous box has been read
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              st_shared_v4(stage + (uint32_t)lane * 128u + (uint32_t)((j ^ (lane & 7)) * 16), o[4 * j], o[4 * j + 1],
                           o[4 * j + 2], o[4 * j + 3]);
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
              // O viewed as [B*Hq][Lq][DV]: rows past a ragged Lq fall outside
              // the tensor and the store clips them
              tma_store_3d(&tmO, stage, 64 * hh, it_qrow * p.bq + wrow, it_b * p.Hq + h);
              bulk_commit_group();
            }
          }
        }
      } else {
      __nv_bfloat16 *orow_ptr = p.out + orow * DV;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t r[32];
        if (it_nb > 0) {
          tmem_ld32(tO + 32u * c, r);
          tmem_wait_ld();
          reg_fence32(r);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) r[x] = 0u;
        }
        if (row_out) {
          uint32_t o[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const f32x2 y = fmul2(f32x2{__uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1])}, f32x2{inv, inv});
            o[x] = pack_bf16x2(y.x, y.y);
          }
          // two 32-byte stores (whole sectors) per 32 columns
          st_global_v8(orow_ptr + c * 32, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
          st_global_v8(orow_ptr + c * 32 + 16, o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15]);
        }
      }
      }
      if (row_out) {
        const float lse_v = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        if (p.o_part != nullptr)
          p.lse_part[(int64_t)it_split * p.part_rows + orow] = lse_v;
        else
          p.lse[orow] = lse_v;
      }
    }
    if (!ok) raise_error(p, abort, SPLASH_DEV_TIMEOUT_SOFTMAX);
    if (C::STAGE && lane == 0) bulk_wait_all();  // this warp's O stores have completed
  }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------- self test
__global__ void wait_selftest_kernel(uint64_t timeout_ns, uint32_t *err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on `bar`: the bounded wait must give up
    if (!mbar_wait(smem_u32(&bar), 0, &abort_flag, timeout_ns)) atomicOr(err, SPLASH_DEV_TIMEOUT_SELFTEST);
  }
}

// --------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool make_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [planes][rows][cols] bf16 with 64-column x box_rows x 1 boxes (128B swizzle)
bool make_map_3d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t planes,
                 uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cols, rows, planes};
  const cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DQK, int DV, int BK, int PM, bool TALL, bool CAP>
splash_status launch(const void *q, const void *k, const void *v, const FwdParams &prm, cudaStream_t stream) {
  using C = Cfg<DQK, DV, BK>;
  CUtensorMap tq, tk, tv, to;
  if (!make_map(&tq, q, DQK, (uint64_t)prm.B * prm.Hq * prm.Lq, 128) ||
      !make_map(&tk, k, DQK, (uint64_t)prm.B * prm.Hkv * prm.Lk, BK) ||
      !make_map(&tv, v, DV, (uint64_t)prm.B * prm.Hkv * prm.Lk, BK) ||
      (C::STAGE && prm.o_part == nullptr &&
       !make_map_3d(&to, prm.out, DV, (uint64_t)prm.Lq, (uint64_t)prm.B * prm.Hq, 32)))
    return SPLASH_ERR_CUDA;
  if (!C::STAGE || prm.o_part != nullptr) to = tq;  // unused (no staging, or split partials)
  static int configured_device = -1;
  int dev = 0;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  int sms = 148;
  SPLASH_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (configured_device != dev) {
    SPLASH_CUDA_TRY(cudaFuncSetAttribute(splash_fwd_kernel<DQK, DV, BK, PM, TALL, CAP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
    configured_device = dev;
  }
  const int64_t grid = prm.num_items < sms ? prm.num_items : sms;
  if (grid <= 0) return SPLASH_OK;
  FwdParams run = prm;
  const int64_t items_per_head = (int64_t)prm.nbm * prm.nq * (prm.nbm == 1 ? prm.B : 1) * prm.nsplit;
  run.head_group = splash_choose_head_group(prm.dense_rows != 0, items_per_head, prm.npairs,
                                            (int64_t)prm.B * prm.Hkv * prm.Lk * (DQK + DV) * 2, grid);
  splash_fwd_kernel<DQK, DV, BK, PM, TALL, CAP><<<(unsigned)grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, to, run);
  SPLASH_CUDA_TRY(cudaGetLastError());
  splash_count_launches(1);
  return SPLASH_OK;
}

template <int PM, bool CAP>
splash_status launch_shape(const void *q, const void *k, const void *v, const FwdParams &prm, int32_t dqk,
                           int32_t dv, int32_t bk, cudaStream_t stream) {
  if (prm.t1_off) {  // 256-row q-blocks: two halves of one head per item (bk = 128)
    if (dqk == 128 && dv == 128 && bk == 128) return launch<128, 128, 128, PM, true, CAP>(q, k, v, prm, stream);
    if (dqk == 192 && dv == 128 && bk == 128) return launch<192, 128, 128, PM, true, CAP>(q, k, v, prm, stream);
    if (dqk == 64 && dv == 64 && bk == 128) return launch<64, 64, 128, PM, true, CAP>(q, k, v, prm, stream);
    return SPLASH_ERR_UNSUPPORTED;
  }
  if (dqk == 128 && dv == 128 && bk == 128) return launch<128, 128, 128, PM, false, CAP>(q, k, v, prm, stream);
  if (dqk == 192 && dv == 128 && bk == 128) return launch<192, 128, 128, PM, false, CAP>(q, k, v, prm, stream);
  if (dqk == 64 && dv == 64 && bk == 64) return launch<64, 64, 64, PM, false, CAP>(q, k, v, prm, stream);
  if (dqk == 64 && dv == 64 && bk == 128) return launch<64, 64, 128, PM, false, CAP>(q, k, v, prm, stream);
  if (dqk == 128 && dv == 128 && bk == 64) return launch<128, 128, 64, PM, false, CAP>(q, k, v, prm, stream);
  return SPLASH_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace splash

using namespace splash;

namespace {

// The pattern source of a MaskInfo: stored, or from positions (with segment
// IDs when the table has them).
int pattern_mode(const splash_mask_info *mi) {
  return !mi->patterns_from_positions ? kPatStored : (mi->has_segments ? kPatBandSeg : kPatBand);
}

// The kernel parameters of a forward call (SPLASH_OK) or the argument error.
splash_status make_fwd_params(int32_t B, int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk,
                              const int32_t *q_segment_ids, const int32_t *kv_segment_ids,
                              const splash_mask_info *mi, float scale, float softcap, float max_logit, void *out,
                              float *lse, int32_t nsplit, float *o_part, float *lse_part, uint32_t *err_word,
                              FwdParams &prm) {
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = Hq / Hkv;
  prm.Lq = Lq;
  prm.Lk = Lk;
  prm.bq = mi->bq;
  prm.nq = (int32_t)mi->nq;
  prm.nk = (int32_t)mi->nk;
  prm.nbm = mi->batch_rows;
  prm.t1_off = mi->bq == 256 ? 128 : 0;
  prm.npairs = prm.t1_off ? Hq : (Hq + 1) / 2;
  prm.head_group = prm.npairs;  // chosen per launch (splash_choose_head_group)
  prm.dense_rows = (!mi->has_segments && mi->window_left < 0 && mi->window_right < 0) ? 1 : 0;
  const int64_t rows = (int64_t)mi->batch_rows * mi->nq;
  prm.nsplit = nsplit > 1 ? nsplit : 1;
  prm.num_items = (mi->batch_rows == 1 ? rows * B : rows) * prm.npairs * prm.nsplit;
  prm.o_part = o_part;
  prm.lse_part = lse_part;
  prm.part_rows = (int64_t)B * Hq * Lq;
  prm.row_ptr = mi->row_ptr;
  prm.active_cols = mi->active_cols;
  prm.mask_next = mi->mask_next;
  prm.pattern_bits = mi->pattern_bits;
  // pattern source: stored, or from positions (with segment IDs when the
  // table has them; the caller passes the arrays it was built from)
  const int pm = pattern_mode(mi);
  if (pm == kPatBandSeg && q_segment_ids == nullptr) return SPLASH_ERR_INVALID_ARG;
  prm.band_bits = pm != kPatStored ? 1 : 0;
  prm.seg_q = q_segment_ids;
  prm.seg_kv = kv_segment_ids != nullptr ? kv_segment_ids : q_segment_ids;
  prm.band_causal = mi->causal;
  prm.band_wl = mi->window_left;
  prm.band_wr = mi->window_right;
  prm.row_order = mi->row_order;
  // bound for the kernel's check of mask_next (the true count may still be in
  // flight after an asynchronous build; it never exceeds the buffer capacity)
  prm.num_patterns = mi->counts_pending ? mi->cap_patterns : mi->num_patterns;
  prm.scale_log2 = scale * kLog2e;
  prm.use_softcap = softcap > 0.f ? 1 : 0;
  prm.use_mle = std::isnan(max_logit) ? 0 : 1;  // NaN: off
  prm.mle_ref = prm.use_mle ? max_logit * kLog2e : 0.f;
  // one issuer per tile only when the two query heads of an item read
  // different KV heads (MHA with two heads per item); shared K/V (GQA heads,
  // or the two halves of a 256-row q-block) keeps one issuer for both tiles
  prm.dual_issuer = (prm.G == 1 && !prm.t1_off) ? 1 : 0;
  prm.cap_inner = softcap > 0.f ? scale / softcap : 0.f;
  prm.cap_log2 = softcap > 0.f ? softcap * kLog2e : 0.f;
  {
    const double sc = scale, cp = softcap > 0.f ? softcap : 1.0, l2e = 1.4426950408889634;
    prm.cap_c1 = softcap > 0.f ? (float)(kTanhC1 * sc * sc * sc * l2e / (cp * cp)) : 0.f;
    prm.cap_c2 = softcap > 0.f ? (float)(kTanhC2 * sc * sc * sc * sc * sc * l2e / (cp * cp * cp * cp)) : 0.f;
  }
  prm.out = reinterpret_cast<__nv_bfloat16 *>(out);
  prm.lse = lse;
  prm.err = err_word;
  prm.timeout_ns = 1000000000ull;  // 1 s per wait
  return SPLASH_OK;
}

}  // namespace

// The launcher of one pattern mode (its kernels only are compiled here).
#define SPLASH_FWD_MODE_LAUNCHER(PM, NAME)                                                                        \
  splash_status NAME(const void *q, const void *k, const void *v, int32_t B, int32_t Hq, int32_t Hkv, int64_t Lq, \
                     int64_t Lk, int32_t dqk, int32_t dv, const int32_t *q_segment_ids,                          \
                     const int32_t *kv_segment_ids, const splash_mask_info *mi, float scale, float softcap,     \
                     float max_logit, void *out, float *lse, int32_t nsplit, float *o_part, float *lse_part,    \
                     cudaStream_t stream, uint32_t *err_word) {                                                  \
    FwdParams prm;                                                                                               \
    const splash_status st = make_fwd_params(B, Hq, Hkv, Lq, Lk, q_segment_ids, kv_segment_ids, mi, scale,       \
                                             softcap, max_logit, out, lse, nsplit, o_part, lse_part, err_word,   \
                                             prm);                                                               \
    if (st != SPLASH_OK) return st;                                                                              \
    if (prm.use_softcap) return launch_shape<PM, true>(q, k, v, prm, dqk, dv, mi->bk, stream);                 \
    return launch_shape<PM, false>(q, k, v, prm, dqk, dv, mi->bk, stream);                                      \
  }

#if !defined(SPLASH_FWD_PM) || SPLASH_FWD_PM == 0
SPLASH_FWD_MODE_LAUNCHER(kPatStored, splash_fwd_launch_stored)
#endif
#if !defined(SPLASH_FWD_PM) || SPLASH_FWD_PM == 1
SPLASH_FWD_MODE_LAUNCHER(kPatBand, splash_fwd_launch_band)
#endif
#if !defined(SPLASH_FWD_PM) || SPLASH_FWD_PM == 2
SPLASH_FWD_MODE_LAUNCHER(kPatBandSeg, splash_fwd_launch_band_seg)
#endif

#if !defined(SPLASH_FWD_PM) || SPLASH_FWD_PM == 0
splash_status splash_attention_fwd_launch(const void *q, const void *k, const void *v, int32_t B,
                                          int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk,
                                          int32_t dqk, int32_t dv, const int32_t *q_segment_ids,
                                          const int32_t *kv_segment_ids, const splash_mask_info *mi,
                                          float scale, float softcap, float max_logit, void *out,
                                          float *lse, int32_t nsplit, float *o_part, float *lse_part,
                                          cudaStream_t stream, uint32_t *err_word) {
  const int pm = pattern_mode(mi);
  auto launcher = pm == kPatBandSeg ? splash_fwd_launch_band_seg
                                    : (pm == kPatBand ? splash_fwd_launch_band : splash_fwd_launch_stored);
  return launcher(q, k, v, B, Hq, Hkv, Lq, Lk, dqk, dv, q_segment_ids, kv_segment_ids, mi, scale, softcap,
                  max_logit, out, lse, nsplit, o_part, lse_part, stream, err_word);
}

splash_status splash_wait_selftest_launch(uint64_t timeout_ns, cudaStream_t stream, uint32_t *err_word) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns, err_word);
  SPLASH_CUDA_TRY(cudaGetLastError());
  splash_count_launches(1);
  return SPLASH_OK;
}

// ------------------------------------------------------------------ merge
namespace splash {
namespace {

// LSE merge of split-KV partials ("The maths and infra behind core LLM
// operations" (joto.ai), "LSE and Online Softmax": softmax segments combine
// through their log-sum-exp): per row, lse = m + ln sum_s exp(lse_s - m) with
// m = max_s lse_s, and out = sum_s exp(lse_s - lse) o_s.  One warp per row;
// each lane holds DV / 32 consecutive columns (vector loads of the fp32
// partials, one 8- or 4-byte store of the bf16 result).
template <int DV>
__global__ void __launch_bounds__(256) splash_merge_kernel(const float *o_part, const float *lse_part, int32_t nsplit,
                                                           int64_t rows, __nv_bfloat16 *out, float *lse) {
  constexpr int PER = DV / 32;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows; row += nwarps) {
    float m = -INFINITY;
    for (int32_t sp = 0; sp < nsplit; ++sp) m = fmaxf(m, __ldg(lse_part + sp * rows + row));
    float acc[PER];
#pragma unroll
    for (int x = 0; x < PER; ++x) acc[x] = 0.f;
    float den = 0.f;
    if (m != -INFINITY) {
      for (int32_t sp = 0; sp < nsplit; ++sp) {
        const float ls = __ldg(lse_part + sp * rows + row);
        if (ls == -INFINITY) continue;
        const float wgt = __expf(ls - m);
        den += wgt;
        const float *src = o_part + (sp * rows + row) * DV + lane * PER;
        if constexpr (PER == 4) {
          const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
          acc[0] += wgt * v.x;
          acc[1] += wgt * v.y;
          acc[2] += wgt * v.z;
          acc[3] += wgt * v.w;
        } else {
          const float2 v = __ldg(reinterpret_cast<const float2 *>(src));
          acc[0] += wgt * v.x;
          acc[1] += wgt * v.y;
        }
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16 *dst = out + row * DV + lane * PER;
    if constexpr (PER == 4) {
      const uint32_t a = pack_bf16x2(acc[0] * inv, acc[1] * inv), b = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2 *>(dst) = make_uint2(a, b);
    } else {
      *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) lse[row] = den > 0.f ? m + __logf(den) : -INFINITY;
  }
}

}  // namespace
}  // namespace splash

splash_status splash_attention_merge_launch(const float *o_part, const float *lse_part, int32_t nsplit, int64_t rows,
                                            int32_t dv, void *out, float *lse, cudaStream_t stream) {
  using namespace splash;
  if (rows <= 0) return SPLASH_OK;
  int dev = 0, sms = 148;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  SPLASH_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t want = (rows + 7) / 8;  // 8 rows (warps) per CTA
  const unsigned grid = (unsigned)std::min<int64_t>(want, (int64_t)sms * 16);
  __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(out);
  if (dv == 128)
    splash_merge_kernel<128><<<grid, 256, 0, stream>>>(o_part, lse_part, nsplit, rows, o, lse);
  else if (dv == 64)
    splash_merge_kernel<64><<<grid, 256, 0, stream>>>(o_part, lse_part, nsplit, rows, o, lse);
  else
    return SPLASH_ERR_UNSUPPORTED;
  SPLASH_CUDA_TRY(cudaGetLastError());
  splash_count_launches(1);
  return SPLASH_OK;
}
#endif  // the entry point, the self test and the merge: the compilation for the stored patterns
