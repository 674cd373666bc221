// api.cu -- the extern "C" boundary of libsplash.so (declared in splash.h):
// argument validation, MaskInfo handles, the device error word.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

namespace {

// The device error word: kernels atomicOr error bits into it.  One copy per
// device (a __device__ variable); host code reaches it through
// cudaGetSymbolAddress, resolved once per device.
__device__ uint32_t g_error_word;

constexpr int kMaxDevices = 64;
uint32_t *g_error_addr[kMaxDevices];
std::mutex g_error_mu;

bool valid_block(int32_t b) { return b == 64 || b == 128; }
// query blocks may also be 256 rows tall (two 128-row tiles of one head)
bool valid_q_block(int32_t b) { return valid_block(b) || b == 256; }

splash_status check_spec(const splash_mask_spec *spec, int64_t Lq, int64_t Lk) {
  if (spec == nullptr) return SPLASH_ERR_INVALID_ARG;
  if (spec->causal != 0 && spec->causal != 1) return SPLASH_ERR_INVALID_ARG;
  if (spec->window_left < -1 || spec->window_right < -1) return SPLASH_ERR_INVALID_ARG;
  if (spec->q_segment_ids != nullptr) {
    if (spec->batch <= 0) return SPLASH_ERR_INVALID_ARG;
    if (spec->kv_segment_ids == nullptr && Lq != Lk) return SPLASH_ERR_SHAPE;
  } else if (spec->kv_segment_ids != nullptr) {
    return SPLASH_ERR_INVALID_ARG;
  }
  return SPLASH_OK;
}

splash_status check_geometry(int64_t Lq, int64_t Lk, int32_t bq, int32_t bk) {
  if (Lq <= 0 || Lk <= 0 || bq <= 0 || bk <= 0) return SPLASH_ERR_INVALID_ARG;
  if (!valid_q_block(bq) || !valid_block(bk)) return SPLASH_ERR_UNSUPPORTED;
  // ragged lengths are padded to whole blocks (the padding is masked)
  if ((Lq + bq - 1) / bq > 65535 || Lk > (int64_t)1 << 30 || Lq > (int64_t)1 << 30) return SPLASH_ERR_UNSUPPORTED;
  return SPLASH_OK;
}

}  // namespace

// Item order across heads.  The static schedule deals the items in rounds of
// `grid` (one per CTA), rows longest first, every head (pair) of a row
// together.  When rows reach across the keys (no window, no segments) and the
// K / V of all heads is larger than L2 can keep (budget 64 MB, about half of
// the 129 MB: each die has its own half), the CTAs of a round would stream it
// from DRAM for every row.  Then the items are ordered
// by groups of head_group heads whose K / V fits the budget, and among the
// group sizes from half that bound up to it, the one whose group fills whole
// rounds best (the fewest items left in a partial round; a group that ends
// mid-round leaves that round unbalanced).  Measured on the wide-head causal
// MHA workload (128 heads, K / V 335 MB): 19 heads per group (two whole
// rounds of 152) 0.468 ms, 32 heads 0.489 ms, all 128 heads 0.556 ms.
// (Windowed and document rows read short, overlapping key ranges; there the
// row-major order already keeps the K / V in L2, and grouping was measured a
// few per cent slower.)
int32_t splash_choose_head_group(bool dense_rows, int64_t items_per_head, int32_t npairs, int64_t kv_bytes, int64_t grid) {
  constexpr int64_t kBudget = 64ll << 20;
  if (!dense_rows || npairs <= 1 || kv_bytes <= kBudget) return npairs;
  const int32_t cap = std::max<int32_t>(1, (int32_t)((int64_t)npairs * kBudget / kv_bytes));
  int32_t best = cap;
  int64_t best_rem = LLONG_MAX;
  for (int32_t h = cap; h >= std::max<int32_t>(1, cap / 2); --h) {
    const int64_t rem = (items_per_head * h) % grid;
    if (rem < best_rem) {
      best_rem = rem;
      best = h;
      if (rem == 0) break;
    }
  }
  return best;
}

static std::atomic<uint64_t> g_launches{0};

void splash_count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

uint32_t *splash_device_error_word(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_error_mu);
  if (g_error_addr[device] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_error_addr[device] = static_cast<uint32_t *>(p);
  }
  return g_error_addr[device];
}

extern "C" {

const char *splash_status_string(splash_status s) {
  switch (s) {
    case SPLASH_OK: return "SPLASH_OK";
    case SPLASH_ERR_INVALID_ARG: return "SPLASH_ERR_INVALID_ARG: invalid argument";
    case SPLASH_ERR_SHAPE: return "SPLASH_ERR_SHAPE: inconsistent shapes";
    case SPLASH_ERR_UNSUPPORTED: return "SPLASH_ERR_UNSUPPORTED: shape or block size not supported by this build";
    case SPLASH_ERR_CUDA: return "SPLASH_ERR_CUDA: a CUDA call failed";
    case SPLASH_ERR_DEVICE_TIMEOUT: return "SPLASH_ERR_DEVICE_TIMEOUT: a kernel's bounded wait ran out";
    case SPLASH_ERR_OOM: return "SPLASH_ERR_OOM: device allocation failed";
    case SPLASH_ERR_DEVICE_CHECK: return "SPLASH_ERR_DEVICE_CHECK: a kernel rejected a table entry";
  }
  return "SPLASH_ERR_UNKNOWN";
}

const char *splash_version(void) { return "splash-gb300 0.1 sm_103a"; }

uint64_t splash_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t splash_schedule_head_group(int32_t dense_rows, int64_t items_per_head, int32_t npairs, int64_t kv_bytes,
                                   int64_t grid) {
  if (npairs < 1 || items_per_head < 1 || grid < 1 || kv_bytes < 0) return 0;
  return splash_choose_head_group(dense_rows != 0, items_per_head, npairs, kv_bytes, grid);
}

splash_status splash_shard_items(int32_t B, int32_t Hkv, int32_t world, int32_t rank, int64_t *begin,
                                int64_t *end) {
  if (begin == nullptr || end == nullptr) return SPLASH_ERR_INVALID_ARG;
  if (B <= 0 || Hkv <= 0 || world <= 0 || rank < 0 || rank >= world) return SPLASH_ERR_INVALID_ARG;
  // balanced contiguous ranges: rank r takes [floor(n r / G), floor(n (r+1) / G))
  const int64_t n = (int64_t)B * Hkv;
  *begin = n * rank / world;
  *end = n * (rank + 1) / world;
  return SPLASH_OK;
}

splash_status splash_mask_info_rebuild(splash_mask_info *mi, const splash_mask_spec *spec, int64_t Lq,
                                       int64_t Lk, int32_t bq, int32_t bk, void *cuda_stream) {
  if (mi == nullptr) return SPLASH_ERR_INVALID_ARG;
  splash_status st = check_spec(spec, Lq, Lk);
  if (st != SPLASH_OK) return st;
  if ((st = check_geometry(Lq, Lk, bq, bk)) != SPLASH_OK) return st;
  int dev = 0;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  if (mi->device >= 0 && mi->device != dev) return SPLASH_ERR_INVALID_ARG;
  mi->device = dev;
  st = splash_mask_info_build_into(mi, spec, Lq, Lk, bq, bk, static_cast<cudaStream_t>(cuda_stream));
  if (st != SPLASH_OK) {
    mi->num_active = mi->num_partial = mi->num_patterns = mi->allowed_pairs = 0;
    mi->nq = mi->nk = 0;
  }
  return st;
}

splash_status splash_build_mask_info(const splash_mask_spec *spec, int64_t Lq, int64_t Lk, int32_t bq,
                                     int32_t bk, void *cuda_stream, splash_mask_info **out) {
  if (out == nullptr) return SPLASH_ERR_INVALID_ARG;
  *out = nullptr;
  splash_status st = check_spec(spec, Lq, Lk);
  if (st != SPLASH_OK) return st;
  if ((st = check_geometry(Lq, Lk, bq, bk)) != SPLASH_OK) return st;
  splash_mask_info *mi = new (std::nothrow) splash_mask_info();
  if (mi == nullptr) return SPLASH_ERR_OOM;
  st = splash_mask_info_rebuild(mi, spec, Lq, Lk, bq, bk, cuda_stream);
  if (st != SPLASH_OK) {
    splash_mask_info_free_buffers(mi);
    delete mi;
    return st;
  }
  *out = mi;
  return SPLASH_OK;
}

splash_status splash_mask_info_shape(const splash_mask_info *mi, int32_t *batch_rows, int64_t *nq,
                                     int64_t *nk, int32_t *bq, int32_t *bk) {
  if (mi == nullptr) return SPLASH_ERR_INVALID_ARG;
  if (batch_rows) *batch_rows = mi->batch_rows;
  if (nq) *nq = mi->nq;
  if (nk) *nk = mi->nk;
  if (bq) *bq = mi->bq;
  if (bk) *bk = mi->bk;
  return SPLASH_OK;
}

splash_status splash_mask_info_counts(const splash_mask_info *mi, int64_t *num_active, int64_t *num_partial,
                                      int64_t *num_patterns, int64_t *allowed_pairs) {
  if (mi == nullptr) return SPLASH_ERR_INVALID_ARG;
  const splash_status st = splash_mask_info_sync_counts(const_cast<splash_mask_info *>(mi));
  if (st != SPLASH_OK) return st;
  if (num_active) *num_active = mi->num_active;
  if (num_partial) *num_partial = mi->num_partial;
  if (num_patterns) *num_patterns = mi->num_patterns;
  if (allowed_pairs) *allowed_pairs = mi->allowed_pairs;
  return SPLASH_OK;
}

splash_status splash_mask_info_set_pattern_source(splash_mask_info *mi, int32_t source) {
  if (mi == nullptr || (source != SPLASH_PATTERNS_STORED && source != SPLASH_PATTERNS_FROM_POSITIONS))
    return SPLASH_ERR_INVALID_ARG;
  mi->patterns_from_positions = source == SPLASH_PATTERNS_FROM_POSITIONS ? 1 : 0;
  return SPLASH_OK;
}

splash_status splash_mask_info_to_host(const splash_mask_info *mi, int8_t *block_mask, int32_t *row_ptr,
                                       int32_t *active_rows, int32_t *active_cols, int32_t *mask_next,
                                       uint8_t *bounds_start, uint8_t *bounds_end,
                                       uint8_t *partial_mask_blocks) {
  if (mi == nullptr || mi->nq <= 0) return SPLASH_ERR_INVALID_ARG;
  const splash_status st = splash_mask_info_sync_counts(const_cast<splash_mask_info *>(mi));
  if (st != SPLASH_OK) return st;
  const int64_t R = (int64_t)mi->batch_rows * mi->nq, A = mi->num_active;
  const int64_t P = mi->num_patterns;
  if (block_mask) SPLASH_CUDA_TRY(cudaMemcpy(block_mask, mi->block_mask, R * mi->nk, cudaMemcpyDeviceToHost));
  if (row_ptr) SPLASH_CUDA_TRY(cudaMemcpy(row_ptr, mi->row_ptr, 4 * (R + 1), cudaMemcpyDeviceToHost));
  if (A > 0) {
    if (active_rows) SPLASH_CUDA_TRY(cudaMemcpy(active_rows, mi->active_rows, 4 * A, cudaMemcpyDeviceToHost));
    if (active_cols) SPLASH_CUDA_TRY(cudaMemcpy(active_cols, mi->active_cols, 4 * A, cudaMemcpyDeviceToHost));
    if (mask_next) SPLASH_CUDA_TRY(cudaMemcpy(mask_next, mi->mask_next, 4 * A, cudaMemcpyDeviceToHost));
    if (bounds_start) SPLASH_CUDA_TRY(cudaMemcpy(bounds_start, mi->bounds_start, A, cudaMemcpyDeviceToHost));
    if (bounds_end) SPLASH_CUDA_TRY(cudaMemcpy(bounds_end, mi->bounds_end, A, cudaMemcpyDeviceToHost));
  }
  if (P > 0 && partial_mask_blocks) {
    // the device keeps the patterns bit-packed; expand them to one byte per element
    const int64_t words = mi->bk / 32, per = (int64_t)mi->bq * words;
    std::vector<uint32_t> bits((size_t)(P * per));
    SPLASH_CUDA_TRY(cudaMemcpy(bits.data(), mi->pattern_bits, bits.size() * sizeof(uint32_t), cudaMemcpyDeviceToHost));
    for (int64_t x = 0; x < P * mi->bq; ++x)
      for (int64_t j = 0; j < mi->bk; ++j)
        partial_mask_blocks[x * mi->bk + j] = (uint8_t)((bits[(size_t)(x * words + j / 32)] >> (j % 32)) & 1u);
  }
  return SPLASH_OK;
}

void splash_mask_info_destroy(splash_mask_info *mi) {
  if (mi == nullptr) return;
  splash_mask_info_free_buffers(mi);
  delete mi;
}

namespace {

// Argument checks shared by the attention entry points; on success *err is
// the device's error word.
splash_status check_attention(const void *q, const void *k, const void *v, int32_t B, int32_t Hq, int32_t Hkv,
                              int64_t Lq, int64_t Lk, int32_t dqk, int32_t dv, const splash_mask_info *mi,
                              float scale, float softcap, const void *out, const void *lse, uint32_t **err) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || lse == nullptr || mi == nullptr)
    return SPLASH_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || dqk <= 0 || dv <= 0)
    return SPLASH_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY) || !(softcap == softcap) || softcap == INFINITY)
    return SPLASH_ERR_INVALID_ARG;  // scale must be positive and finite; NaN / inf cap rejected
  if (Hq % Hkv != 0) return SPLASH_ERR_SHAPE;
  if (mi->nq <= 0 || mi->Lq != Lq || mi->Lk != Lk) return SPLASH_ERR_SHAPE;
  if (mi->batch_rows != 1 && mi->batch_rows != B) return SPLASH_ERR_SHAPE;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
  if (mis & 15u) return SPLASH_ERR_INVALID_ARG;
  const bool shape_ok = ((dqk == 128 && dv == 128) || (dqk == 192 && dv == 128) || (dqk == 64 && dv == 64)) &&
                        (mi->bq == mi->bk || (mi->bq == 256 && mi->bk == 128));
  if (!shape_ok) return SPLASH_ERR_UNSUPPORTED;
  if (mi->bk == 64 && dqk == 192) return SPLASH_ERR_UNSUPPORTED;
  if ((int64_t)B * Hq * Lq >= ((int64_t)1 << 31) || (int64_t)B * Hkv * Lk >= ((int64_t)1 << 31))
    return SPLASH_ERR_UNSUPPORTED;
  int dev = 0;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != mi->device) return SPLASH_ERR_INVALID_ARG;
  *err = splash_device_error_word(dev);
  if (*err == nullptr) return SPLASH_ERR_CUDA;
  return SPLASH_OK;
}

}  // namespace

splash_status splash_attention_fwd(const void *q, const void *k, const void *v, int32_t B, int32_t Hq,
                                   int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk, int32_t dv,
                                   const int32_t *q_segment_ids, const int32_t *kv_segment_ids,
                                   const splash_mask_info *mi, float scale, float softcap, void *out,
                                   float *lse, void *cuda_stream) {
  uint32_t *err = nullptr;
  splash_status st = check_attention(q, k, v, B, Hq, Hkv, Lq, Lk, dqk, dv, mi, scale, softcap, out, lse, &err);
  if (st != SPLASH_OK) return st;
  return splash_attention_fwd_launch(q, k, v, B, Hq, Hkv, Lq, Lk, dqk, dv, q_segment_ids, kv_segment_ids, mi, scale,
                                     softcap, NAN, out, lse, 1, nullptr, nullptr,
                                     static_cast<cudaStream_t>(cuda_stream), err);
}

splash_status splash_attention_fwd_mle(const void *q, const void *k, const void *v, int32_t B, int32_t Hq,
                                       int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk, int32_t dv,
                                       const int32_t *q_segment_ids, const int32_t *kv_segment_ids,
                                       const splash_mask_info *mi, float scale, float softcap, float max_logit,
                                       void *out, float *lse, void *cuda_stream) {
  if (!std::isfinite(max_logit)) return SPLASH_ERR_INVALID_ARG;
  uint32_t *err = nullptr;
  splash_status st = check_attention(q, k, v, B, Hq, Hkv, Lq, Lk, dqk, dv, mi, scale, softcap, out, lse, &err);
  if (st != SPLASH_OK) return st;
  return splash_attention_fwd_launch(q, k, v, B, Hq, Hkv, Lq, Lk, dqk, dv, q_segment_ids, kv_segment_ids, mi, scale,
                                     softcap, max_logit, out, lse, 1, nullptr, nullptr,
                                     static_cast<cudaStream_t>(cuda_stream), err);
}

splash_status splash_attention_fwd_host(const void *q_host, const void *k_host, const void *v_host, int32_t B,
                                        int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk, int32_t dv,
                                        const int32_t *q_segment_ids, const int32_t *kv_segment_ids,
                                        const splash_mask_info *mi, float scale, float softcap, void *out_host,
                                        float *lse_host, void *q_dev, void *k_dev, void *v_dev, void *out_dev,
                                        float *lse_dev, void *cuda_stream) {
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr || out_host == nullptr || lse_host == nullptr)
    return SPLASH_ERR_INVALID_ARG;
  uint32_t *err = nullptr;
  splash_status st =
      check_attention(q_dev, k_dev, v_dev, B, Hq, Hkv, Lq, Lk, dqk, dv, mi, scale, softcap, out_dev, lse_dev, &err);
  if (st != SPLASH_OK) return st;
  return splash_attention_fwd_host_launch(q_host, k_host, v_host, B, Hq, Hkv, Lq, Lk, dqk, dv, q_segment_ids,
                                          kv_segment_ids, mi, scale, softcap,
                                          out_host, lse_host, q_dev, k_dev, v_dev, out_dev, lse_dev, 8,
                                          static_cast<cudaStream_t>(cuda_stream), err);
}

splash_status splash_attention_bwd_workspace_size(int32_t B, int32_t Hq, int64_t Lq, int32_t dqk, size_t *bytes) {
  if (bytes == nullptr || B <= 0 || Hq <= 0 || Lq <= 0 || dqk <= 0) return SPLASH_ERR_INVALID_ARG;
  *bytes = splash_attention_bwd_workspace_bytes(B, Hq, Lq, dqk);
  return SPLASH_OK;
}

splash_status splash_attention_bwd(const void *q, const void *k, const void *v, const void *out, const float *lse,
                                   const void *dout, int32_t B, int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk,
                                   int32_t dqk, int32_t dv, const int32_t *q_segment_ids,
                                   const int32_t *kv_segment_ids, splash_mask_info *mi, float scale, float softcap,
                                   void *dq, void *dk, void *dv_out, void *workspace, size_t workspace_bytes,
                                   void *cuda_stream) {
  (void)q_segment_ids;
  (void)kv_segment_ids;
  if (dout == nullptr || dq == nullptr || dk == nullptr || dv_out == nullptr || workspace == nullptr)
    return SPLASH_ERR_INVALID_ARG;
  uint32_t *err = nullptr;
  splash_status st = check_attention(q, k, v, B, Hq, Hkv, Lq, Lk, dqk, dv, mi, scale, softcap, out, lse, &err);
  if (st != SPLASH_OK) return st;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                        reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv_out) |
                        reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(workspace);
  if (mis & 15u) return SPLASH_ERR_INVALID_ARG;
  if (workspace_bytes < splash_attention_bwd_workspace_bytes(B, Hq, Lq, dqk)) return SPLASH_ERR_INVALID_ARG;
  if (dqk != dv || (dqk != 64 && dqk != 128) || (mi->bq != 128 && mi->bq != 256) || mi->bk != 128)
    return SPLASH_ERR_UNSUPPORTED;
  return splash_attention_bwd_launch(q, k, v, out, lse, dout, B, Hq, Hkv, Lq, Lk, dqk, mi, scale, softcap, dq, dk,
                                     dv_out, workspace, static_cast<cudaStream_t>(cuda_stream), err);
}

splash_status splash_attention_fwd_split(const void *q, const void *k, const void *v, int32_t B, int32_t Hq,
                                         int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk, int32_t dv,
                                         const int32_t *q_segment_ids, const int32_t *kv_segment_ids,
                                         const splash_mask_info *mi, float scale, float softcap,
                                         int32_t num_splits, float *o_part, float *lse_part, void *cuda_stream) {
  if (num_splits < 1 || num_splits > SPLASH_MAX_SPLITS) return SPLASH_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(o_part) & 31u) != 0) return SPLASH_ERR_INVALID_ARG;
  uint32_t *err = nullptr;
  splash_status st =
      check_attention(q, k, v, B, Hq, Hkv, Lq, Lk, dqk, dv, mi, scale, softcap, o_part, lse_part, &err);
  if (st != SPLASH_OK) return st;
  return splash_attention_fwd_launch(q, k, v, B, Hq, Hkv, Lq, Lk, dqk, dv, q_segment_ids, kv_segment_ids, mi, scale,
                                     softcap, NAN, nullptr, nullptr, num_splits, o_part, lse_part,
                                     static_cast<cudaStream_t>(cuda_stream), err);
}

splash_status splash_attention_merge(const float *o_part, const float *lse_part, int32_t num_splits, int64_t rows,
                                     int32_t dv, void *out, float *lse, void *cuda_stream) {
  if (o_part == nullptr || lse_part == nullptr || out == nullptr || lse == nullptr) return SPLASH_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > SPLASH_MAX_SPLITS || rows < 0) return SPLASH_ERR_INVALID_ARG;
  if (dv != 64 && dv != 128) return SPLASH_ERR_UNSUPPORTED;
  if (((reinterpret_cast<uintptr_t>(o_part) | reinterpret_cast<uintptr_t>(out)) & 15u) != 0)
    return SPLASH_ERR_INVALID_ARG;
  return splash_attention_merge_launch(o_part, lse_part, num_splits, rows, dv, out, lse,
                                       static_cast<cudaStream_t>(cuda_stream));
}

splash_status splash_classify_blocks_noalloc(const splash_mask_spec *spec, int64_t Lq, int64_t Lk, int32_t bq,
                                             int32_t bk, int8_t *block_mask, int64_t *totals, void *cuda_stream) {
  if (block_mask == nullptr || totals == nullptr) return SPLASH_ERR_INVALID_ARG;
  splash_status st = check_spec(spec, Lq, Lk);
  if (st != SPLASH_OK) return st;
  if ((st = check_geometry(Lq, Lk, bq, bk)) != SPLASH_OK) return st;
  return splash_classify_blocks_noalloc_impl(spec, Lq, Lk, bq, bk, block_mask, totals,
                                             static_cast<cudaStream_t>(cuda_stream));
}

splash_status splash_last_device_error(void *cuda_stream) {
  int dev = 0;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  SPLASH_CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)));
  uint32_t *addr = splash_device_error_word(dev);
  if (addr == nullptr) return SPLASH_ERR_CUDA;
  uint32_t word = 0;
  SPLASH_CUDA_TRY(cudaMemcpy(&word, addr, sizeof word, cudaMemcpyDeviceToHost));
  if (word != 0) SPLASH_CUDA_TRY(cudaMemset(addr, 0, sizeof word));
  if (word & (SPLASH_DEV_TIMEOUT_PRODUCER | SPLASH_DEV_TIMEOUT_MMA | SPLASH_DEV_TIMEOUT_SOFTMAX |
              SPLASH_DEV_TIMEOUT_DRAIN | SPLASH_DEV_TIMEOUT_SELFTEST | SPLASH_DEV_TIMEOUT_BUILD))
    return SPLASH_ERR_DEVICE_TIMEOUT;
  if (word & (SPLASH_DEV_BAD_TABLE | SPLASH_DEV_SMEM_ALIGN)) return SPLASH_ERR_DEVICE_CHECK;
  return SPLASH_OK;
}

splash_status splash_debug_wait_selftest(uint64_t timeout_ns, void *cuda_stream) {
  if (timeout_ns == 0 || timeout_ns > 2000000000ull) return SPLASH_ERR_INVALID_ARG;
  int dev = 0;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  uint32_t *err = splash_device_error_word(dev);
  if (err == nullptr) return SPLASH_ERR_CUDA;
  splash_status st = splash_wait_selftest_launch(timeout_ns, static_cast<cudaStream_t>(cuda_stream), err);
  if (st != SPLASH_OK) return st;
  return splash_last_device_error(cuda_stream);
}

}  // extern "C"
