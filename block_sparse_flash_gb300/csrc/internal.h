// internal.h -- declarations shared by the translation units of libsplash.so.
// Not part of the public ABI (that is include/splash.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "splash.h"

// Error bits of the device error word (set with atomicOr by kernels).
enum : uint32_t {
  SPLASH_DEV_TIMEOUT_PRODUCER = 1u << 0,
  SPLASH_DEV_TIMEOUT_MMA = 1u << 1,
  SPLASH_DEV_TIMEOUT_SOFTMAX = 1u << 2,
  SPLASH_DEV_TIMEOUT_DRAIN = 1u << 3,
  SPLASH_DEV_TIMEOUT_SELFTEST = 1u << 4,
  SPLASH_DEV_TIMEOUT_BUILD = 1u << 5,  // the one-launch MaskInfo build gave up at a grid barrier
  SPLASH_DEV_BAD_TABLE = 1u << 8,
  SPLASH_DEV_SMEM_ALIGN = 1u << 9,  // dynamic shared memory not 1024-byte aligned: the kernel did nothing
};

// The library-owned sparse execution table ("Pallas Kernels and Splash
// Attention" §6.2).  All arrays are device memory of `device`.
struct splash_mask_info {
  int device = -1;
  // geometry
  int32_t batch_rows = 0;  // B_mask
  int64_t Lq = 0, Lk = 0, nq = 0, nk = 0;
  int32_t bq = 0, bk = 0;
  // the mask it was built from (segment arrays are not retained)
  int32_t causal = 0;
  int64_t window_left = -1, window_right = -1;
  int32_t has_segments = 0;
  // the forward computes partial blocks' masks from positions (and, for a
  // table with segment IDs, from the arrays the caller passes to it) instead
  // of reading the stored patterns
  int32_t patterns_from_positions = 0;
  // totals (host copies)
  int64_t num_active = 0, num_partial = 0, num_patterns = 0, allowed_pairs = 0;
  int32_t max_row_blocks = 0;

  // --- table arrays (public content) ---
  int8_t *block_mask = nullptr;    // [R*nk]
  int32_t *row_ptr = nullptr;      // [R+1]
  int32_t *active_rows = nullptr;  // [cap_active]
  int32_t *active_cols = nullptr;  // [cap_active]
  int32_t *mask_next = nullptr;    // [cap_active]
  uint8_t *bounds_start = nullptr; // [cap_active]
  uint8_t *bounds_end = nullptr;   // [cap_active]
  // --- derived arrays used by the attention kernel ---
  // the partial patterns, bit-packed (partial_mask_blocks in byte form is
  // expanded from these when the table is copied to the host)
  uint32_t *pattern_bits = nullptr;  // [cap_patterns][bq][bk/32], bit dj of word dj/32 = allowed
  int32_t *row_order = nullptr;      // [R] rows by descending active count (longest first)
  // --- build scratch ---
  int32_t *row_cnt = nullptr;      // [R]
  int32_t *row_pcnt = nullptr;     // [R]
  int32_t *prow_ptr = nullptr;     // [R+1]
  int32_t *seg_summary = nullptr;  // [R*2 + B_mask*nk*2] (min, max) per q-block then per kv-block
  int32_t *part_row = nullptr;     // [cap_active] global row (b_mask*nq + r) of the k-th partial block
  int32_t *part_col = nullptr;     // [cap_active]
  int32_t *part_g = nullptr;       // [cap_active] its active index
  uint64_t *part_hash = nullptr;   // [cap_active]
  int32_t *part_rep = nullptr;     // [cap_active] first partial with identical content
  int32_t *part_pidx = nullptr;    // [cap_active] pattern index (valid for representatives)
  int32_t *rep_list = nullptr;     // [cap_active] partial index of pattern u
  int32_t *row_hist = nullptr;     // [nk+1] counting-sort bins
  unsigned long long *counters = nullptr;  // [8]: A, A_p, P, allowed, max_row, deferred blocks
  unsigned int *grid_sync = nullptr;       // the one-launch build: barrier counter, spare, first-occurrence bitmap
  uint32_t *part_bits = nullptr;           // [cap_part_bits] one-launch build: each partial block's words
  unsigned long long *ht_key = nullptr;    // [cap_ht] one-launch build: content hash table (keys)
  int32_t *ht_val = nullptr;               // [cap_ht] smallest partial index per key
  int64_t cap_part_bits = 0, cap_ht = 0;
  // host staging
  unsigned long long *h_counters = nullptr;  // pinned [8]
  // counts of an asynchronous build: `counts_ready` is recorded after its last
  // kernel; splash_mask_info_sync_counts waits for it and copies the totals
  cudaEvent_t counts_ready = nullptr;
  bool counts_pending = false;
  bool counts_captured = false;  // the last build was captured into a graph (no event recorded)

  // capacities (elements)
  int64_t cap_rows = 0, cap_blocks = 0, cap_seg = 0, cap_patterns = 0, cap_hist = 0;

  // incremented by every build of the table
  uint64_t build_gen = 0;

  // --- column-major (transposed) table for the backward pass, made by the
  // first backward call after each build and reused while build_gen is
  // unchanged; allocated on first use ---
  int32_t *t_col_cnt = nullptr;       // [B_mask*nk]
  int32_t *t_col_ptr = nullptr;       // [B_mask*nk + 1]
  int32_t *t_col_rows = nullptr;      // [cap_blocks] q-block of each active block, by column
  int32_t *t_col_next = nullptr;      // [cap_blocks] its pattern index or -1
  uint32_t *t_pattern_bits = nullptr; // [cap_patterns][bk][bq/32], bit of (query, key) by key row
  int64_t t_cap_cols = 0, t_cap_active = 0, t_cap_patterns = 0;  // (t_cap_patterns counts words)
  uint64_t t_gen = 0;             // build_gen the copy was made from (0: none)
  cudaEvent_t t_ready = nullptr;  // recorded on the stream that made it
};

// mask_info.cu
splash_status splash_mask_info_build_into(splash_mask_info *mi, const splash_mask_spec *spec,
                                          int64_t Lq, int64_t Lk, int32_t bq, int32_t bk,
                                          cudaStream_t stream);
void splash_mask_info_free_buffers(splash_mask_info *mi);
void splash_mask_info_free_transposed(splash_mask_info *mi);
// attention_fwd.cu: the forward's head-group choice (see splash_schedule_head_group)
int32_t splash_choose_head_group(bool dense_rows, int64_t items_per_head, int32_t npairs, int64_t kv_bytes,
                                 int64_t grid);
// Makes the host totals current (waits for an asynchronous build's copy).
splash_status splash_mask_info_sync_counts(splash_mask_info *mi);
splash_status splash_classify_blocks_noalloc_impl(const splash_mask_spec *spec, int64_t Lq, int64_t Lk,
                                                  int32_t bq, int32_t bk, int8_t *block_mask,
                                                  int64_t *totals, cudaStream_t stream);

// api.cu
uint32_t *splash_device_error_word(int device);  // device address of the error word (or NULL)

// attention_fwd.cu
// nsplit > 1: split-KV partials into o_part / lse_part (out / lse unused).
splash_status splash_attention_fwd_launch(const void *q, const void *k, const void *v, int32_t B,
                                          int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk,
                                          int32_t dqk, int32_t dv, const int32_t *q_segment_ids,
                                          const int32_t *kv_segment_ids, const splash_mask_info *mi,
                                          float scale, float softcap, float max_logit, void *out,
                                          float *lse, int32_t nsplit, float *o_part, float *lse_part,
                                          cudaStream_t stream, uint32_t *err_word);
// attention_fwd.cu, compiled once per pattern mode (stored, band, band and
// segment IDs) so that the three sets of kernel instantiations build in
// parallel: the launchers of each mode (same arguments as
// splash_attention_fwd_launch, which picks one)
#define SPLASH_FWD_LAUNCHER_ARGS                                                                                 \
  const void *q, const void *k, const void *v, int32_t B, int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk,      \
      int32_t dqk, int32_t dv, const int32_t *q_segment_ids, const int32_t *kv_segment_ids,                       \
      const splash_mask_info *mi, float scale, float softcap, float max_logit, void *out, float *lse,             \
      int32_t nsplit, float *o_part, float *lse_part, cudaStream_t stream, uint32_t *err_word
splash_status splash_fwd_launch_stored(SPLASH_FWD_LAUNCHER_ARGS);
splash_status splash_fwd_launch_band(SPLASH_FWD_LAUNCHER_ARGS);
splash_status splash_fwd_launch_band_seg(SPLASH_FWD_LAUNCHER_ARGS);
splash_status splash_attention_merge_launch(const float *o_part, const float *lse_part, int32_t nsplit,
                                            int64_t rows, int32_t dv, void *out, float *lse,
                                            cudaStream_t stream);
// attention_bwd.cu (bq = bk = 128, dqk = dv = d in {64, 128})
size_t splash_attention_bwd_workspace_bytes(int32_t B, int32_t Hq, int64_t Lq, int32_t dqk);
splash_status splash_attention_bwd_launch(const void *q, const void *k, const void *v, const void *out,
                                          const float *lse, const void *dout, int32_t B, int32_t Hq, int32_t Hkv,
                                          int64_t Lq, int64_t Lk, int32_t d, splash_mask_info *mi, float scale,
                                          float softcap, void *dq, void *dk, void *dv, void *workspace,
                                          cudaStream_t stream, uint32_t *err_word);
// host_pipeline.cu
splash_status splash_attention_fwd_host_launch(const void *q_h, const void *k_h, const void *v_h, int32_t B,
                                               int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk,
                                               int32_t dv, const int32_t *q_segment_ids,
                                               const int32_t *kv_segment_ids, const splash_mask_info *mi,
                                               float scale, float softcap, void *out_h, float *lse_h, void *q_d, void *k_d, void *v_d,
                                               void *out_d, float *lse_d, int32_t target_chunks,
                                               cudaStream_t stream, uint32_t *err);
splash_status splash_wait_selftest_launch(uint64_t timeout_ns, cudaStream_t stream,
                                          uint32_t *err_word);

// Counts kernel launches (splash_kernel_launches); call once per launch.
void splash_count_launches(uint64_t n);

#define SPLASH_CUDA_TRY(expr)                         \
  do {                                                \
    cudaError_t _e = (expr);                          \
    if (_e != cudaSuccess) return SPLASH_ERR_CUDA;    \
  } while (0)
