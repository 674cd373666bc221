/*
 * splash.h -- C ABI of the GB300 (sm_103a) block-sparse masked attention
 * library (libsplash.so).
 *
 * The operation is the forward pass of "Splash" attention: a mask made of a
 * causal part, a local window and document segment IDs, joined by AND, is
 * preprocessed into a sparse execution table (MaskInfo), and an attention
 * kernel walks only the non-empty key/value blocks of each query block with an
 * online softmax, writing O and the per-row log-sum-exp.
 *
 * Sources:
 *   "Pallas Kernels and Splash Attention" (CMU 11-868 Lecture 13 notes):
 *     §5.1 online softmax; §5.2 the Flash kernel body (m, l, o accumulators,
 *     alpha rescale, deferred normalisation), MHA/GQA; §5.4 soft cap;
 *     §6.1 empty / partial / full blocks; §6.2 MaskInfo (block_mask,
 *     partial_mask_blocks, mask_next, bounds_start / bounds_end); §6.3 the
 *     Splash grid over active blocks and the residual LSE; §6.4 segment IDs
 *     and masks joined by AND.
 *   "The maths and infra behind core LLM operations" (joto.ai): sections
 *     "Causal Mask" (skip blocks above the diagonal, mask only the diagonal
 *     ones) and "LSE and Online Softmax" (LSE = m + log l).
 *
 * Conventions that hold for every call:
 *   - All tensors are caller-owned.  Pointers documented as "device" must be
 *     device memory of the current CUDA device; "host" pointers are ordinary
 *     host memory.  Nothing is retained after a call returns except inside a
 *     splash_mask_info handle.
 *   - `cuda_stream` is a cudaStream_t (NULL = the legacy default stream).
 *     Kernels are launched asynchronously on it.
 *   - No call throws, exits or traps.  Invalid arguments are detected on the
 *     host before any launch and reported as a status; the output buffers are
 *     then untouched.
 *   - Tensor layouts are dense row-major (contiguous), innermost dimension
 *     last.
 */
#ifndef SPLASH_H
#define SPLASH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPLASH_OK = 0,
    SPLASH_ERR_INVALID_ARG = 1,    /* NULL pointer, negative size, bad flag */
    SPLASH_ERR_SHAPE = 2,          /* sizes inconsistent with each other or with the MaskInfo */
    SPLASH_ERR_UNSUPPORTED = 3,    /* valid, but outside what this build implements */
    SPLASH_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
    SPLASH_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait ran out (see splash_last_device_error) */
    SPLASH_ERR_OOM = 6,            /* device allocation failed */
    SPLASH_ERR_DEVICE_CHECK = 7    /* a kernel's bounds check rejected table contents */
} splash_status;

/*
 * The joint mask (AND of the enabled parts), "Pallas Kernels and Splash
 * Attention" §6.1 and §6.4.  Query position i and key position j are 0-based
 * within their sequence; for batch row b the pair is allowed when
 *     (!causal || j <= i)
 *  && (window_left  < 0 || i - j <= window_left)
 *  && (window_right < 0 || j - i <= window_right)
 *  && (q_segment_ids == NULL || q_segment_ids[b][i] == kv_segment_ids[b][j]).
 * A window of W keys including the query itself is window_left = W - 1.
 */
typedef struct {
    int32_t causal;                 /* 0 or 1 */
    int64_t window_left;            /* inclusive distance to the left; -1 = unbounded */
    int64_t window_right;           /* inclusive distance to the right; -1 = unbounded */
    const int32_t *q_segment_ids;   /* device int32 [batch][Lq], or NULL for no document mask */
    const int32_t *kv_segment_ids;  /* device int32 [batch][Lk]; NULL means "same as q_segment_ids"
                                       (then Lq must equal Lk) */
    int32_t batch;                  /* rows of the segment arrays; ignored when q_segment_ids is NULL */
} splash_mask_spec;

/* Opaque, library-owned MaskInfo; freed by splash_mask_info_destroy. */
typedef struct splash_mask_info splash_mask_info;

/*
 * splash_build_mask_info -- preprocess a mask into the sparse execution table
 * ("Pallas Kernels and Splash Attention" §6.2, §6.3, §6.6).
 *
 * Every (bq x bk) block of the [Lq, Lk] mask is classified as empty (0),
 * partial (1) or full (2) (block_mask).  Active (non-empty) blocks are listed
 * in row-major order (q-block ascending, then kv-block ascending) as
 * active_rows / active_cols, with row_ptr giving each q-block row's range
 * (CSR) and bounds_start / bounds_end flagging the first / last active block
 * of a row.  Each partial block's bq x bk element pattern (1 = allowed) is
 * deduplicated by exact content in first-occurrence order into
 * partial_mask_blocks; mask_next[g] is the pattern index of active block g, or
 * -1 when the block is full.
 *
 * With segment IDs the table has B_mask = spec->batch batch rows (one per
 * segment-array row); without them B_mask = 1 and it serves every batch row
 * and head.  Rows are then ordered (b_mask, q-block).
 *
 *   spec        host pointer to the mask; its segment arrays are device memory
 *               and are read on `cuda_stream` before this call returns.
 *   Lq, Lk      sequence lengths (> 0).  When one is not a multiple of its
 *               block, the grid is padded to nq = ceil(Lq/bq) by
 *               nk = ceil(Lk/bk) whole blocks and the padding positions are
 *               masked (§2.3: ragged edges are padded so that every block has
 *               the same size); a block holding padding is never full.
 *   bq, bk      block sizes; this build supports bk in {64, 128} and
 *               bq in {64, 128, 256} (the worked example of "Pallas Kernels
 *               and Splash Attention" §6.2 already uses bq != bk).
 *   cuda_stream stream for the build kernels.
 *   out         receives a new handle (set to NULL on error).
 *
 * Synchronisation: the build kernels are queued on `cuda_stream` and the
 * call returns without waiting, in the usual case: the pattern buffer is
 * sized from a bound known before the build (band-only masks: at most
 * 2 * (ceil((bq-1)/bk) + 1) partial blocks per q-block row, plus one block per
 * row and the last row on a ragged grid; with segment IDs: the number of
 * blocks the causal / window part alone leaves non-empty, since segments only
 * remove pairs).  Only when that bound's bit-packed patterns would exceed
 * 256 MB does the call wait once on `cuda_stream` for the exact pattern
 * count; that path is not capturable in a CUDA graph.  The table may be used
 * by later work on `cuda_stream` at once (work on another stream must wait
 * for it); the totals reach the host only when splash_mask_info_counts or
 * splash_mask_info_to_host asks for them.  A first build allocates the
 * table's device memory (cudaMalloc, which synchronises the device); a
 * rebuild into a handle whose buffers are large enough can then be captured
 * into a CUDA graph on `cuda_stream` (with the attention calls that use it);
 * after a replay, synchronise the stream before asking for the totals.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA, OOM; *out is NULL then.
 */
splash_status splash_build_mask_info(const splash_mask_spec *spec, int64_t Lq, int64_t Lk,
                                     int32_t bq, int32_t bk, void *cuda_stream,
                                     splash_mask_info **out);

/*
 * splash_mask_info_rebuild -- the same computation as splash_build_mask_info,
 * written into an existing handle whose buffers are reused when they are large
 * enough (no device allocation then).  The handle's previous contents are
 * replaced; on error the handle is left empty but valid (destroy it or rebuild
 * it).  Same synchronisation as splash_build_mask_info.
 */
splash_status splash_mask_info_rebuild(splash_mask_info *mi, const splash_mask_spec *spec,
                                       int64_t Lq, int64_t Lk, int32_t bq, int32_t bk,
                                       void *cuda_stream);

/*
 * splash_mask_info_shape -- host-side read of the table's geometry.
 *   batch_rows = B_mask, nq = Lq/bq, nk = Lk/bk.  Any output may be NULL.
 */
splash_status splash_mask_info_shape(const splash_mask_info *mi, int32_t *batch_rows, int64_t *nq,
                                     int64_t *nk, int32_t *bq, int32_t *bk);

/*
 * splash_mask_info_counts -- totals of the table:
 *   num_active    active blocks A (over all batch rows),
 *   num_partial   partial blocks,
 *   num_patterns  distinct partial patterns P,
 *   allowed_pairs allowed (query, key) pairs summed over the batch rows (the
 *                 "useful" entries of the score matrix).  This output is an
 *                 extension of the table the pages describe: the FLOP counts
 *                 of the benchmark are taken from it.
 * After an asynchronous build the first call waits for the build's kernels
 * and copies the totals from the device (later calls read the host copy).
 * Any output may be NULL.
 */
splash_status splash_mask_info_counts(const splash_mask_info *mi, int64_t *num_active,
                                      int64_t *num_partial, int64_t *num_patterns,
                                      int64_t *allowed_pairs);

/*
 * splash_mask_info_to_host -- copy the table into caller-allocated HOST arrays
 * (synchronous).  Sizes: block_mask [B_mask*nq*nk], row_ptr [B_mask*nq + 1],
 * active_rows / active_cols / mask_next / bounds_start / bounds_end [A],
 * partial_mask_blocks [P*bq*bk] (one byte per element, 1 = allowed; the
 * device keeps the patterns bit-packed and they are expanded here).  Any
 * pointer may be NULL to skip that array.
 */
splash_status splash_mask_info_to_host(const splash_mask_info *mi, int8_t *block_mask,
                                       int32_t *row_ptr, int32_t *active_rows,
                                       int32_t *active_cols, int32_t *mask_next,
                                       uint8_t *bounds_start, uint8_t *bounds_end,
                                       uint8_t *partial_mask_blocks);

/*
 * splash_mask_info_set_pattern_source -- where the attention forward takes the
 * element masks of partial blocks from:
 *   SPLASH_PATTERNS_STORED (default): the deduplicated partial_mask_blocks;
 *   SPLASH_PATTERNS_FROM_POSITIONS: computed in the kernel from the query and
 *     key positions (causal / window bounds and ragged-length padding) and,
 *     for a table built with segment IDs, from the segment arrays, the
 *     alternative of "Pallas Kernels and Splash Attention" §6.6 (no pattern
 *     reads; the results are identical).  With segment IDs every forward
 *     call (splash_attention_fwd, _fwd_mle, _fwd_split, _fwd_host) must pass
 *     the arrays the table was built from (same values; device memory, read
 *     by the kernel); a NULL q_segment_ids there returns INVALID_ARG.
 * The setting stays with the handle across rebuilds.  The backward always
 * reads the stored patterns.  Errors: INVALID_ARG (NULL handle, unknown
 * source).
 */
#define SPLASH_PATTERNS_STORED 0
#define SPLASH_PATTERNS_FROM_POSITIONS 1
splash_status splash_mask_info_set_pattern_source(splash_mask_info *mi, int32_t source);

/* Frees the handle and its device memory (NULL is a no-op).  Work queued on
 * other streams that still reads the table must be complete first. */
void splash_mask_info_destroy(splash_mask_info *mi);

/*
 * splash_attention_fwd -- block-sparse masked attention forward
 * ("Pallas Kernels and Splash Attention" §5.1-§5.4, §6.3).
 *
 * For every batch b, query head h and query i, with kv head g = h / (Hq/Hkv):
 *   s_j  = scale * q[b,h,i,:] . k[b,g,j,:]              (fp32 accumulation)
 *   s_j  = softcap * tanh(s_j / softcap)                 (only if softcap > 0)
 *   over the keys j allowed by the MaskInfo's mask:
 *   out[b,h,i,:] = sum_j exp(s_j - m) v[b,g,j,:] / sum_j exp(s_j - m)
 *   lse[b,h,i]   = m + ln(sum_j exp(s_j - m))            (natural log)
 * Rows with no allowed key get out = 0 and lse = -inf.  Only the MaskInfo's
 * active blocks are loaded or computed; partial blocks are masked element by
 * element from partial_mask_blocks (or from positions and segment IDs, see
 * splash_mask_info_set_pattern_source).
 *
 *   q    device bf16 [B][Hq][Lq][dqk]      k  device bf16 [B][Hkv][Lk][dqk]
 *   v    device bf16 [B][Hkv][Lk][dv]      (all 16-byte aligned)
 *   q_segment_ids, kv_segment_ids  the device arrays the MaskInfo was built
 *        from, or NULL.  Read only when the table has segment IDs and its
 *        pattern source is SPLASH_PATTERNS_FROM_POSITIONS (then q_segment_ids
 *        is required; kv_segment_ids NULL means q_segment_ids); the stored
 *        patterns already encode them otherwise.
 *   mi   a MaskInfo built for (Lq, Lk) with B_mask == 1 or B_mask == B.
 *   scale  multiplies q.k (e.g. 1/sqrt(dqk)); must be positive and finite.
 *   softcap <= 0 disables the cap (NaN or +inf is rejected).
 *   out  device bf16 [B][Hq][Lq][dv]       lse device fp32 [B][Hq][Lq]
 *
 * Supported in this build: (dqk, dv) in {(64, 64), (128, 128), (192, 128)},
 * Hq % Hkv == 0, and the MaskInfo's blocks bq == bk in {64, 128} (bk = 128
 * for dqk = 192), or bq = 256 with bk = 128.  The kernel computes in query
 * tiles of 128 rows, two per work item: with bq <= 128 the two tiles are
 * two query heads of one q-block (sharing K / V within a GQA group), with
 * bq = 256 they are the two halves of one q-block of one head and share
 * every K / V tile (this halves the K / V traffic of MHA; blocks of the
 * union that are masked for one half are computed and contribute nothing).
 * Other valid shapes return SPLASH_ERR_UNSUPPORTED.
 * Errors are returned before any launch; kernel-side bounded waits and table
 * checks are reported by splash_last_device_error.
 */
splash_status splash_attention_fwd(const void *q, const void *k, const void *v, int32_t B,
                                   int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk,
                                   int32_t dv, const int32_t *q_segment_ids,
                                   const int32_t *kv_segment_ids, const splash_mask_info *mi,
                                   float scale, float softcap, void *out, float *lse,
                                   void *cuda_stream);

/*
 * splash_attention_fwd_mle -- the same forward with the Max Logit Estimate
 * ("Pallas Kernels and Splash Attention" §5.4): every row's softmax reference
 * is the constant max_logit (natural-log units, the same units as s_j after
 * scale and soft cap) instead of a running maximum, so no block maximum is
 * taken and the accumulator is never rescaled (alpha = 1):
 *   out = sum_j exp(s_j - c) v_j / sum_j exp(s_j - c),  lse = c + ln sum_j exp(s_j - c)
 * which equals splash_attention_fwd's result (c cancels) while c is in the
 * safe range of §5.4 / exercise 10: with a soft cap, c = softcap always is.
 * Outside it:
 *   - a block whose sum of exponentials (base 2, fp32) would reach 2^64
 *     (scores some 40 or more above c) moves that row's reference to the
 *     block's maximum (the overflow guard of the plain kernel), so too small a
 *     c costs time, not accuracy;
 *   - a row whose scores all lie more than about 87 below c underflows: its
 *     sum flushes to 0 and it gets out = 0, lse = -inf, like a fully masked
 *     row (the underflow the lecture warns about; not detected).
 *   max_logit  finite (else SPLASH_ERR_INVALID_ARG)
 * Other arguments, supported shapes and errors as for splash_attention_fwd.
 */
splash_status splash_attention_fwd_mle(const void *q, const void *k, const void *v, int32_t B,
                                       int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk,
                                       int32_t dv, const int32_t *q_segment_ids,
                                       const int32_t *kv_segment_ids, const splash_mask_info *mi,
                                       float scale, float softcap, float max_logit, void *out,
                                       float *lse, void *cuda_stream);

/*
 * splash_attention_fwd_host -- splash_attention_fwd for tensors in host
 * memory: copies q, k, v to the caller's device buffers, runs the forward and
 * copies out and lse back, overlapping the three.  The work is cut into
 * contiguous chunks (whole GQA groups of one batch row when the MaskInfo is
 * shared by the batch; the whole batch at once for a per-batch table) and
 * pipelined on library-owned streams: host -> device copies of one chunk,
 * the attention of the previous one and device -> host copies of the one
 * before run at the same time.  Ordered after prior work on cuda_stream;
 * work queued on cuda_stream afterwards waits for the last copy back.
 *
 *   q_host, k_host, v_host   host bf16, layouts as splash_attention_fwd
 *   out_host, lse_host       host bf16 [B][Hq][Lq][dv] and fp32 [B][Hq][Lq]
 *   q_dev .. lse_dev         device buffers of the full sizes (caller-owned,
 *                            overwritten; alignment as splash_attention_fwd)
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister):
 * copies from pageable memory are correct but do not overlap.  Other
 * arguments, supported shapes and errors as for splash_attention_fwd.
 */
splash_status splash_attention_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                                        int32_t B, int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk,
                                        int32_t dqk, int32_t dv, const int32_t *q_segment_ids,
                                        const int32_t *kv_segment_ids, const splash_mask_info *mi,
                                        float scale, float softcap, void *out_host, float *lse_host,
                                        void *q_dev, void *k_dev, void *v_dev, void *out_dev,
                                        float *lse_dev, void *cuda_stream);

/* Largest num_splits accepted by the split-KV entry points. */
#define SPLASH_MAX_SPLITS 256

/*
 * splash_attention_fwd_split -- the same forward with each q-block row's
 * active list cut into num_splits consecutive ranges ("split-KV"), each a
 * separate work item, so that rows with many active blocks and few rows in
 * total (long keys, few queries) still fill the GPU.  For split s (blocks
 * [nb*s/num_splits, nb*(s+1)/num_splits) of a row with nb active blocks), with
 * J_s its allowed keys and R = B*Hq*Lq:
 *   o_part[s][b][h][i][:]  = sum_{j in J_s} exp(s_j - lse_s) v[b,g,j,:]   (fp32)
 *   lse_part[s][b][h][i]   = ln sum_{j in J_s} exp(s_j)
 * with o_part = 0 and lse_part = -inf where J_s is empty.  splash_attention_merge
 * turns them into out / lse equal to splash_attention_fwd's: this is the merge
 * of softmax segments through their log-sum-exp ("The maths and infra behind
 * core LLM operations" (joto.ai), "LSE and Online Softmax"; "Pallas Kernels
 * and Splash Attention" §5.1).
 *
 *   num_splits  1 .. SPLASH_MAX_SPLITS (splits beyond a row's block count are
 *               empty)
 *   o_part      device fp32 [num_splits][B][Hq][Lq][dv], 32-byte aligned
 *   lse_part    device fp32 [num_splits][B][Hq][Lq]
 * Both are caller-owned workspace, fully overwritten.  Other arguments,
 * supported shapes and errors as for splash_attention_fwd.
 */
splash_status splash_attention_fwd_split(const void *q, const void *k, const void *v, int32_t B,
                                         int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk,
                                         int32_t dv, const int32_t *q_segment_ids,
                                         const int32_t *kv_segment_ids, const splash_mask_info *mi,
                                         float scale, float softcap, int32_t num_splits, float *o_part,
                                         float *lse_part, void *cuda_stream);

/*
 * splash_attention_merge -- combines split-KV partials (layout above, rows =
 * B*Hq*Lq):  m = max_s lse_part[s][r];  lse[r] = m + ln sum_s exp(lse_part[s][r] - m);
 * out[r][:] = sum_s exp(lse_part[s][r] - lse[r]) o_part[s][r][:]  (bf16);
 * rows whose splits are all empty get out = 0, lse = -inf.
 *   o_part  device fp32, 16-byte aligned     lse_part  device fp32
 *   dv      64 or 128 (else SPLASH_ERR_UNSUPPORTED)
 *   out     device bf16 [rows][dv], 16-byte aligned    lse  device fp32 [rows]
 */
splash_status splash_attention_merge(const float *o_part, const float *lse_part, int32_t num_splits,
                                     int64_t rows, int32_t dv, void *out, float *lse, void *cuda_stream);

/*
 * splash_attention_bwd -- gradients of splash_attention_fwd with respect to
 * q, k and v for an upstream gradient dout, from the forward's out and lse
 * ("Pallas Kernels and Splash Attention" §6.3: the forward's residual outputs
 * serve the backward; "The maths and infra behind core LLM operations"
 * (joto.ai), "LSE and Online Softmax": the probabilities are recomputed from
 * the scores and LSE, P_ij = exp(s_ij - lse_i), instead of being stored).
 * With dP_ij = dout_i . v_j, D_i = dout_i . out_i and
 *   dS_ij = P_ij (dP_ij - D_i)  (times 1 - tanh^2(scale q.k / softcap) with a cap):
 *   dv[b,g,j,:] = sum over heads h of group g, allowed i: P_ij dout[b,h,i,:]
 *   dk[b,g,j,:] = scale * sum over h, i: dS_ij q[b,h,i,:]
 *   dq[b,h,i,:] = scale * sum over allowed j: dS_ij k[b,g,j,:]
 * (masked pairs contribute nothing; a key no query sees gets dk = dv = 0).
 * Only the MaskInfo's active blocks are computed, visited column by column:
 * the first call after each build (or rebuild) of the MaskInfo makes a
 * column-major copy of the table inside it (device memory allocated on
 * first use, hence the non-const handle), and later calls reuse it; a call
 * on another stream waits for the copy's completion.
 *
 *   q, k, v, mi, scale, softcap   exactly as given to the forward
 *   out  device bf16 [B][Hq][Lq][dv], lse device fp32 [B][Hq][Lq]: the forward's outputs
 *   dout device bf16 [B][Hq][Lq][dv]
 *   dq   device bf16 [B][Hq][Lq][dqk]   dk device bf16 [B][Hkv][Lk][dqk]
 *   dv_out device bf16 [B][Hkv][Lk][dv]   (all fully overwritten)
 *   workspace  device, 16-byte aligned, at least
 *              splash_attention_bwd_workspace_size(B, Hq, Lq, dqk) bytes
 *              (an fp32 dq accumulator, D and a copy of lse, over whole
 *              256-row blocks per head); caller-owned, overwritten.
 * All device pointers 16-byte aligned.  Supported: dqk == dv in {64, 128}
 * and MaskInfo blocks bk = 128 with bq = 128 or 256 (a 256-row q-block is
 * taken as two 128-row halves), any Lq / Lk (ragged lengths as in the
 * forward); other valid shapes return SPLASH_ERR_UNSUPPORTED.  dq is accumulated with fp32 atomic additions, so
 * its last bits may differ between runs; dk and dv are deterministic.
 * Errors as for splash_attention_fwd.
 */
splash_status splash_attention_bwd_workspace_size(int32_t B, int32_t Hq, int64_t Lq, int32_t dqk,
                                                  size_t *bytes);
splash_status splash_attention_bwd(const void *q, const void *k, const void *v, const void *out,
                                   const float *lse, const void *dout, int32_t B, int32_t Hq,
                                   int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk, int32_t dv,
                                   const int32_t *q_segment_ids, const int32_t *kv_segment_ids,
                                   splash_mask_info *mi, float scale, float softcap, void *dq,
                                   void *dk, void *dv_out, void *workspace, size_t workspace_bytes,
                                   void *cuda_stream);

/*
 * splash_classify_blocks_noalloc -- the block classification of a mask
 * (block_mask and its totals), computed without allocating any device memory.
 * The pages have no counterpart: this exists for callers that must not call
 * cudaMalloc, such as a process whose device memory is owned by its own pool
 * allocator under a fixed budget, where an allocation outside the pool can fail
 * or break the pool's accounting.
 *
 * It runs the same classification as splash_build_mask_info, but its working
 * memory (per-row counters, segment summaries, the list of blocks the
 * summaries cannot decide, totals; about 640 KiB) is a fixed array inside the
 * library's module, present on every GPU that loads the library until the
 * process exits.  The first call on a device looks that array up (once per
 * device, under a lock).  Every call ends by copying the totals to the host
 * and synchronising `cuda_stream`, so it cannot be called while that stream
 * is being captured into a CUDA graph.
 *
 *   spec, Lq, Lk, bq, bk  as for splash_build_mask_info.
 *   block_mask  device int8 [B_mask][nq][nk], caller-allocated: 0 empty,
 *               1 partial, 2 full (identical to the MaskInfo's block_mask).
 *   totals      host int64 [4]: active blocks, partial blocks, allowed
 *               (query, key) pairs, and the largest active-block count of a
 *               q-block row.
 * Limits: B_mask * nq <= 16384 and B_mask * nk <= 16384; larger masks return
 * SPLASH_ERR_UNSUPPORTED before any launch.  All calls share the one array
 * (its counters are cleared at the start of each call), so calls that
 * overlap on the GPU -- other streams or other host threads -- race and must
 * be serialised by the caller.
 */
splash_status splash_classify_blocks_noalloc(const splash_mask_spec *spec, int64_t Lq, int64_t Lk,
                                             int32_t bq, int32_t bk, int8_t *block_mask,
                                             int64_t *totals, void *cuda_stream);

/*
 * splash_last_device_error -- synchronises `cuda_stream`, then reads and
 * clears the device error word that the library's kernels set when a bounded
 * wait runs out (SPLASH_ERR_DEVICE_TIMEOUT) or a table entry fails a bounds
 * check (SPLASH_ERR_DEVICE_CHECK).  Returns SPLASH_OK when no kernel
 * reported anything, SPLASH_ERR_CUDA when the synchronisation itself fails.
 */
splash_status splash_last_device_error(void *cuda_stream);

/*
 * splash_debug_wait_selftest -- launches one tiny kernel whose mbarrier wait
 * can never be satisfied (nothing arrives on it), bounded by timeout_ns
 * nanoseconds, and returns what splash_last_device_error then reports
 * (SPLASH_ERR_DEVICE_TIMEOUT when the bound works).  It exercises the same
 * bounded-wait helper the attention kernel uses, without faulting or hanging
 * the device.  timeout_ns must be in (0, 2e9].
 */
splash_status splash_debug_wait_selftest(uint64_t timeout_ns, void *cuda_stream);

/*
 * splash_kernel_launches -- number of kernels this library has launched in
 * this process so far (all devices, all entry points).  Host-side counter,
 * thread-safe; for accounting in benchmarks.
 */
uint64_t splash_kernel_launches(void);

/*
 * splash_shard_items -- the share of one rank when a workload is split
 * across `world` GPUs by (batch, KV head) groups (host logic, no device
 * work).  "Pallas Kernels and Splash Attention" §5.2: heads are independent,
 * and the query heads of a GQA group read the same K / V, so a group is
 * never split: the n = B * Hkv groups, in (batch, KV head) row-major order,
 * are dealt in balanced contiguous ranges, rank r taking groups
 * [floor(n r / world), floor(n (r + 1) / world)).  Group g covers batch
 * g / Hkv and query heads (g % Hkv) * (Hq / Hkv) ... + Hq / Hkv - 1, which
 * in the [B][H][L][d] layouts of q, k, v, out and lse is one contiguous
 * range of memory per tensor, so a rank passes sub-tensors of the caller's
 * tensors as a problem of (end - begin) batch rows with Hq / Hkv query heads
 * and one KV head (with segment IDs, row g / Hkv of the segment array for
 * each group).  The ranges of ranks 0 .. world-1 tile [0, n) with no gap or
 * overlap; a rank may get an empty range when world > n.
 *   B, Hkv        batch size and KV heads of the whole workload (> 0)
 *   world, rank   number of ranks (> 0) and this rank (0 <= rank < world)
 *   begin, end    out: this rank's half-open range of groups
 * Errors: SPLASH_ERR_INVALID_ARG for null outputs or values out of range.
 * Thread-safe, no side effects.
 */
splash_status splash_shard_items(int32_t B, int32_t Hkv, int32_t world, int32_t rank, int64_t *begin,
                                 int64_t *end);

/*
 * splash_schedule_head_group -- the forward's item order across heads, as
 * the attention call chooses it (host logic, no device work): the number of
 * heads (256-row q-blocks) or head pairs whose items are dealt together.
 * The kernel deals its items in rounds of `grid` (one per CTA), rows longest
 * first, all heads of a row together; when the rows reach across the keys
 * (dense_rows: no window, no segment IDs) and the K / V of all heads
 * (kv_bytes) exceeds 64 MB, the items are ordered by groups of heads whose
 * K / V fits that budget, and among the group sizes from half the largest
 * such size up to it, the one whose items (items_per_head per head) leave
 * the fewest in a partial round.  Returns npairs when no grouping applies.
 *   dense_rows      1 if the mask has neither a window nor segment IDs
 *   items_per_head  work items per head (pair): q-block rows x batch x splits
 *   npairs          heads (256-row q-blocks) or head pairs
 *   kv_bytes        bytes of all heads' K and V
 *   grid            CTAs of the launch (min(items, SMs))
 * Invalid arguments (npairs < 1, items_per_head < 1, grid < 1, kv_bytes < 0)
 * return 0.  The pages have no counterpart (their grid is scheduled by the
 * TPU compiler); this is the GB300 kernel's own work order, exposed so that
 * it can be checked without a GPU.  Thread-safe, no side effects.
 */
int32_t splash_schedule_head_group(int32_t dense_rows, int64_t items_per_head, int32_t npairs, int64_t kv_bytes,
                                   int64_t grid);

/* Static description of a status code (never NULL). */
const char *splash_status_string(splash_status status);

/* Library version string, e.g. "splash-gb300 0.1 sm_103a". */
const char *splash_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPLASH_H */
