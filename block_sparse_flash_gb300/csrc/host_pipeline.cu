// host_pipeline.cu -- the attention forward for inputs and outputs in host
// memory, with the host <-> device copies overlapped with the computation.
//
// The work is cut into chunks of whole (batch, GQA group) slices -- every
// chunk is one contiguous range of q / k / v / out / lse rows -- and run as a
// three-stage pipeline on library-owned streams: host -> device copies of
// chunk c+1 (one copy engine), the attention kernel of chunk c, and device ->
// host copies of chunk c-1 (the other copy engine) proceed at the same time.
// Ordering with the caller's stream is kept by events at entry and exit.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "internal.h"

namespace {

constexpr int kMaxChunks = 32;

struct PipelineContext {
  bool ready = false;
  cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_done[kMaxChunks] = {}, comp_done[kMaxChunks] = {};
};

std::mutex g_mu;
std::vector<PipelineContext> g_ctx;  // per device

splash_status context_for(int dev, PipelineContext **out) {
  if ((int)g_ctx.size() <= dev) g_ctx.resize(dev + 1);
  PipelineContext &c = g_ctx[dev];
  if (!c.ready) {
    SPLASH_CUDA_TRY(cudaStreamCreateWithFlags(&c.s_in, cudaStreamNonBlocking));
    SPLASH_CUDA_TRY(cudaStreamCreateWithFlags(&c.s_comp, cudaStreamNonBlocking));
    SPLASH_CUDA_TRY(cudaStreamCreateWithFlags(&c.s_out, cudaStreamNonBlocking));
    SPLASH_CUDA_TRY(cudaEventCreateWithFlags(&c.start, cudaEventDisableTiming));
    SPLASH_CUDA_TRY(cudaEventCreateWithFlags(&c.done, cudaEventDisableTiming));
    for (int x = 0; x < kMaxChunks; ++x) {
      SPLASH_CUDA_TRY(cudaEventCreateWithFlags(&c.in_done[x], cudaEventDisableTiming));
      SPLASH_CUDA_TRY(cudaEventCreateWithFlags(&c.comp_done[x], cudaEventDisableTiming));
    }
    c.ready = true;
  }
  *out = &c;
  return SPLASH_OK;
}

}  // namespace

splash_status splash_attention_fwd_host_launch(const void *q_h, const void *k_h, const void *v_h, int32_t B,
                                               int32_t Hq, int32_t Hkv, int64_t Lq, int64_t Lk, int32_t dqk,
                                               int32_t dv, const int32_t *q_segment_ids,
                                               const int32_t *kv_segment_ids, const splash_mask_info *mi,
                                               float scale, float softcap, void *out_h, float *lse_h, void *q_d, void *k_d, void *v_d,
                                               void *out_d, float *lse_d, int32_t target_chunks,
                                               cudaStream_t stream, uint32_t *err) {
  int dev = 0;
  SPLASH_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_mu);
  PipelineContext *c = nullptr;
  splash_status st = context_for(dev, &c);
  if (st != SPLASH_OK) return st;

  // chunks: whole GQA groups of one batch row while the table is shared by
  // the batch (B_mask = 1); a per-batch table (segment IDs with B > 1) keeps
  // the batch whole, so the kernel sees every batch row it indexes
  const int32_t G = Hq / Hkv;
  int32_t per_batch = 1;  // chunks per batch row
  if (mi->batch_rows == 1) {
    const int32_t want = std::max(1, std::min(target_chunks, kMaxChunks) / std::max(1, B));
    per_batch = std::max(1, std::min(Hkv, want));
  }
  struct Chunk {
    int32_t b0, nb, kv0, nkv;
  };
  std::vector<Chunk> chunks;
  if (mi->batch_rows == 1) {
    for (int32_t b = 0; b < B; ++b)
      for (int32_t g = 0; g < per_batch; ++g) {
        const int32_t kv0 = (int32_t)((int64_t)Hkv * g / per_batch), kv1 = (int32_t)((int64_t)Hkv * (g + 1) / per_batch);
        if (kv1 > kv0) chunks.push_back({b, 1, kv0, kv1 - kv0});
      }
  } else {
    chunks.push_back({0, B, 0, Hkv});
  }
  if ((int)chunks.size() > kMaxChunks) return SPLASH_ERR_UNSUPPORTED;

  SPLASH_CUDA_TRY(cudaEventRecord(c->start, stream));
  SPLASH_CUDA_TRY(cudaStreamWaitEvent(c->s_in, c->start, 0));
  SPLASH_CUDA_TRY(cudaStreamWaitEvent(c->s_comp, c->start, 0));
  SPLASH_CUDA_TRY(cudaStreamWaitEvent(c->s_out, c->start, 0));
  const size_t q_row = (size_t)dqk * 2, kv_row = (size_t)dqk * 2, v_row = (size_t)dv * 2, o_row = (size_t)dv * 2;
  for (size_t x = 0; x < chunks.size(); ++x) {
    const Chunk &ch = chunks[x];
    // a chunk is contiguous: batch rows b0 .. b0+nb-1 are whole when nb > 1,
    // else heads kv0*G .. (kv0+nkv)*G-1 of batch b0
    const int64_t q_first = ((int64_t)ch.b0 * Hq + (int64_t)ch.kv0 * G) * Lq;  // q / out / lse rows
    const int64_t q_rows = (int64_t)ch.nb * ch.nkv * G * Lq;
    const int64_t kv_first = ((int64_t)ch.b0 * Hkv + ch.kv0) * Lk;
    const int64_t kv_rows = (int64_t)ch.nb * ch.nkv * Lk;
    char *qd = static_cast<char *>(q_d) + q_first * q_row;
    char *kd = static_cast<char *>(k_d) + kv_first * kv_row;
    char *vd = static_cast<char *>(v_d) + kv_first * v_row;
    char *od = static_cast<char *>(out_d) + q_first * o_row;
    float *ld = lse_d + q_first;
    SPLASH_CUDA_TRY(cudaMemcpyAsync(qd, static_cast<const char *>(q_h) + q_first * q_row, q_rows * q_row,
                                    cudaMemcpyHostToDevice, c->s_in));
    SPLASH_CUDA_TRY(cudaMemcpyAsync(kd, static_cast<const char *>(k_h) + kv_first * kv_row, kv_rows * kv_row,
                                    cudaMemcpyHostToDevice, c->s_in));
    SPLASH_CUDA_TRY(cudaMemcpyAsync(vd, static_cast<const char *>(v_h) + kv_first * v_row, kv_rows * v_row,
                                    cudaMemcpyHostToDevice, c->s_in));
    SPLASH_CUDA_TRY(cudaEventRecord(c->in_done[x], c->s_in));
    SPLASH_CUDA_TRY(cudaStreamWaitEvent(c->s_comp, c->in_done[x], 0));
    // segment arrays: their rows follow the table's batch rows (one row
    // when B_mask = 1; the whole batch is one chunk when B_mask = B)
    st = splash_attention_fwd_launch(qd, kd, vd, ch.nb, ch.nkv * G, ch.nkv, Lq, Lk, dqk, dv, q_segment_ids,
                                     kv_segment_ids, mi, scale, softcap, NAN, od, ld, 1, nullptr, nullptr, c->s_comp,
                                     err);
    if (st != SPLASH_OK) return st;
    SPLASH_CUDA_TRY(cudaEventRecord(c->comp_done[x], c->s_comp));
    SPLASH_CUDA_TRY(cudaStreamWaitEvent(c->s_out, c->comp_done[x], 0));
    SPLASH_CUDA_TRY(cudaMemcpyAsync(static_cast<char *>(out_h) + q_first * o_row, od, q_rows * o_row,
                                    cudaMemcpyDeviceToHost, c->s_out));
    SPLASH_CUDA_TRY(cudaMemcpyAsync(lse_h + q_first, ld, q_rows * sizeof(float), cudaMemcpyDeviceToHost, c->s_out));
  }
  // the caller's stream continues after the last copy back (and after the
  // other two streams' work, which the last copy depends on)
  SPLASH_CUDA_TRY(cudaEventRecord(c->done, c->s_out));
  SPLASH_CUDA_TRY(cudaStreamWaitEvent(stream, c->done, 0));
  return SPLASH_OK;
}
