// sv_internal.h -- host-side plumbing between the C ABI and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "spec_verify.h"

struct spec_verify_ctx {
  spec_verify_config cfg;
  int num_sms;
  int max_cluster;  // largest cluster size the kernels were enabled for (8 or 16)
  int max_dyn_smem; // dynamic shared memory the logits kernels may request per CTA
  int smem_per_sm;  // shared memory of one SM (for the CTAs-per-SM target of the layout)
  int max_dyn_optin;  // dynamic shared memory a CTA without static shared memory may request
};

namespace sv {

// Everything a verifier kernel needs, flattened (device pointers, sizes).
struct VerifyParams {
  int32_t N, G, V;
  int64_t T;
  const int32_t *ids;
  const int32_t *cu;
  const void *target;
  int64_t target_stride;
  const void *draft;
  int64_t draft_stride;
  const float *temperature;
  const int32_t *top_k;
  const float *top_p;
  const float *uniforms;
  const float *exponentials;
  int64_t exp_stride;
  uint32_t seed_lo, seed_hi, off_lo, off_hi;
  uint32_t req_base;
  int32_t *out;
  int32_t *nacc;
  int32_t *ncomp;
  int64_t *slots;
  float *dbg_py;
  float *dbg_qy;
  int32_t *status;
  const float *rates;  // synthetic acceptance rates [G] or nullptr
  // logits processors and stop tokens (per-request lists, inclusive prefix sums)
  const float *rep_penalty;
  const int64_t *pen_cu;
  const int32_t *pen_ids;
  int64_t pen_total;
  const int64_t *ban_cu;
  const int32_t *ban_ids;
  int64_t ban_total;
  const int64_t *stop_cu;
  const int32_t *stop_ids;
  int64_t stop_total;
  uint32_t first_wait;  // polls of the first wait for a bulk row copy (0 under SV_TEST_EXPIRE_COPY_WAIT)
  bool pdl;             // launch with programmatic stream serialization (host side only)
};

// The draft-side sampler's parameters (device pointers, sizes).
struct SampleParams {
  int32_t R, V;
  const void *logits;
  int64_t row_stride;
  const float *temperature;
  const int32_t *top_k;
  const float *top_p;
  const float *exponentials;
  int64_t exp_stride;
  uint32_t seed_lo, seed_hi, off_lo, off_hi;
  uint32_t row_base;
  int32_t *tokens;
  float *probs;
  int64_t probs_stride;
  int32_t *status;
  const float *rep_penalty;
  const int64_t *pen_cu;
  const int32_t *pen_ids;
  int64_t pen_total;
  const int64_t *ban_cu;
  const int32_t *ban_ids;
  int64_t ban_total;
  uint32_t first_wait;  // polls of the first wait for a bulk row copy (0 under SV_TEST_EXPIRE_COPY_WAIT)
  bool pdl;             // launch with programmatic stream serialization (host side only)
};

// The n-gram proposer's parameters (device pointers, sizes).
struct NgramParams {
  int32_t R, min_n, max_n, k;
  int64_t max_model_len, total;
  const int32_t *tokens;
  const int64_t *cu;
  int32_t *out;
  int32_t *num;
  int32_t *status;
  bool pdl;  // launch with programmatic stream serialization (host side only)
};

// The attributes of every kernel launch: a cluster of `cluster` CTAs (none
// for 0) and, with `pdl`, programmatic stream serialization, which lets the
// kernel be scheduled while the previous kernel in the stream finishes (each
// kernel first waits for that grid's completion: pdl_enter in sv_device.cuh).
// Fills attr[0..] and returns the count.
inline unsigned launch_attrs(cudaLaunchAttribute attr[2], unsigned cluster, bool pdl) {
  unsigned n = 0;
  if (cluster) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  return n;
}
cudaError_t launch_ngram(const NgramParams &p, cudaStream_t stream);

// Polls of the ordinary wait for a bulk row copy (each poll may suspend for a while).
constexpr uint32_t kCopyWaitPolls = 1u << 20;

// Picks the CTAs-per-request for a call (power of two, <= ctx->max_cluster).
int choose_cluster(const spec_verify_ctx *ctx, int N, int V);

cudaError_t enable_probs_kernels(int max_cluster);
cudaError_t launch_probs(const VerifyParams &p, int cluster, bool vec, cudaStream_t stream);

size_t logits_static_smem();
int logits_reg_group_chunk();  // largest bf16 chunk whose group maxima stay in registers
// Dynamic shared memory a logits-entry CTA needs besides its row chunks: the
// double-buffered inboxes of the one-barrier row-statistics reduction.
size_t logits_inbox_bytes(int cluster);
cudaError_t enable_sample_kernels(int max_cluster, int max_dyn);
// per kernel, element type and processor setting (sv_logits_{bf16,f32}[_proc].cu,
// sv_sample_{bf16,f32}[_proc].cu); dyn = dynamic shared memory per CTA
#define SV_KERNEL_SET(kind, P, suffix)                                                                          \
  cudaError_t enable_##kind##_kernels_##suffix(int max_cluster, int max_dyn);                                  \
  cudaError_t launch_##kind##_##suffix(const P &p, int cluster, int chunk, size_t dyn, bool vec, bool resident, \
                                       cudaStream_t stream);
SV_KERNEL_SET(logits, VerifyParams, bf16)
SV_KERNEL_SET(logits, VerifyParams, f32)
SV_KERNEL_SET(logits, VerifyParams, bf16_proc)
SV_KERNEL_SET(logits, VerifyParams, f32_proc)
SV_KERNEL_SET(sample, SampleParams, bf16)
SV_KERNEL_SET(sample, SampleParams, f32)
SV_KERNEL_SET(sample, SampleParams, bf16_proc)
SV_KERNEL_SET(sample, SampleParams, f32_proc)
#undef SV_KERNEL_SET
// the one-CTA-per-request form of the logits entry (sv_stream_{bf16,f32}.cu; enabling covers the sampler form too)
cudaError_t enable_stream_kernels_bf16();
cudaError_t enable_stream_kernels_f32();
cudaError_t launch_stream_bf16(const VerifyParams &p, cudaStream_t stream);
cudaError_t launch_stream_f32(const VerifyParams &p, cudaStream_t stream);
// with logits processors (sv_stream_{bf16,f32}_proc.cu); max_dyn bounds the dynamic shared memory
cudaError_t enable_stream_kernels_bf16_proc(int max_dyn);
cudaError_t enable_stream_kernels_f32_proc(int max_dyn);
cudaError_t launch_stream_bf16_proc(const VerifyParams &p, cudaStream_t stream);
cudaError_t launch_stream_f32_proc(const VerifyParams &p, cudaStream_t stream);
cudaError_t launch_stream_sample_bf16_proc(const SampleParams &p, cudaStream_t stream);
cudaError_t launch_stream_sample_f32_proc(const SampleParams &p, cudaStream_t stream);
// dynamic shared memory of one logits-entry CTA in that form (procs: with the row bitmaps)
size_t stream_dyn_smem(int V, bool procs);
// the one-CTA-per-row form of the draft-side sampler (the same translation units)
cudaError_t launch_stream_sample_bf16(const SampleParams &p, cudaStream_t stream);
cudaError_t launch_stream_sample_f32(const SampleParams &p, cudaStream_t stream);
cudaError_t launch_sample(const SampleParams &p, bool bf16, int cluster, int chunk, bool vec, bool resident,
                          cudaStream_t stream);
cudaError_t enable_logits_kernels(int max_cluster, int max_dyn);
// resident: both row chunks of a position in shared memory (needed by
// unaligned rows); otherwise both are read in place.
cudaError_t launch_logits(const VerifyParams &p, bool bf16, int cluster, int chunk, bool vec, bool resident,
                          cudaStream_t stream);
// Dynamic shared memory of the processor bitmaps (banned and penalised keys of a chunk).
size_t logits_bitmap_bytes(int chunk);
// Dynamic shared memory of one logits-entry CTA.
size_t logits_dyn_bytes(int cluster, int chunk, int elem_bytes, bool resident, bool bitmaps);

// Cluster size and per-CTA row chunk (elements, a multiple of 8) for the
// logits entry (chained: positions one after another) and the sampler;
// returns false if no cluster size fits the rows in shared memory.
bool choose_logits_layout(const spec_verify_ctx *ctx, int N, int V, int elem_bytes, int *cluster, int *chunk,
                          bool bitmaps, bool resident, bool chained);

void set_last_error(const char *fmt, ...);

}  // namespace sv
