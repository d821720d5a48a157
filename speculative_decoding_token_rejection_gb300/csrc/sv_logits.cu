// sv_logits.cu -- shared-memory sizes of the logits-entry and sampler kernels,
// and the dispatch of their launches to the per-type and per-processor
// translation units (sv_logits_{bf16,f32}[_proc].cu,
// sv_sample_{bf16,f32}[_proc].cu; the kernels are in sv_logits.cuh).
#include "sv_logits.cuh"

namespace sv {

size_t logits_static_smem() { return sizeof(LogitsSmem); }
int logits_reg_group_chunk() { return kRegGroupChunk; }
size_t logits_inbox_bytes(int cluster) { return 2 * static_cast<size_t>(cluster) * sizeof(Inbox); }
size_t logits_bitmap_bytes(int chunk) { return ((2 * static_cast<size_t>((chunk + 31) / 32) * 4) + 15) & ~size_t{15}; }
size_t logits_dyn_bytes(int cluster, int chunk, int elem_bytes, bool resident, bool bitmaps) {
  return (resident ? 2 : 0) * static_cast<size_t>(chunk) * elem_bytes + logits_inbox_bytes(cluster) +
         (bitmaps ? logits_bitmap_bytes(chunk) : 0);
}

cudaError_t enable_logits_kernels(int max_cluster, int max_dyn) {
  cudaError_t e;
  if ((e = enable_logits_kernels_bf16(max_cluster, max_dyn)) != cudaSuccess) return e;
  if ((e = enable_logits_kernels_f32(max_cluster, max_dyn)) != cudaSuccess) return e;
  if ((e = enable_logits_kernels_bf16_proc(max_cluster, max_dyn)) != cudaSuccess) return e;
  return enable_logits_kernels_f32_proc(max_cluster, max_dyn);
}

cudaError_t enable_sample_kernels(int max_cluster, int max_dyn) {
  cudaError_t e;
  if ((e = enable_sample_kernels_bf16(max_cluster, max_dyn)) != cudaSuccess) return e;
  if ((e = enable_sample_kernels_f32(max_cluster, max_dyn)) != cudaSuccess) return e;
  if ((e = enable_sample_kernels_bf16_proc(max_cluster, max_dyn)) != cudaSuccess) return e;
  return enable_sample_kernels_f32_proc(max_cluster, max_dyn);
}

cudaError_t launch_sample(const SampleParams &p, bool bf16, int cluster, int chunk, bool vec, bool resident,
                          cudaStream_t stream) {
  resident = resident || !vec;
  const bool procs = p.rep_penalty || p.ban_cu;
  const size_t dyn = (resident ? static_cast<size_t>(chunk) * (bf16 ? 2 : 4) : 0) + logits_inbox_bytes(cluster) +
                     (procs ? logits_bitmap_bytes(chunk) : 0);
  if (procs)
    return bf16 ? launch_sample_bf16_proc(p, cluster, chunk, dyn, vec, resident, stream)
                : launch_sample_f32_proc(p, cluster, chunk, dyn, vec, resident, stream);
  return bf16 ? launch_sample_bf16(p, cluster, chunk, dyn, vec, resident, stream)
              : launch_sample_f32(p, cluster, chunk, dyn, vec, resident, stream);
}

cudaError_t launch_logits(const VerifyParams &p, bool bf16, int cluster, int chunk, bool vec, bool resident,
                          cudaStream_t stream) {
  resident = resident || !vec;
  const bool procs = p.rep_penalty || p.ban_cu;
  const size_t dyn = logits_dyn_bytes(cluster, chunk, bf16 ? 2 : 4, resident, procs);
  if (procs)
    return bf16 ? launch_logits_bf16_proc(p, cluster, chunk, dyn, vec, resident, stream)
                : launch_logits_f32_proc(p, cluster, chunk, dyn, vec, resident, stream);
  return bf16 ? launch_logits_bf16(p, cluster, chunk, dyn, vec, resident, stream)
              : launch_logits_f32(p, cluster, chunk, dyn, vec, resident, stream);
}

}  // namespace sv
