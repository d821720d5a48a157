// sv_logits_f32_proc.cu -- the logits-entry kernels for fp32 logits, with logits processors
// (templates in sv_logits.cuh; one translation unit per kernel, element type
// and processor setting, so that they compile in parallel).
#include "sv_logits.cuh"

namespace sv {

cudaError_t enable_logits_kernels_f32_proc(int max_cluster, int max_dyn) {
  return enable_type_logits<float, true>(max_cluster, max_dyn);
}

cudaError_t launch_logits_f32_proc(const VerifyParams &p, int cluster, int chunk, size_t dyn, bool vec, bool resident,
                                   cudaStream_t stream) {
  return launch_type_logits<float, true>(p, cluster, chunk, dyn, vec, resident, stream);
}

}  // namespace sv
