// sv_sample_bf16.cu -- the draft-side sampler kernels for bf16 logits, without logits processors
// (templates in sv_logits.cuh; one translation unit per kernel, element type
// and processor setting, so that they compile in parallel).
#include "sv_logits.cuh"

namespace sv {

cudaError_t enable_sample_kernels_bf16(int max_cluster, int max_dyn) {
  return enable_type_sample<uint16_t, false>(max_cluster, max_dyn);
}

cudaError_t launch_sample_bf16(const SampleParams &p, int cluster, int chunk, size_t dyn, bool vec, bool resident,
                               cudaStream_t stream) {
  return launch_type_sample<uint16_t, false>(p, cluster, chunk, dyn, vec, resident, stream);
}

}  // namespace sv
