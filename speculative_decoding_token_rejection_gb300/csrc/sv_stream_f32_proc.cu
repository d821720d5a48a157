// sv_stream_f32_proc.cu -- the one-CTA-per-request form of the logits entry
// and the one-CTA-per-row sampler for f32 logits, calls with logits
// processors (templates in sv_stream.cuh).
#include "sv_stream.cuh"

namespace sv {

cudaError_t enable_stream_kernels_f32_proc(int max_dyn) { return enable_type_stream<float, true>(max_dyn); }

cudaError_t launch_stream_f32_proc(const VerifyParams &p, cudaStream_t stream) {
  return launch_type_stream<float, true>(p, stream);
}

cudaError_t launch_stream_sample_f32_proc(const SampleParams &p, cudaStream_t stream) {
  return launch_type_stream_sample<float, true>(p, stream);
}

}  // namespace sv
