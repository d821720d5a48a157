// sv_stream_f32.cu -- the one-CTA-per-request form of the logits entry (calls
// without logits processors) and the one-CTA-per-row form of the draft-side
// sampler for f32 logits (templates in sv_stream.cuh).
#include "sv_stream.cuh"

namespace sv {

cudaError_t enable_stream_kernels_f32() { return enable_type_stream<float, false>(0); }

cudaError_t launch_stream_f32(const VerifyParams &p, cudaStream_t stream) {
  return launch_type_stream<float, false>(p, stream);
}

cudaError_t launch_stream_sample_f32(const SampleParams &p, cudaStream_t stream) {
  return launch_type_stream_sample<float, false>(p, stream);
}

}  // namespace sv
