// sv_stream_bf16_proc.cu -- the one-CTA-per-request form of the logits entry
// and the one-CTA-per-row sampler for bf16 logits, calls with logits
// processors (templates in sv_stream.cuh).
#include "sv_stream.cuh"

namespace sv {

cudaError_t enable_stream_kernels_bf16_proc(int max_dyn) { return enable_type_stream<uint16_t, true>(max_dyn); }

cudaError_t launch_stream_bf16_proc(const VerifyParams &p, cudaStream_t stream) {
  return launch_type_stream<uint16_t, true>(p, stream);
}

cudaError_t launch_stream_sample_bf16_proc(const SampleParams &p, cudaStream_t stream) {
  return launch_type_stream_sample<uint16_t, true>(p, stream);
}

}  // namespace sv
