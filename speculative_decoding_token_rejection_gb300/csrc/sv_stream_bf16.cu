// sv_stream_bf16.cu -- the one-CTA-per-request form of the logits entry (calls
// without logits processors) and the one-CTA-per-row form of the draft-side
// sampler for bf16 logits (templates in sv_stream.cuh).
#include "sv_stream.cuh"

namespace sv {

cudaError_t enable_stream_kernels_bf16() { return enable_type_stream<uint16_t, false>(0); }

cudaError_t launch_stream_bf16(const VerifyParams &p, cudaStream_t stream) {
  return launch_type_stream<uint16_t, false>(p, stream);
}

cudaError_t launch_stream_sample_bf16(const SampleParams &p, cudaStream_t stream) {
  return launch_type_stream_sample<uint16_t, false>(p, stream);
}

size_t stream_dyn_smem(int V, bool procs) { return stream_dyn_bytes(V, procs); }

}  // namespace sv
