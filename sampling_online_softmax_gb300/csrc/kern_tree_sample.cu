// kern_tree_sample.cu -- spec_verify_kernel in mode kTreeSample, for fp32 and bf16 logits
// (one translation unit per mode, so the modes compile in parallel).
#include "launch.cuh"

namespace spec {
template spec_status launch<4, kTreeSample>(const Params &, bool, cudaStream_t);
template spec_status launch<2, kTreeSample>(const Params &, bool, cudaStream_t);
}  // namespace spec
