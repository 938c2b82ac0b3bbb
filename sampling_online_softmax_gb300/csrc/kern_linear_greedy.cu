// kern_linear_greedy.cu -- spec_verify_kernel in mode kLinearGreedy, for fp32 and bf16 logits
// (one translation unit per mode, so the modes compile in parallel).
#include "launch.cuh"

namespace spec {
template spec_status launch<4, kLinearGreedy>(const Params &, bool, cudaStream_t);
template spec_status launch<2, kLinearGreedy>(const Params &, bool, cudaStream_t);
}  // namespace spec
