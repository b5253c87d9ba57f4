// Instances of the attention forward kernel for bf16 operands.
#include "attn_fwd.cuh"

namespace fa {
template cudaError_t launch_attn<kBF16, 64, false, false>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 64, true, false>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 128, false, false>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 128, true, false>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 256, false, false>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 256, true, false>(const AttnLaunch&);
}  // namespace fa
