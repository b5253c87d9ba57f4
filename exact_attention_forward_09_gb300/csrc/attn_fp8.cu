// Instances of the attention forward kernel for FP8 E4M3 operands.
#include "attn_fwd.cuh"

namespace fa {
template cudaError_t launch_attn<kE4M3, 128, false>(const AttnLaunch&);
template cudaError_t launch_attn<kE4M3, 128, true>(const AttnLaunch&);
template cudaError_t launch_attn<kE4M3, 256, false>(const AttnLaunch&);
template cudaError_t launch_attn<kE4M3, 256, true>(const AttnLaunch&);
}  // namespace fa
