// Instances of the attention forward kernel for FP8 E4M3 operands.
#include "attn_fwd.cuh"

namespace fa {
template cudaError_t launch_attn<kE4M3, 128, false, false>(const AttnLaunch&);
template cudaError_t launch_attn<kE4M3, 128, true, false>(const AttnLaunch&);
template cudaError_t launch_attn<kE4M3, 256, false, false>(const AttnLaunch&);
template cudaError_t launch_attn<kE4M3, 256, true, false>(const AttnLaunch&);
}  // namespace fa
