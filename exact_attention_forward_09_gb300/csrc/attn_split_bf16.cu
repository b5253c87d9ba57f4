// attn_split_bf16.cu -- split-KV instances of the attention kernel (bf16).
#include "attn_fwd.cuh"

namespace fa {
template cudaError_t launch_attn<kBF16, 64, false, true>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 64, true, true>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 128, false, true>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 128, true, true>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 256, false, true>(const AttnLaunch&);
template cudaError_t launch_attn<kBF16, 256, true, true>(const AttnLaunch&);
}  // namespace fa
