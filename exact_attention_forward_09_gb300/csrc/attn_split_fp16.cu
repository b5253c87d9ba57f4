// attn_split_fp16.cu -- split-KV instances of the attention kernel (fp16).
#include "attn_fwd.cuh"

namespace fa {
template cudaError_t launch_attn<kFP16, 64, false, true>(const AttnLaunch&);
template cudaError_t launch_attn<kFP16, 64, true, true>(const AttnLaunch&);
template cudaError_t launch_attn<kFP16, 128, false, true>(const AttnLaunch&);
template cudaError_t launch_attn<kFP16, 128, true, true>(const AttnLaunch&);
template cudaError_t launch_attn<kFP16, 256, false, true>(const AttnLaunch&);
template cudaError_t launch_attn<kFP16, 256, true, true>(const AttnLaunch&);
}  // namespace fa
