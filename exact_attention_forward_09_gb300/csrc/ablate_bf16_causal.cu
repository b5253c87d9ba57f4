// ablate_bf16_causal.cu -- kernel variants for libfa_ablate.so (own translation
// unit so that the variants compile in parallel).
#include "ablate_inst.h"

namespace fa {
#define FA_INST(E, D, C, V) template cudaError_t launch_attn<E, D, C, false, V>(const AttnLaunch&);
FA_ABLATE_BF16_CAUSAL(FA_INST)
#undef FA_INST
}  // namespace fa
