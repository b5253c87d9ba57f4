// ablate_fp8.cu -- kernel variants for libfa_ablate.so (own translation
// unit so that the variants compile in parallel).
#include "ablate_inst.h"

namespace fa {
#define FA_INST(E, D, C, V) template cudaError_t launch_attn<E, D, C, false, V>(const AttnLaunch&);
FA_ABLATE_FP8(FA_INST)
#undef FA_INST
}  // namespace fa
