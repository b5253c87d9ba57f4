// ablate_api.cu -- fa_ablate_fwd (include/fa_ablate.h): the forward with one
// design choice of the kernel switched, for timing ablations.  Argument
// checks and tensor maps are the product's (internal_prepare_fwd, from
// libfa.so, which this library links against); only the kernel instance
// differs.
#include "ablate_inst.h"
#include "fa_ablate.h"

namespace fa {
#define FA_EXTERN(E, D, C, V) extern template cudaError_t launch_attn<E, D, C, false, V>(const AttnLaunch&);
FA_ABLATE_BF16_NONCAUSAL(FA_EXTERN)
FA_ABLATE_BF16_CAUSAL(FA_EXTERN)
FA_ABLATE_FP8(FA_EXTERN)
FA_ABLATE_BF16_D64(FA_EXTERN)
#undef FA_EXTERN
}  // namespace fa

extern "C" fa_status fa_ablate_fwd(int variant, int fp8, const void* q, const void* k, const void* v, void* o,
                                   float* lse, int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                                   const float* q_descale, const float* k_descale, const float* v_descale,
                                   cudaStream_t stream) {
  if ((d != 64 && d != 128) || (fp8 != 0 && fp8 != 1)) return FA_ERR_UNSUPPORTED;
  if (variant == 0) {
    // the shipped kernel, through the product's entry points
    if (fp8) return fa_fwd_fp8(q, k, v, o, lse, B, H, N, d, causal, scale, q_descale, k_descale, v_descale, stream);
    return fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, FA_DTYPE_BF16, stream);
  }
  fa::AttnLaunch L;
  bool empty = false;
  const fa_status st = fa::internal_prepare_fwd(q, k, v, o, lse, B, H, H, N, N, d, causal, scale,
                                                fp8 ? fa::kDtypeE4M3 : FA_DTYPE_BF16, q_descale, k_descale,
                                                v_descale, stream, &L, &empty);
  if (st != FA_OK || empty) return st;
  cudaError_t e = cudaErrorInvalidValue;
  bool built = false;
#define FA_CASE(E, D, C, V)                                                                      \
  if (!built && (E == fa::kE4M3) == (fp8 != 0) && D == d && C == (causal != 0) && V == variant) { \
    e = fa::launch_attn<fa::E, D, C, false, V>(L);                                                 \
    built = true;                                                                                  \
  }
  using fa::kBF16;
  using fa::kE4M3;
  FA_ABLATE_BF16_NONCAUSAL(FA_CASE)
  FA_ABLATE_BF16_CAUSAL(FA_CASE)
  FA_ABLATE_FP8(FA_CASE)
  FA_ABLATE_BF16_D64(FA_CASE)
#undef FA_CASE
  if (!built) return FA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
