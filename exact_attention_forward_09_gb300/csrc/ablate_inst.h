// ablate_inst.h -- the kernel variants built into libfa_ablate.so
// (include/fa_ablate.h lists what each code switches).  Variant 0, the
// shipped kernel, is not among them: fa_ablate_fwd runs it through
// libfa.so's own entry points, so no kernel is loaded twice in a process.
#pragma once

#include "attn_fwd.cuh"

// X(element type, head dimension, causal, variant)
#define FA_ABLATE_BF16_NONCAUSAL(X) X(kBF16, 128, false, 1) X(kBF16, 128, false, 2) X(kBF16, 128, false, 4) \
  X(kBF16, 128, false, 8) X(kBF16, 128, false, 16) X(kBF16, 128, false, 64) \
  X(kBF16, 128, false, 128) X(kBF16, 128, false, 256)
#define FA_ABLATE_BF16_CAUSAL(X) X(kBF16, 128, true, 1) X(kBF16, 128, true, 8) X(kBF16, 128, true, 16) \
  X(kBF16, 128, true, 256)
#define FA_ABLATE_FP8(X) X(kE4M3, 128, false, 1) X(kE4M3, 128, false, 2) X(kE4M3, 128, false, 4) \
  X(kE4M3, 128, false, 8) X(kE4M3, 128, false, 16) X(kE4M3, 128, false, 64) \
  X(kE4M3, 128, false, 128) X(kE4M3, 128, false, 256)
// head dimension 64: split softmax, separate P (tensor memory holds S, P
// and O of two Q tiles only there), polynomial exponentials, early partial
// Q K^T, direct O stores
#define FA_ABLATE_BF16_D64(X) X(kBF16, 64, false, 1) X(kBF16, 64, false, 32) X(kBF16, 64, true, 32) X(kBF16, 64, false, 64) \
  X(kBF16, 64, false, 128) X(kBF16, 64, false, 256)
