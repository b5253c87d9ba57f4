// splitkv.h -- combine step of the split-KV forward pass.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

// O[row] = sum_s w_s O_s[row] / sum_s w_s, LSE[row] = m + ln sum_s w_s with
// w_s = exp(LSE_s[row] - m), m = max_s LSE_s[row]; rows = BH * N.  o_part is
// [splits][rows][d] fp32 (each O_s normalised over its split's keys),
// lse_part [splits][rows]; o is bf16 (f16 = false) or f16, lse fp32.
cudaError_t launch_splitkv_combine(const float* o_part, const float* lse_part, void* o, float* lse, int splits,
                                   long long rows, int d, bool f16, cudaStream_t stream);

}  // namespace fa
