// quant_fp8.h -- launch interface of the FP8 E4M3 quantisation kernel.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

// d <= 256 sign bits of the random diagonal: bit i set <=> sigma_i = -1.
struct SignBits {
  uint32_t w[8];
};

struct QuantLaunch {
  const float* x;   // [BH, N, d] fp32
  uint8_t* x8;      // [BH, N, d] E4M3 codes
  float* descale;   // [BH, nblk]
  float* amax_ws;   // per-tensor mode: one float of scratch
  int* err;         // device error word (may be null)
  int BH, N, d, nblk;
  int per_tensor;
  int rot;
  float rinv;       // 1/sqrt(d) as fp32 when rotating, else 1
  SignBits signs;
  // rotary position embedding applied to each row before the rotation:
  // 0 off, 1 pairs (2i, 2i+1), 2 pairs (i, i + d/2); angle tables
  // [N, d/2] fp32 (row n uses row n of each table)
  const float* rope_cos;
  const float* rope_sin;
  int rope;
  cudaStream_t stream;
};

cudaError_t launch_quant(const QuantLaunch& L);

// Per-tensor mode with caller-provided scratch: per-block maxima go to
// partials[BH * nblk], their maximum to *amax_out, then the encode pass runs.
// Every partial is written before it is read, so nothing needs clearing.
cudaError_t launch_quant_per_tensor_partials(const QuantLaunch& L, float* partials, float* amax_out);

}  // namespace fa
