// quant_fp8.h -- launch interface of the FP8 E4M3 quantisation kernel, and
// the library internals its C-ABI entry points share with api.cu.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// d <= 256 sign bits of the random diagonal: bit i set <=> sigma_i = -1.
struct SignBits {
  uint32_t w[8];
};

struct QuantLaunch {
  CUtensorMap map;  // x as [BH, N, d] fp32: 32-float x 64-row boxes, 128-byte swizzle
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
  // the tables as [N, d/2] maps of 32-float x 128-row boxes (128-byte
  // swizzle, rows past N read as 0), for the kernels that stage them in
  // shared memory (d = 64 and 128); unused otherwise
  CUtensorMap map_cos;
  CUtensorMap map_sin;
  // test hook: the first CTA of the first launch of this call never fills
  // this slot position (-1: none), so the bounded waits on it run out
  int drop_pos;
  cudaStream_t stream;
};

cudaError_t launch_quant(const QuantLaunch& L);

// Per-tensor mode with caller-provided scratch: per-block maxima go to
// partials[BH * nblk], their maximum to *amax_out, then the encode pass runs.
// Every partial is written before it is read, so nothing needs clearing (a
// block whose load timed out writes +inf, never leaves an old value).
cudaError_t launch_quant_per_tensor_partials(const QuantLaunch& L, float* partials, float* amax_out);

// Library internals defined in api.cu.
// Once per device: architecture check, the device error word's address and
// the tensor-map encoder; then the current device and its error word.
fa_status internal_device_setup(int* dev, int** err);
// Tensor map of a contiguous fp32 [BH, N, d] tensor for the quantiser.
fa_status internal_encode_quant_map(CUtensorMap* map, const float* x, int64_t BH, int64_t N, int64_t d);
fa_status internal_encode_rope_maps(CUtensorMap* map_cos, CUtensorMap* map_sin, const float* rope_cos,
                                    const float* rope_sin, int64_t N, int64_t d);
// Consume a pending quantiser failure injection (fa_debug_inject flag 2):
// the slot position to leave unfilled, or -1.
int internal_take_quant_inject();

}  // namespace fa
