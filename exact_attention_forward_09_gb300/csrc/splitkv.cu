// splitkv.cu -- combine step of the split-KV forward pass.
//
// When a row's keys are processed in S separate runs (split-KV, for
// decode-like shapes where batch x heads x query tiles leave the GPU short of
// work: "FlashAttention-3: async pipelines on Hopper", sections "why GQA/MQA
// changes the kernel's task count" and "prefill, decode and training gain
// differently"), each run leaves O_s = sum_{j in s} e^{S_j - m_s} v_j / l_s and
// LSE_s = m_s + ln l_s.  Softmax over the union of disjoint key sets is the
// LSE-weighted mean of the parts, exactly: with m = max_s LSE_s and
// w_s = e^{LSE_s - m}, O = sum_s w_s O_s / sum_s w_s and LSE = m + ln sum_s w_s.
// A run whose rows saw no key has LSE_s = -inf and weight 0; a row with no
// visible key at all gets O = 0, LSE = -inf.
//
// One warp per row; lane l holds columns l*E .. l*E+E-1 (E = d/32).  The
// work is a read of S*d fp32 and a write of d 16-bit values per row: HBM-bound.
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "splitkv.h"

namespace fa {

template <int D, bool F16>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ o_part,
                                                              const float* __restrict__ lse_part,
                                                              void* __restrict__ o, float* __restrict__ lse,
                                                              int S, long long rows) {
  constexpr int E = D / 32;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int s = 0; s < S; ++s) m = fmaxf(m, lse_part[(long long)s * rows + row]);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;
  float wsum = 0.0f;
  if (m != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float ls = lse_part[(long long)s * rows + row];
      // a run without visible keys (LSE -inf) has weight 0 and is skipped;
      // a run's LSE is never NaN, but a NaN would be skipped the same way
      // rather than spread to the row
      if (!(ls > -INFINITY)) continue;
      const float w = expf(ls - m);
      wsum += w;
      const float* src = o_part + ((long long)s * rows + row) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float2 x = *reinterpret_cast<const float2*>(src + e);
        acc[e] = fmaf(w, x.x, acc[e]);
        acc[e + 1] = fmaf(w, x.y, acc[e + 1]);
      }
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
  uint32_t* dst = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(o) + (row * D + lane * E) * 2);
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const float a = acc[e] * inv, b = acc[e + 1] * inv;
    uint32_t pk;
    if constexpr (F16) {
      const __half2 h = __floats2half2_rn(a, b);
      pk = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
      pk = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[e / 2] = pk;
  }
  if (lane == 0) lse[row] = (m == -INFINITY) ? -INFINITY : m + logf(wsum);
}

template <int D>
static cudaError_t launch_d(const float* o_part, const float* lse_part, void* o, float* lse, int S, long long rows,
                            bool f16, cudaStream_t stream) {
  const long long blocks = (rows + 7) / 8;
  if (f16)
    splitkv_combine_kernel<D, true><<<(unsigned)blocks, 256, 0, stream>>>(o_part, lse_part, o, lse, S, rows);
  else
    splitkv_combine_kernel<D, false><<<(unsigned)blocks, 256, 0, stream>>>(o_part, lse_part, o, lse, S, rows);
  return cudaGetLastError();
}

cudaError_t launch_splitkv_combine(const float* o_part, const float* lse_part, void* o, float* lse, int splits,
                                   long long rows, int d, bool f16, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_d<64>(o_part, lse_part, o, lse, splits, rows, f16, stream);
    case 128: return launch_d<128>(o_part, lse_part, o, lse, splits, rows, f16, stream);
    case 256: return launch_d<256>(o_part, lse_part, o, lse, splits, rows, f16, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
