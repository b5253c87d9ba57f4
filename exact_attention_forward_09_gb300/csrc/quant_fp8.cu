// quant_fp8.cu -- fp32 -> FP8 E4M3 with one scale per 128-row block (or one
// per tensor), optionally after the incoherent-processing rotation
// x -> x diag(sigma) H_d / sqrt(d) ("FlashAttention-3: async pipelines on
// Hopper", sections "why block quantization beats a per-tensor scale" and
// "how incoherent processing flattens outliers"; E4M3 maximum 448 from the
// wmrh.cn FlashAttention V3 article, sec. 3.3).
//
// Optionally each row first gets a rotary position embedding (the pages
// let RoPE and the block-scale / Hadamard prep share one pass: same article,
// sections "why block quantization beats a per-tensor scale" and "how
// incoherent processing flattens outliers").  Pairs (a, b) of channels turn
// by the row's angle: a' = a*cos - b*sin, b' = a*sin + b*cos, in fp32 with
// each product rounded before the sum; the caller supplies the cos / sin
// tables and picks the pairing, (2i, 2i+1) or (i, i + d/2).
//
// One CTA per (head, 128-row block).  The block's rows are contiguous in
// memory, so one bulk copy (cp.async.bulk, completion on an mbarrier) brings
// the whole block into shared memory; then one warp per row at a time.  Each lane
// holds d/32 consecutive elements; the Walsh-Hadamard butterfly runs inside
// the lane for strides below d/32 and across lanes (shuffle) above, stride
// 1, 2, 4, ... in fp32, so every element sees the same sequence of fp32
// additions as the plain in-place butterfly.  The rotated rows stay in shared
// memory between the amax pass and the encode pass.  The 1/sqrt(d) factor is
// folded into the stored descale, so the codes are RNE(y * r) with
// r = RN(1 / s), s = amax(y) / 448 of the unnormalised rotated block y (one
// correctly rounded reciprocal per block instead of a division per element).
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "quant_fp8.h"

namespace fa {

template <int D>
__device__ __forceinline__ void rotate_row(float (&v)[D / 32], int lane, const SignBits& sg, bool rot) {
  constexpr int E = D / 32;
  if (!rot) return;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane * E + e;
    if ((sg.w[i >> 5] >> (i & 31)) & 1u) v[e] = -v[e];
  }
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (!(e & h)) {
        const float a = v[e], b = v[e + h];
        v[e] = __fadd_rn(a, b);
        v[e + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float p = __shfl_xor_sync(0xffffffffu, v[e], m);
      v[e] = (lane & m) ? __fsub_rn(p, v[e]) : __fadd_rn(v[e], p);
    }
  }
}

// n consecutive floats (16-byte aligned when n >= 4, 8-byte when n == 2)
template <int n>
__device__ __forceinline__ void load_row_f32(float (&out)[n], const float* __restrict__ p) {
  if constexpr (n % 4 == 0) {
#pragma unroll
    for (int i = 0; i < n; i += 4) {
      const float4 t = *reinterpret_cast<const float4*>(p + i);
      out[i] = t.x; out[i + 1] = t.y; out[i + 2] = t.z; out[i + 3] = t.w;
    }
  } else if constexpr (n == 2) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    out[0] = t.x; out[1] = t.y;
  } else {
#pragma unroll
    for (int i = 0; i < n; ++i) out[i] = p[i];
  }
}

// Rotary embedding of one row (lane holds channels lane*E .. lane*E+E-1);
// c, s: this row's cos / sin tables (d/2 entries each).
template <int D>
__device__ __forceinline__ void rope_row(float (&v)[D / 32], int lane, const float* __restrict__ c,
                                         const float* __restrict__ s, int mode) {
  constexpr int E = D / 32;
  if (mode == 1) {
    // pairs (2i, 2i+1), both in this lane: angles lane*E/2 .. +E/2
    float cv[E / 2], sv[E / 2];
    load_row_f32<E / 2>(cv, c + lane * (E / 2));
    load_row_f32<E / 2>(sv, s + lane * (E / 2));
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float cs = cv[e / 2], sn = sv[e / 2];
      const float a = v[e], b = v[e + 1];
      v[e] = __fsub_rn(__fmul_rn(a, cs), __fmul_rn(b, sn));
      v[e + 1] = __fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, cs));
    }
  } else if (mode == 2) {
    // pairs (i, i + D/2): lane L < 16 holds i = L*E + e, lane L + 16 its partner
    const bool first = lane < 16;
    float cv[E], sv[E];
    load_row_f32<E>(cv, c + (lane & 15) * E);
    load_row_f32<E>(sv, s + (lane & 15) * E);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float cs = cv[e], sn = sv[e];
      const float o = __shfl_xor_sync(0xffffffffu, v[e], 16);
      const float a = first ? v[e] : o, b = first ? o : v[e];
      v[e] = first ? __fsub_rn(__fmul_rn(a, cs), __fmul_rn(b, sn)) : __fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, cs));
    }
  }
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// MODE 0: per-block scale.  MODE 1: per-tensor amax into *amax_ws (atomic).
// MODE 2: per-tensor encode with the amax in *amax_ws.
// MODE 3: per-block amax stored to amax_ws[bh * nblk + blk] (no atomics).
// ROPE: rotary embedding first (pairing `rope`, 1 or 2); separate instances
// keep the plain path's code unchanged.
template <int D, int MODE, bool ROPE>
__global__ void __launch_bounds__(256) quant_e4m3_kernel(const float* __restrict__ x, uint8_t* __restrict__ x8,
                                                         float* __restrict__ descale, int N, int nblk,
                                                         SignBits sg, int rot, float rinv,
                                                         const float* __restrict__ rcos, const float* __restrict__ rsin,
                                                         int rope, float* __restrict__ amax_ws, int* err) {
  constexpr int E = D / 32;
  constexpr int ROWS = 128;
  extern __shared__ __align__(128) float ys[];  // [ROWS][D]: the block, rotated in place
  __shared__ float red[8];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int failed;
  const int blk = blockIdx.x;
  const int bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blk * ROWS;
  const int nrows = min(ROWS, N - r0);
  const size_t base = ((size_t)bh * N + r0) * D;

  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    failed = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)(nrows * D * sizeof(float));
    mbar_arrive_expect_tx(&bar, bytes);
    bulk_load(ys, x + base, bytes, &bar);
    // bounded wait for the block
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&bar, 0)) {
      if (globaltimer() - t0 > FA_WAIT_LIMIT_NS) {
        failed = 1;
        if (err) atomicExch(err, FA_DEVERR_TIMEOUT);
        break;
      }
    }
  }
  __syncthreads();
  if (failed) return;

  float amax = 0.0f;
  for (int r = warp; r < nrows; r += 8) {
    float v[E];
    float* yrow = ys + r * D + lane * E;
    if constexpr (E == 2) {
      const float2 t = *reinterpret_cast<const float2*>(yrow);
      v[0] = t.x; v[1] = t.y;
    } else {
#pragma unroll
      for (int q = 0; q < E / 4; ++q) {
        const float4 t = reinterpret_cast<const float4*>(yrow)[q];
        v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
      }
    }
    if constexpr (ROPE) rope_row<D>(v, lane, rcos + (size_t)(r0 + r) * (D / 2), rsin + (size_t)(r0 + r) * (D / 2), rope);
    rotate_row<D>(v, lane, sg, rot != 0);
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[e]));
    if constexpr (MODE == 0) {
      if (rot || ROPE) {
#pragma unroll
        for (int e = 0; e < E; ++e) yrow[e] = v[e];
      }
    } else if constexpr (MODE == 2) {
      // per-tensor encode: scale known up front
      const float am = *amax_ws;
      const float s = (am > 0.0f) ? __fdiv_rn(am, 448.0f) : 1.0f;
      const float rs = __frcp_rn(s);
      uint8_t* dst = x8 + base + (size_t)r * D + lane * E;
      if constexpr (E == 2) {
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)e4m3x2(__fmul_rn(v[0], rs), __fmul_rn(v[1], rs));
      } else {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
          const uint32_t lo = e4m3x2(__fmul_rn(v[4 * q], rs), __fmul_rn(v[4 * q + 1], rs));
          const uint32_t hi = e4m3x2(__fmul_rn(v[4 * q + 2], rs), __fmul_rn(v[4 * q + 3], rs));
          reinterpret_cast<uint32_t*>(dst)[q] = lo | (hi << 16);
        }
      }
    }
  }
  if constexpr (MODE == 2) {
    if (threadIdx.x == 0) {
      const float am = *amax_ws;
      const float s = (am > 0.0f) ? __fdiv_rn(am, 448.0f) : 1.0f;
      descale[(size_t)bh * nblk + blk] = __fmul_rn(s, rinv);
    }
    return;
  }
  // block amax
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float a = (lane < 8) ? red[lane] : 0.0f;
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
    if (lane == 0) red[0] = a;
  }
  __syncthreads();
  amax = red[0];
  if constexpr (MODE == 1) {
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<int*>(amax_ws), __float_as_int(amax));
    return;
  } else if constexpr (MODE == 3) {
    if (threadIdx.x == 0) amax_ws[(size_t)bh * nblk + blk] = amax;
    return;
  } else {
    const float s = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
    const float rs = __frcp_rn(s);
    for (int r = warp; r < nrows; r += 8) {
      uint8_t* dst = x8 + base + (size_t)r * D + lane * E;
      const float* y = ys + r * D + lane * E;
      if constexpr (E == 2) {
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)e4m3x2(__fmul_rn(y[0], rs), __fmul_rn(y[1], rs));
      } else {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
          const uint32_t lo = e4m3x2(__fmul_rn(y[4 * q], rs), __fmul_rn(y[4 * q + 1], rs));
          const uint32_t hi = e4m3x2(__fmul_rn(y[4 * q + 2], rs), __fmul_rn(y[4 * q + 3], rs));
          reinterpret_cast<uint32_t*>(dst)[q] = lo | (hi << 16);
        }
      }
    }
    if (threadIdx.x == 0) descale[(size_t)bh * nblk + blk] = __fmul_rn(s, rinv);
  }
}

// Dynamic shared memory of one block (128 rows x D fp32), set once per
// device for each instance.
template <int D, int MODE, bool ROPE>
static cudaError_t prep_quant() {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(quant_e4m3_kernel<D, MODE, ROPE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(128u * D * sizeof(float)));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  return cudaSuccess;
}

template <int D, int MODE, bool ROPE>
static cudaError_t launch_mode_r(const QuantLaunch& L, float* ws) {
  cudaError_t e = prep_quant<D, MODE, ROPE>();
  if (e != cudaSuccess) return e;
  const dim3 grid(L.nblk, L.BH, 1);
  quant_e4m3_kernel<D, MODE, ROPE><<<grid, 256, 128u * D * sizeof(float), L.stream>>>(
      L.x, L.x8, L.descale, L.N, L.nblk, L.signs, L.rot, L.rinv, L.rope_cos, L.rope_sin, L.rope, ws, L.err);
  return cudaGetLastError();
}

template <int D, int MODE>
static cudaError_t launch_mode(const QuantLaunch& L, float* ws) {
  return L.rope ? launch_mode_r<D, MODE, true>(L, ws) : launch_mode_r<D, MODE, false>(L, ws);
}

template <int D>
static cudaError_t launch_quant_d(const QuantLaunch& L) {
  if (!L.per_tensor) return launch_mode<D, 0>(L, nullptr);
  cudaError_t e = cudaMemsetAsync(L.amax_ws, 0, sizeof(float), L.stream);
  if (e != cudaSuccess) return e;
  e = launch_mode<D, 1>(L, L.amax_ws);
  if (e != cudaSuccess) return e;
  return launch_mode<D, 2>(L, L.amax_ws);
}

// Maximum of n partial maxima -> *out (one CTA).
__global__ void __launch_bounds__(1024) reduce_max_kernel(const float* __restrict__ part, int n,
                                                          float* __restrict__ out) {
  __shared__ float red[32];
  float a = 0.0f;
  for (int i = threadIdx.x; i < n; i += 1024) a = fmaxf(a, part[i]);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x < 32) {
    a = red[threadIdx.x];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
    if (threadIdx.x == 0) *out = a;
  }
}

template <int D>
static cudaError_t launch_quant_partials_d(const QuantLaunch& L, float* partials, float* amax_out) {
  cudaError_t e = launch_mode<D, 3>(L, partials);
  if (e != cudaSuccess) return e;
  reduce_max_kernel<<<1, 1024, 0, L.stream>>>(partials, L.BH * L.nblk, amax_out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_mode<D, 2>(L, amax_out);
}

cudaError_t launch_quant_per_tensor_partials(const QuantLaunch& L, float* partials, float* amax_out) {
  switch (L.d) {
    case 64: return launch_quant_partials_d<64>(L, partials, amax_out);
    case 128: return launch_quant_partials_d<128>(L, partials, amax_out);
    case 256: return launch_quant_partials_d<256>(L, partials, amax_out);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quant(const QuantLaunch& L) {
  switch (L.d) {
    case 64: return launch_quant_d<64>(L);
    case 128: return launch_quant_d<128>(L);
    case 256: return launch_quant_d<256>(L);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
