// attn_bwd.h -- launch interface of the attention backward kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

struct BwdParams {
  float* dq_acc;       // [BHq, Nq, D] fp32, zeroed by the preprocessing kernel (added to through tm dq_acc)
  void* dk;            // [BHkv, Nk, D] bf16 / f16
  void* dv;            // [BHkv, Nk, D]
  // [BHq, nrec, 2, 64]: per 64-row record, -LSE_i * log2(e) (-inf for a
  // row with no key or past Nq) then -D_i (0 past Nq)
  const float* vecs;
  int nrec;            // records per query head (whole kernel steps)
  int* err;            // device error word
  int Nq, Nk;          // query rows / keys per head
  int Hq, Hkv;         // heads (Hq % Hkv == 0)
  int BHkv;            // batch x key/value heads
  float scale_log2;    // scale * log2(e)
  float scale;         // dK = scale * dS^T Q
  int drop_step;       // test hook: step whose Q/dO stage CTA 0 never fills (-1: none)
};

struct BwdLaunch {
  CUtensorMap q, dout;  // [BHq, Nq, D], 64-row boxes
  CUtensorMap k, v;     // [BHkv, Nk, D], 128-row boxes
  CUtensorMap dq_acc;   // fp32 [BHq, Nq, D], 32-column x step-row boxes, 128-byte swizzle
  CUtensorMap dk, dv;   // [BHkv, Nk, D], 128-row boxes (epilogue stores)
  BwdParams prm;
  cudaStream_t stream;
};

// ELEM: 0 bf16, 1 f16 (the forward's element kinds)
template <int ELEM, int D, bool CAUSAL>
cudaError_t launch_attn_bwd(const BwdLaunch& L);

// Records of -LSE_i * log2(e) and -D_i (D_i = dO_i . O_i) for every query
// row, padded to nrec 64-row records per head, and dq_acc := 0.
cudaError_t launch_bwd_prep(const void* o, const void* dout, const float* lse, float* vecs, float* dq_acc,
                            long long bhq, int nq, int nrec, int d, bool f16, cudaStream_t stream);

// Query rows per kernel step for head dimension d, and the records per
// query head the kernel reads (whole steps).
int bwd_step_rows(int d);
long long bwd_records_per_head(long long nq, int d);

// dq = RN(scale * dq_acc) in the element type.
cudaError_t launch_bwd_dq_convert(const float* dq_acc, void* dq, float scale, long long elems, bool f16,
                                  cudaStream_t stream);

// Zero `bytes` bytes (a multiple of 16, 16-byte aligned).
cudaError_t launch_zero_fill(void* p, long long bytes, cudaStream_t stream);

}  // namespace fa
