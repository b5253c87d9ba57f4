// api.cu -- the C ABI of libfa.so (declared in include/fa.h): argument checks,
// TMA descriptor encoding, kernel selection and launch on the caller's
// stream.  No device memory is allocated here; the only device state is the
// library's error word (a __device__ int per device).
#include <cmath>
#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "attn_fwd.cuh"
#include "splitkv.h"
#include "quant_fp8.h"
#include "attn_bwd.h"

// The attention kernels are instantiated in their own translation units
// (attn_bf16.cu, attn_fp16.cu, attn_fp8.cu, attn_split_*.cu), compiled in
// parallel; this one only calls them.
namespace fa {
#define FA_EXTERN_ATTN(E, D, C, S) extern template cudaError_t launch_attn<E, D, C, S, 0>(const AttnLaunch&);
#define FA_EXTERN_ATTN_DC(E, S) \
  FA_EXTERN_ATTN(E, 64, false, S) FA_EXTERN_ATTN(E, 64, true, S) FA_EXTERN_ATTN(E, 128, false, S) \
  FA_EXTERN_ATTN(E, 128, true, S) FA_EXTERN_ATTN(E, 256, false, S) FA_EXTERN_ATTN(E, 256, true, S)
FA_EXTERN_ATTN_DC(kBF16, false)
FA_EXTERN_ATTN_DC(kFP16, false)
FA_EXTERN_ATTN_DC(kBF16, true)
FA_EXTERN_ATTN_DC(kFP16, true)
FA_EXTERN_ATTN(kE4M3, 128, false, false)
FA_EXTERN_ATTN(kE4M3, 128, true, false)
FA_EXTERN_ATTN(kE4M3, 256, false, false)
FA_EXTERN_ATTN(kE4M3, 256, true, false)
#undef FA_EXTERN_ATTN_DC
#undef FA_EXTERN_ATTN
}  // namespace fa


namespace {

__device__ int g_fa_device_error;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool checked = false;
  bool supported = false;
  int* err_word = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Streams and events of the host-buffer path (fa_fwd_host), created once
// per device on first use: two host->device copy streams, two compute
// streams (consecutive chunks alternate, so that a chunk's kernel can start
// on the SMs the previous chunk's last units leave free) and a
// device->host copy stream, fanned out from and joined back into the
// caller's stream with events on every call.
constexpr int kHostChunks = 16;
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d[2] = {nullptr, nullptr};
  cudaStream_t comp[2] = {nullptr, nullptr};
  cudaStream_t d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t copied[kHostChunks] = {};
  cudaEvent_t computed[kHostChunks] = {};
  cudaEvent_t done[5] = {};
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDevices];

// Streams of fa_quant_fp8_qkv, created once per device on first use: the
// three quantisations run one per stream, fanned out from and joined back
// into the caller's stream, so that each launch's CTAs start on the SMs the
// others' last CTAs leave free (one CTA per SM each).
struct QkvPipe {
  bool ready = false;
  cudaStream_t s[3] = {nullptr, nullptr, nullptr};
  cudaEvent_t start = nullptr;
  cudaEvent_t done[3] = {};
};
std::mutex g_qkv_mu;
QkvPipe g_qkv[kMaxDevices];
std::atomic<int> g_inject{0};  // one-shot failure injection for the next attention launch
std::atomic<int> g_inject_quant{0};  // ... and for the next quantiser call
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

fa_status device_setup(int* dev_out, int** err_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_fa_device_error) != cudaSuccess) return FA_ERR_CUDA;
      st.err_word = static_cast<int*>(p);
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FA_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.checked = true;
  }
  if (!st.supported) return FA_ERR_UNSUPPORTED;
  *dev_out = dev;
  *err_out = st.err_word;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D tiled map over a contiguous [BH, N, d] tensor: box = (128-byte row
// chunk) x box_rows rows x 1 head, 128-byte swizzle, out-of-range rows read
// as 0.
fa_status encode_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int64_t BH,
                     int64_t N, int64_t d, uint32_t box_rows = 128) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)(d * elem_bytes), (cuuint64_t)(N * d * elem_bytes)};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), box_rows, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

fa_status check_common(const void* q, const void* k, const void* v, const void* o, const float* lse, int64_t B,
                       int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, float scale, bool* empty) {
  if (B < 0 || Hq < 0 || Hkv < 0 || Nq < 0 || Nk < 0 || d < 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  *empty = (B == 0 || Hq == 0 || Nq == 0);
  if (*empty) return FA_OK;
  if (Hkv == 0 || Hq % Hkv != 0 || Nk == 0) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  // index ranges used by the kernels: a 1-D grid of B*Hq*ceil(Nq/256) blocks
  // (at most B*Hq*ceil(Nq/128) for one Q tile per block) and int row indices
  const int64_t lim = 0x7fffffffLL - 256;
  if (Nq > lim || Nk > lim || B * Hq > 0x7fffffffLL || B * Hq * ((Nq + 127) / 128) > 0x7fffffffLL)
    return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

template <int ELEM, bool SPLIT = false>
fa_status dispatch(const fa::AttnLaunch& L, int64_t d, int causal) {
  cudaError_t e = cudaErrorInvalidValue;
  if (d == 64) {
    if constexpr (ELEM == fa::kE4M3) return FA_ERR_UNSUPPORTED;
    else e = causal ? fa::launch_attn<ELEM, 64, true, SPLIT>(L) : fa::launch_attn<ELEM, 64, false, SPLIT>(L);
  } else if (d == 128) {
    e = causal ? fa::launch_attn<ELEM, 128, true, SPLIT>(L) : fa::launch_attn<ELEM, 128, false, SPLIT>(L);
  } else if (d == 256) {
    e = causal ? fa::launch_attn<ELEM, 256, true, SPLIT>(L) : fa::launch_attn<ELEM, 256, false, SPLIT>(L);
  } else {
    return FA_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Split-KV plan: the query heads of a key/value group are packed into one
// head of g * Nq rows (contiguous in [B, Hq, Nq, d]), and each row's key
// tiles are cut into S runs of T tiles.  Chosen S (when 0 is asked): about
// eight units per SM -- the runs are memory-bound with little fixed cost, and
// several waves keep the last one from leaving most SMs idle -- but at least
// 8 key tiles per run.  Workspace: partial O [S][B*Hkv][g*Nq][d] fp32, then
// partial LSE [S][B*Hkv][g*Nq] fp32 (256-byte aligned start).
struct SplitPlan {
  int64_t BHp, Np;
  int S, T;
  size_t o_bytes, ws_bytes;
};

fa_status splitkv_plan(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int num_splits,
                       int sms, SplitPlan* p) {
  p->BHp = B * Hkv;
  p->Np = (Hq / Hkv) * Nq;
  if (p->Np > 0x7fffffffLL - 256) return FA_ERR_UNSUPPORTED;
  const int64_t rows_per_unit = d <= 128 ? 256 : 128;
  const int64_t base = p->BHp * ((p->Np + rows_per_unit - 1) / rows_per_unit);
  const int64_t nkv = (Nk + 127) / 128;
  int64_t S = num_splits;
  if (S == 0) {
    S = (8 * (int64_t)sms + base - 1) / base;
    const int64_t most = (nkv + 7) / 8;  // at least 8 key tiles per run
    if (S > most) S = most;
  }
  if (S > nkv) S = nkv;
  if (S > 1024) S = 1024;
  if (S < 1) S = 1;
  const int64_t T = (nkv + S - 1) / S;
  S = (nkv + T - 1) / T;  // no empty run
  if (base * S > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if ((p->BHp * p->Np + 7) / 8 > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;  // combine: one block per 8 rows
  p->S = (int)S;
  p->T = (int)T;
  p->o_bytes = S > 1 ? (((size_t)S * p->BHp * p->Np * d * 4 + 255) / 256) * 256 : 0;
  p->ws_bytes = S > 1 ? p->o_bytes + (size_t)S * p->BHp * p->Np * 4 : 0;
  return FA_OK;
}

int device_sm_count(int dev) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
  return sms;
}

}  // namespace

namespace fa {
fa_status internal_prepare_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                               int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale,
                               int dtype, const float* q_descale, const float* k_descale, const float* v_descale,
                               cudaStream_t stream, AttnLaunch* out, bool* empty) {
  const bool fp8 = (dtype == kDtypeE4M3);
  if (!fp8 && dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  fa_status st = check_common(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, empty);
  if (st != FA_OK || *empty) return st;
  if (fp8) {
    if (d == 64) return FA_ERR_UNSUPPORTED;  // FP8 rows must span the 128-byte swizzle
    if (!q_descale || !k_descale || !v_descale) return FA_ERR_INVALID_ARG;
    if (((uintptr_t)k_descale & 3u) || ((uintptr_t)v_descale & 3u) || ((uintptr_t)q_descale & 3u))
      return FA_ERR_INVALID_ARG;
  }
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;

  AttnLaunch& L = *out;
  std::memset(&L, 0, sizeof(L));
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : (dtype == FA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  const int es = fp8 ? 1 : 2;
  if ((st = encode_map(&L.q, q, dt, es, B * Hq, Nq, d)) != FA_OK) return st;
  if ((st = encode_map(&L.k, k, dt, es, B * Hkv, Nk, d)) != FA_OK) return st;
  if ((st = encode_map(&L.v, v, dt, es, B * Hkv, Nk, d)) != FA_OK) return st;
  // O (bf16 for the FP8 path) in 64-column x 32-row boxes: one per softmax warp
  const CUtensorMapDataType dt_o = fp8 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : dt;
  if ((st = encode_map(&L.o, o, dt_o, 2, B * Hq, Nq, d, 32)) != FA_OK) return st;
  L.prm.o = o;
  L.prm.o_vec32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  L.prm.lse = lse;
  L.prm.q_ds = q_descale;
  L.prm.k_ds = k_descale;
  L.prm.v_ds = v_descale;
  L.prm.err = err;
  L.prm.N = (int)Nq;
  L.prm.Nk = (int)Nk;
  L.prm.Hq = (int)Hq;
  L.prm.Hkv = (int)Hkv;
  L.prm.nblk = (int)((Nq + 127) / 128);
  L.prm.nblk_k = (int)((Nk + 127) / 128);
  L.prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  L.BH = (int)(B * Hq);
  L.prm.BH = L.BH;
  L.prm.drop_pos = (g_inject.exchange(0) & 1) ? 3 : -1;
  L.prm.q_period = (int)Nq;
  L.prm.splits = 1;
  L.prm.split_tiles = (int)((Nk + 127) / 128);
  L.stream = stream;
  return FA_OK;
}

// the two ways the forward kernels compute an exponential of P, one pair
// per thread (fa_debug_exp2)
template <int METHOD>
__global__ void exp2_eval_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  const int64_t i = 2 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float2 a = make_float2(x[i], (i + 1 < n) ? x[i + 1] : 0.0f);
  float2 r;
  if constexpr (METHOD == 0) r = make_float2(ex2(a.x), ex2(a.y));
  else r = ex2_poly2<METHOD>(a);
  y[i] = r.x;
  if (i + 1 < n) y[i + 1] = r.y;
}
}  // namespace fa

extern "C" {

fa_status fa_splitkv_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                                     int num_splits, size_t* bytes) {
  if (!bytes) return FA_ERR_INVALID_ARG;
  *bytes = 0;
  if (B < 0 || Hq < 0 || Hkv < 0 || Nq < 0 || Nk < 0 || d < 0 || num_splits < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (B == 0 || Hq == 0 || Nq == 0) return FA_OK;
  if (Hkv == 0 || Hq % Hkv != 0 || Nk == 0) return FA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  SplitPlan p;
  const fa_status st = splitkv_plan(B, Hq, Hkv, Nq, Nk, d, num_splits, device_sm_count(dev), &p);
  if (st == FA_OK) *bytes = p.ws_bytes;
  return st;
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t Hq,
                         int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale, int dtype,
                         int num_splits, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  bool empty = false;
  fa_status st = check_common(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, &empty);
  if (st != FA_OK || empty) return st;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  SplitPlan p;
  if ((st = splitkv_plan(B, Hq, Hkv, Nq, Nk, d, num_splits, device_sm_count(dev), &p)) != FA_OK) return st;
  if (p.S > 1 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < p.ws_bytes))
    return FA_ERR_INVALID_ARG;

  fa::AttnLaunch L;
  std::memset(&L, 0, sizeof(L));
  const CUtensorMapDataType dt =
      dtype == FA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  // packed: head (b, kv head) with g * Nq rows; K/V heads map one to one
  if ((st = encode_map(&L.q, q, dt, 2, p.BHp, p.Np, d)) != FA_OK) return st;
  if ((st = encode_map(&L.k, k, dt, 2, p.BHp, Nk, d)) != FA_OK) return st;
  if ((st = encode_map(&L.v, v, dt, 2, p.BHp, Nk, d)) != FA_OK) return st;
  if ((st = encode_map(&L.o, o, dt, 2, p.BHp, p.Np, d, 32)) != FA_OK) return st;
  L.prm.o = o;
  L.prm.o_vec32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  L.prm.lse = lse;
  L.prm.err = err;
  L.prm.N = (int)p.Np;
  L.prm.Nk = (int)Nk;
  L.prm.Hq = 1;
  L.prm.Hkv = 1;
  L.prm.nblk = (int)((p.Np + 127) / 128);
  L.prm.nblk_k = (int)((Nk + 127) / 128);
  L.prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  L.BH = (int)p.BHp;
  L.prm.BH = L.BH;
  L.prm.drop_pos = -1;
  L.prm.q_period = (int)Nq;
  L.prm.splits = p.S;
  L.prm.split_tiles = p.T;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = p.S > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + p.o_bytes) : nullptr;
  L.prm.o_part = p.S > 1 ? o_part : nullptr;
  L.prm.lse_part = lse_part;
  L.stream = stream;
  // the split-KV instance (packed rows; partial results when S > 1)
  st = dtype == FA_DTYPE_BF16 ? dispatch<fa::kBF16, true>(L, d, causal) : dispatch<fa::kFP16, true>(L, d, causal);
  if (st != FA_OK || p.S == 1) return st;
  return fa::launch_splitkv_combine(o_part, lse_part, o, lse, p.S, (long long)(p.BHp * p.Np), (int)d,
                                    dtype == FA_DTYPE_FP16, stream) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t Hq,
                     int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale, int dtype,
                     cudaStream_t stream) {
  fa::AttnLaunch L;
  bool empty = false;
  const fa_status st = fa::internal_prepare_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, dtype,
                                                nullptr, nullptr, nullptr, stream, &L, &empty);
  if (st != FA_OK || empty) return st;
  return dtype == FA_DTYPE_BF16 ? dispatch<fa::kBF16>(L, d, causal) : dispatch<fa::kFP16>(L, d, causal);
}

fa_status fa_fwd_host_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                                     size_t* bytes) {
  if (!bytes) return FA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 0 || Hkv < 0 || Nq < 0 || Nk < 0 || d < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (Hkv == 0 || Hq % Hkv != 0) {
    if (B == 0 || Hq == 0) {
      *bytes = 0;
      return FA_OK;
    }
    return FA_ERR_INVALID_ARG;
  }
  auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t qo = B * Hq * Nq * d * 2, kv = B * Hkv * Nk * d * 2;
  *bytes = (size_t)(2 * up(qo) + 2 * up(kv) + up(B * Hq * Nq * 4));  // q, o, k, v, lse
  return FA_OK;
}

fa_status fa_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                      int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale,
                      int dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  size_t need = 0;
  fa_status st = fa_fwd_host_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, &need);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (B == 0 || Hq == 0 || Nq == 0) return FA_OK;
  if (Nk == 0) return FA_ERR_INVALID_ARG;
  if (!q_host || !k_host || !v_host || !o_host || !lse_host) return FA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
    return FA_ERR_INVALID_ARG;
  const int64_t lim = 0x7fffffffLL - 256;
  if (Nq > lim || Nk > lim || B * Hq > 0x7fffffffLL || B * Hq * ((Nq + 127) / 128) > 0x7fffffffLL)
    return FA_ERR_UNSUPPORTED;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;

  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe& P = g_pipe[dev];
  if (!P.ready) {
    bool ok = true;
    for (auto* sp : {&P.h2d[0], &P.h2d[1], &P.comp[0], &P.comp[1], &P.d2h})
      ok = ok && cudaStreamCreateWithFlags(sp, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&P.start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < kHostChunks; ++i) {
      ok = ok && cudaEventCreateWithFlags(&P.copied[i], cudaEventDisableTiming) == cudaSuccess;
      ok = ok && cudaEventCreateWithFlags(&P.computed[i], cudaEventDisableTiming) == cudaSuccess;
    }
    for (int i = 0; i < 5; ++i) ok = ok && cudaEventCreateWithFlags(&P.done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      // release what was made, so that a later call starts again from nothing
      for (cudaStream_t* sp : {&P.h2d[0], &P.h2d[1], &P.comp[0], &P.comp[1], &P.d2h}) {
        if (*sp) cudaStreamDestroy(*sp);
        *sp = nullptr;
      }
      for (cudaEvent_t* ep : {&P.start}) {
        if (*ep) cudaEventDestroy(*ep);
        *ep = nullptr;
      }
      for (int i = 0; i < kHostChunks; ++i) {
        if (P.copied[i]) cudaEventDestroy(P.copied[i]);
        if (P.computed[i]) cudaEventDestroy(P.computed[i]);
        P.copied[i] = P.computed[i] = nullptr;
      }
      for (int i = 0; i < 5; ++i) {
        if (P.done[i]) cudaEventDestroy(P.done[i]);
        P.done[i] = nullptr;
      }
      return FA_ERR_CUDA;
    }
    P.ready = true;
  }
  // device copies inside the workspace: q, o, k, v, lse
  auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t g = Hq / Hkv;
  const int64_t q_row = g * Nq * d * 2;   // bytes of one key/value head's query rows (= its o rows)
  const int64_t kv_row = Nk * d * 2;      // bytes of one key/value head's K (or V)
  const int64_t BHkv = B * Hkv;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  uint8_t* qd = w;
  uint8_t* od = qd + up(BHkv * q_row);
  uint8_t* kd = od + up(BHkv * q_row);
  uint8_t* vd = kd + up(BHkv * kv_row);
  float* ld = reinterpret_cast<float*>(vd + up(BHkv * kv_row));
  const uint8_t* qh = static_cast<const uint8_t*>(q_host);
  const uint8_t* kh = static_cast<const uint8_t*>(k_host);
  const uint8_t* vh = static_cast<const uint8_t*>(v_host);
  uint8_t* oh = static_cast<uint8_t*>(o_host);

  // fan out from the caller's stream
  if (cudaEventRecord(P.start, stream) != cudaSuccess) return FA_ERR_CUDA;
  fa_status result = FA_OK;
  for (cudaStream_t s : {P.h2d[0], P.h2d[1], P.comp[0], P.comp[1], P.d2h})
    if (cudaStreamWaitEvent(s, P.start, 0) != cudaSuccess) result = FA_ERR_CUDA;
  // chunks of whole key/value heads (each with its g query heads): the
  // copies of chunk c+1 run while chunk c computes and chunk c-1 copies back
  // chunk boundaries at multiples of `step` key/value heads, so that every
  // chunk's LSE rows start 16-byte aligned (g * Nq * step rows of 4 bytes)
  const int64_t rows = g * Nq;
  const int64_t step = (rows % 4 == 0) ? 1 : (rows % 2 == 0) ? 2 : 4;
  // 4 chunks, or up to 16 when every chunk still holds a wave of units or
  // more: the first chunk's copy in and the last one's copy out are what the
  // overlap leaves exposed
  const int64_t units = BHkv * ((g * Nq + 255) / 256);
  int64_t nch = units / (int64_t)device_sm_count(dev);
  nch = nch < 4 ? 4 : nch > kHostChunks ? kHostChunks : nch;
  if (nch > BHkv) nch = BHkv;
  for (int64_t c = 0; c < nch && result == FA_OK; ++c) {
    const int64_t j0 = (BHkv * c / nch) / step * step;
    const int64_t j1 = (c + 1 == nch) ? BHkv : (BHkv * (c + 1) / nch) / step * step;
    const int64_t nj = j1 - j0;
    if (nj <= 0) continue;
    cudaStream_t hs = P.h2d[c & 1];
    if (cudaMemcpyAsync(qd + j0 * q_row, qh + j0 * q_row, (size_t)(nj * q_row), cudaMemcpyHostToDevice, hs) !=
            cudaSuccess ||
        cudaMemcpyAsync(kd + j0 * kv_row, kh + j0 * kv_row, (size_t)(nj * kv_row), cudaMemcpyHostToDevice, hs) !=
            cudaSuccess ||
        cudaMemcpyAsync(vd + j0 * kv_row, vh + j0 * kv_row, (size_t)(nj * kv_row), cudaMemcpyHostToDevice, hs) !=
            cudaSuccess ||
        cudaEventRecord(P.copied[c], hs) != cudaSuccess ||
        cudaStreamWaitEvent(P.comp[c & 1], P.copied[c], 0) != cudaSuccess) {
      result = FA_ERR_CUDA;
      break;
    }
    // the chunk as nj batches of one key/value head and its g query heads
    st = fa_fwd_gqa(qd + j0 * q_row, kd + j0 * kv_row, vd + j0 * kv_row, od + j0 * q_row, ld + j0 * g * Nq, nj, g,
                    1, Nq, Nk, d, causal, scale, dtype, P.comp[c & 1]);
    if (st != FA_OK) {
      result = st;
      break;
    }
    if (cudaEventRecord(P.computed[c], P.comp[c & 1]) != cudaSuccess ||
        cudaStreamWaitEvent(P.d2h, P.computed[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(oh + j0 * q_row, od + j0 * q_row, (size_t)(nj * q_row), cudaMemcpyDeviceToHost, P.d2h) !=
            cudaSuccess ||
        cudaMemcpyAsync(lse_host + j0 * g * Nq, ld + j0 * g * Nq, (size_t)(nj * g * Nq * 4), cudaMemcpyDeviceToHost,
                        P.d2h) != cudaSuccess) {
      result = FA_ERR_CUDA;
      break;
    }
  }
  // join back into the caller's stream -- after an error too, so that work
  // the caller enqueues next never runs ahead of copies that still read or
  // write its host buffers
  cudaStream_t all[5] = {P.h2d[0], P.h2d[1], P.comp[0], P.comp[1], P.d2h};
  for (int i = 0; i < 5; ++i)
    if (cudaEventRecord(P.done[i], all[i]) != cudaSuccess || cudaStreamWaitEvent(stream, P.done[i], 0) != cudaSuccess)
      if (result == FA_OK) result = FA_ERR_CUDA;
  return result;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H, int64_t N,
                 int64_t d, int causal, float scale, int dtype, cudaStream_t stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, N, d, causal, scale, dtype, stream);
}

fa_status fa_fwd_fp8_gqa(const void* q8, const void* k8, const void* v8, void* o, float* lse, int64_t B, int64_t Hq,
                         int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale,
                         const float* q_descale, const float* k_descale, const float* v_descale,
                         cudaStream_t stream) {
  fa::AttnLaunch L;
  bool empty = false;
  const fa_status st = fa::internal_prepare_fwd(q8, k8, v8, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale,
                                                fa::kDtypeE4M3, q_descale, k_descale, v_descale, stream, &L, &empty);
  if (st != FA_OK || empty) return st;
  return dispatch<fa::kE4M3>(L, d, causal);
}

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* v8, void* o, float* lse, int64_t B, int64_t H,
                     int64_t N, int64_t d, int causal, float scale, const float* q_descale, const float* k_descale,
                     const float* v_descale, cudaStream_t stream) {
  return fa_fwd_fp8_gqa(q8, k8, v8, o, lse, B, H, H, N, N, d, causal, scale, q_descale, k_descale, v_descale,
                        stream);
}

namespace {
// Argument checks of one quantiser call, before any CUDA call (*empty:
// nothing to do).
fa_status quant_check(const float* x, const void* x8, const float* descale, int64_t B, int64_t H, int64_t N,
                      int64_t d, const float* rope_cos, const float* rope_sin, int rope_layout,
                      const int8_t* hadamard_signs, int per_tensor, const float* workspace, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || N < 0 || d < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (per_tensor != 0 && per_tensor != 1) return FA_ERR_INVALID_ARG;
  if (rope_layout != 0 && rope_layout != FA_ROPE_INTERLEAVED && rope_layout != FA_ROPE_HALF) return FA_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || N == 0) {
    *empty = true;
    return FA_OK;
  }
  if (rope_layout != 0 && (!rope_cos || !rope_sin || !aligned16(rope_cos) || !aligned16(rope_sin)))
    return FA_ERR_INVALID_ARG;
  if (!x || !x8 || !descale) return FA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x8) || ((uintptr_t)descale & 3u)) return FA_ERR_INVALID_ARG;
  if (per_tensor && (!workspace || ((uintptr_t)workspace & 3u))) return FA_ERR_INVALID_ARG;
  if (hadamard_signs)
    for (int64_t i = 0; i < d; ++i)
      if (hadamard_signs[i] != 1 && hadamard_signs[i] != -1) return FA_ERR_INVALID_ARG;
  // 128-row blocks are numbered with int
  if (N > ((int64_t)1 << 31) - 128 || B * H > 0x7fffffffLL / ((N + 127) / 128)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// The launch of a checked, non-empty quantiser call (after device_setup).
fa_status quant_fill(const float* x, void* x8, float* descale, int64_t B, int64_t H, int64_t N, int64_t d,
                     const float* rope_cos, const float* rope_sin, int rope_layout, const int8_t* hadamard_signs,
                     int per_tensor, float* workspace, int* err, cudaStream_t stream, fa::QuantLaunch* out) {
  fa::QuantLaunch& L = *out;
  std::memset(&L, 0, sizeof(L));
  if (hadamard_signs) {
    for (int64_t i = 0; i < d; ++i)
      if (hadamard_signs[i] < 0) L.signs.w[i >> 5] |= 1u << (i & 31);
    L.rot = 1;
    L.rinv = (float)(1.0 / std::sqrt((double)d));
  } else {
    L.rot = 0;
    L.rinv = 1.0f;
  }
  L.x = x;
  L.x8 = static_cast<uint8_t*>(x8);
  L.descale = descale;
  L.amax_ws = workspace;
  L.err = err;
  L.BH = (int)(B * H);
  L.N = (int)N;
  L.d = (int)d;
  L.nblk = (int)((N + 127) / 128);
  L.per_tensor = per_tensor;
  L.rope = rope_layout;
  L.rope_cos = rope_cos;
  L.rope_sin = rope_sin;
  L.stream = stream;
  L.drop_pos = -1;
  fa_status st = fa::internal_encode_quant_map(&L.map, x, B * H, N, d);
  if (st == FA_OK && rope_layout != 0 && d != 256)
    st = fa::internal_encode_rope_maps(&L.map_cos, &L.map_sin, rope_cos, rope_sin, N, d);
  return st;
}

fa_status quant_impl(const float* x, void* x8, float* descale, int64_t B, int64_t H, int64_t N, int64_t d,
                     const float* rope_cos, const float* rope_sin, int rope_layout, const int8_t* hadamard_signs,
                     int per_tensor, float* workspace, cudaStream_t stream) {
  bool empty = false;
  fa_status st = quant_check(x, x8, descale, B, H, N, d, rope_cos, rope_sin, rope_layout, hadamard_signs, per_tensor,
                             workspace, &empty);
  if (st != FA_OK || empty) return st;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  fa::QuantLaunch L;
  if ((st = quant_fill(x, x8, descale, B, H, N, d, rope_cos, rope_sin, rope_layout, hadamard_signs, per_tensor,
                       workspace, err, stream, &L)) != FA_OK)
    return st;
  L.drop_pos = fa::internal_take_quant_inject();
  return fa::launch_quant(L) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
}  // namespace

}  // extern "C"

namespace fa {
fa_status internal_device_setup(int* dev, int** err) { return device_setup(dev, err); }

fa_status internal_encode_quant_map(CUtensorMap* map, const float* x, int64_t BH, int64_t N, int64_t d) {
  // 32-float (128-byte) x 64-row boxes, 128-byte swizzle, rows past N read as 0
  return encode_map(map, x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, BH, N, d, 64);
}

fa_status internal_encode_rope_maps(CUtensorMap* map_cos, CUtensorMap* map_sin, const float* rope_cos,
                                    const float* rope_sin, int64_t N, int64_t d) {
  // each table as one head of N rows of d/2 floats: 32-float x 128-row boxes
  fa_status st = encode_map(map_cos, rope_cos, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 1, N, d / 2, 128);
  if (st != FA_OK) return st;
  return encode_map(map_sin, rope_sin, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 1, N, d / 2, 128);
}

int internal_take_quant_inject() { return g_inject_quant.exchange(0) ? 1 : -1; }
}  // namespace fa

extern "C" {

fa_status fa_quant_fp8(const float* x, void* x8, float* descale, int64_t B, int64_t H, int64_t N, int64_t d,
                       const int8_t* hadamard_signs, int per_tensor, float* workspace, cudaStream_t stream) {
  return quant_impl(x, x8, descale, B, H, N, d, nullptr, nullptr, 0, hadamard_signs, per_tensor, workspace, stream);
}

fa_status fa_quant_fp8_rope(const float* x, void* x8, float* descale, int64_t B, int64_t H, int64_t N, int64_t d,
                            const float* rope_cos, const float* rope_sin, int rope_layout,
                            const int8_t* hadamard_signs, int per_tensor, float* workspace, cudaStream_t stream) {
  if (rope_layout != FA_ROPE_INTERLEAVED && rope_layout != FA_ROPE_HALF) return FA_ERR_INVALID_ARG;
  return quant_impl(x, x8, descale, B, H, N, d, rope_cos, rope_sin, rope_layout, hadamard_signs, per_tensor,
                    workspace, stream);
}

fa_status fa_quant_fp8_qkv(const float* q, const float* k, const float* v, void* q8, void* k8, void* v8,
                           float* q_descale, float* k_descale, float* v_descale, int64_t B, int64_t Hq, int64_t Hkv,
                           int64_t Nq, int64_t Nk, int64_t d, const int8_t* hadamard_signs, cudaStream_t stream) {
  // every argument of the three is checked before any CUDA call
  const float* xs[3] = {q, k, v};
  void* x8s[3] = {q8, k8, v8};
  float* dss[3] = {q_descale, k_descale, v_descale};
  const int64_t Hs[3] = {Hq, Hkv, Hkv}, Ns[3] = {Nq, Nk, Nk};
  const int8_t* sgs[3] = {hadamard_signs, hadamard_signs, nullptr};
  bool empty[3];
  fa_status st;
  for (int i = 0; i < 3; ++i)
    if ((st = quant_check(xs[i], x8s[i], dss[i], B, Hs[i], Ns[i], d, nullptr, nullptr, 0, sgs[i], 0, nullptr,
                          &empty[i])) != FA_OK)
      return st;
  if (empty[0] && empty[1] && empty[2]) return FA_OK;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  fa::QuantLaunch L[3];
  for (int i = 0; i < 3; ++i)
    if (!empty[i] && (st = quant_fill(xs[i], x8s[i], dss[i], B, Hs[i], Ns[i], d, nullptr, nullptr, 0, sgs[i], 0,
                                      nullptr, err, stream, &L[i])) != FA_OK)
      return st;
  std::lock_guard<std::mutex> lk(g_qkv_mu);
  QkvPipe& P = g_qkv[dev];
  if (!P.ready) {
    bool ok = cudaEventCreateWithFlags(&P.start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 3; ++i) {
      ok = ok && cudaStreamCreateWithFlags(&P.s[i], cudaStreamNonBlocking) == cudaSuccess;
      ok = ok && cudaEventCreateWithFlags(&P.done[i], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
      // release what was made, so that a later call starts again from nothing
      if (P.start) cudaEventDestroy(P.start);
      P.start = nullptr;
      for (int i = 0; i < 3; ++i) {
        if (P.s[i]) cudaStreamDestroy(P.s[i]);
        if (P.done[i]) cudaEventDestroy(P.done[i]);
        P.s[i] = nullptr;
        P.done[i] = nullptr;
      }
      return FA_ERR_CUDA;
    }
    P.ready = true;
  }
  // fan out from the caller's stream, one quantisation per stream, and join
  // back -- after an error too, so that work the caller enqueues next never
  // runs ahead of a launch that was made
  fa_status result = FA_OK;
  if (cudaEventRecord(P.start, stream) != cudaSuccess) return FA_ERR_CUDA;
  const int drop = fa::internal_take_quant_inject();
  for (int i = 0; i < 3; ++i) {
    if (cudaStreamWaitEvent(P.s[i], P.start, 0) != cudaSuccess) {
      result = FA_ERR_CUDA;
      continue;
    }
    if (empty[i] || result != FA_OK) continue;
    L[i].stream = P.s[i];
    L[i].drop_pos = (i == 0) ? drop : -1;
    if (fa::launch_quant(L[i]) != cudaSuccess) result = FA_ERR_CUDA;
  }
  for (int i = 0; i < 3; ++i)
    if (cudaEventRecord(P.done[i], P.s[i]) != cudaSuccess || cudaStreamWaitEvent(stream, P.done[i], 0) != cudaSuccess)
      if (result == FA_OK) result = FA_ERR_CUDA;
  return result;
}

fa_status fa_bwd_workspace_bytes(int64_t B, int64_t Hq, int64_t Nq, int64_t d, size_t* bytes) {
  if (!bytes) return FA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 0 || Nq < 0 || d < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  const int64_t rows = B * Hq * Nq;
  if (rows > (int64_t)1 << 40) return FA_ERR_UNSUPPORTED;
  const int64_t acc = (rows * d * 4 + 255) / 256 * 256;   // fp32 dQ accumulator
  // per 64-row record: 64 x (-LSE log2 e), 64 x (-D), whole kernel steps per head
  const int64_t recs = B * Hq * (int64_t)fa::bwd_records_per_head(Nq, d == 64 ? 64 : 128) * 512;
  *bytes = (size_t)(acc + recs);
  return FA_OK;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                 int causal, float scale, int dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 0 || Hkv < 0 || Nq < 0 || Nk < 0 || d < 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (d == 256) return FA_ERR_UNSUPPORTED;  // the backward kernel covers d = 64 and 128
  if (B == 0 || Hq == 0) return FA_OK;
  if (Hkv == 0 || Hq % Hkv != 0 || Nk == 0) return FA_ERR_INVALID_ARG;
  const int64_t lim = 0x7fffffffLL - 256;
  if (Nq > lim || Nk > lim || B * Hq > 0x7fffffffLL || B * Hkv * ((Nk + 127) / 128) > 0x7fffffffLL ||
      B * Hq * Nq > ((int64_t)1 << 40))
    return FA_ERR_UNSUPPORTED;
  if (!k || !v || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv)) return FA_ERR_INVALID_ARG;
  int dev = 0;
  int* err = nullptr;
  fa_status st;
  if (Nq == 0) {
    // no query: dK = dV = 0
    if ((st = device_setup(&dev, &err)) != FA_OK) return st;
    const long long bytes = (long long)(B * Hkv * Nk * d * 2);
    if (fa::launch_zero_fill(dk, bytes, stream) != cudaSuccess) return FA_ERR_CUDA;
    if (fa::launch_zero_fill(dv, bytes, stream) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
  }
  if (!q || !o || !lse || !dout || !dq) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) || !aligned16(dq))
    return FA_ERR_INVALID_ARG;
  // the preprocessing kernel runs one block per 8 padded query rows
  if ((B * Hq * fa::bwd_records_per_head(Nq, (int)d) * 64 + 7) / 8 > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  size_t need = 0;
  if ((st = fa_bwd_workspace_bytes(B, Hq, Nq, d, &need)) != FA_OK) return st;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < need)
    return FA_ERR_INVALID_ARG;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;

  const int64_t rows = B * Hq * Nq;
  float* dq_acc = static_cast<float*>(workspace);
  float* vecs = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + (rows * d * 4 + 255) / 256 * 256);
  const bool f16 = dtype == FA_DTYPE_FP16;
  const long long nrec = fa::bwd_records_per_head(Nq, (int)d);
  if (fa::launch_bwd_prep(o, dout, lse, vecs, dq_acc, (long long)(B * Hq), (int)Nq, (int)nrec, (int)d, f16,
                          stream) != cudaSuccess)
    return FA_ERR_CUDA;

  fa::BwdLaunch L;
  std::memset(&L, 0, sizeof(L));
  const CUtensorMapDataType dt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t step_rows = (uint32_t)fa::bwd_step_rows((int)d);
  if ((st = encode_map(&L.q, q, dt, 2, B * Hq, Nq, d, step_rows)) != FA_OK) return st;
  if ((st = encode_map(&L.dout, dout, dt, 2, B * Hq, Nq, d, step_rows)) != FA_OK) return st;
  if ((st = encode_map(&L.k, k, dt, 2, B * Hkv, Nk, d)) != FA_OK) return st;
  if ((st = encode_map(&L.v, v, dt, 2, B * Hkv, Nk, d)) != FA_OK) return st;
  // fp32 dQ accumulator: 32-column (128-byte) x step-row boxes
  if ((st = encode_map(&L.dq_acc, dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, B * Hq, Nq, d, step_rows)) != FA_OK)
    return st;
  if ((st = encode_map(&L.dk, dk, dt, 2, B * Hkv, Nk, d)) != FA_OK) return st;
  if ((st = encode_map(&L.dv, dv, dt, 2, B * Hkv, Nk, d)) != FA_OK) return st;
  L.prm.dq_acc = dq_acc;
  L.prm.dk = dk;
  L.prm.dv = dv;
  L.prm.vecs = vecs;
  L.prm.nrec = (int)nrec;
  L.prm.err = err;
  L.prm.Nq = (int)Nq;
  L.prm.Nk = (int)Nk;
  L.prm.Hq = (int)Hq;
  L.prm.Hkv = (int)Hkv;
  L.prm.BHkv = (int)(B * Hkv);
  L.prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  L.prm.scale = scale;
  L.prm.drop_step = (g_inject.exchange(0) & 1) ? 1 : -1;
  L.stream = stream;
  cudaError_t e;
  if (d == 64) {
    if (f16) e = causal ? fa::launch_attn_bwd<1, 64, true>(L) : fa::launch_attn_bwd<1, 64, false>(L);
    else e = causal ? fa::launch_attn_bwd<0, 64, true>(L) : fa::launch_attn_bwd<0, 64, false>(L);
  } else {
    if (f16) e = causal ? fa::launch_attn_bwd<1, 128, true>(L) : fa::launch_attn_bwd<1, 128, false>(L);
    else e = causal ? fa::launch_attn_bwd<0, 128, true>(L) : fa::launch_attn_bwd<0, 128, false>(L);
  }
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (fa::launch_bwd_dq_convert(dq_acc, dq, scale, (long long)(rows * d), f16, stream) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

const char* fa_status_string(fa_status status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dimension or device (needs sm_103)";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA call or kernel launch failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel pipeline wait ran out of time";
    case FA_ERR_SCRATCH_LIMIT:
      return "FA_ERR_SCRATCH_LIMIT: B*H*ceil(N/128) exceeds FA_QUANT_NOALLOC_MAX_BLOCKS (static scratch)";
  }
  return "FA_ERR_UNKNOWN";
}

fa_status fa_check_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  int dev = 0;
  int* err = nullptr;
  fa_status st = device_setup(&dev, &err);
  if (st != FA_OK) return st;
  int h = 0;
  if (cudaMemcpyFromSymbol(&h, g_fa_device_error, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_device_error, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

fa_status fa_debug_inject(int flags) {
  if (flags < 0 || flags > 3) return FA_ERR_INVALID_ARG;
  g_inject.store(flags & 1);
  g_inject_quant.store((flags >> 1) & 1);
  return FA_OK;
}

fa_status fa_debug_exp2(const float* x, float* y, int64_t n, int method, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (x == nullptr || y == nullptr)) || !(method == 0 || method == 3 || method == 4))
    return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  int dev = 0;
  int* err = nullptr;
  fa_status st = device_setup(&dev, &err);
  if (st != FA_OK) return st;
  const int64_t pairs = (n + 1) / 2;
  if (pairs > (int64_t)256 * 0x7fffffff) return FA_ERR_INVALID_ARG;
  const unsigned grid = (unsigned)((pairs + 255) / 256);
  if (method == 0) fa::exp2_eval_kernel<0><<<grid, 256, 0, stream>>>(x, y, n);
  else if (method == 3) fa::exp2_eval_kernel<3><<<grid, 256, 0, stream>>>(x, y, n);
  else fa::exp2_eval_kernel<4><<<grid, 256, 0, stream>>>(x, y, n);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_version(void) { return 100; }

}  // extern "C"
