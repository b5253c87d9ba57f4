// quant_fp8_noalloc.cu -- per-tensor FP8 quantisation for callers that cannot
// allocate device memory.
//
// fa_quant_fp8 in per-tensor mode needs one float of device scratch from the
// caller.  Some callers cannot provide it: code that runs while a stream is
// being captured into a CUDA graph by a framework that owns every buffer,
// plug-ins whose host application hands out all device memory and forbids
// cudaMalloc (which can also synchronise the device and stall other work),
// and runtimes with a fixed memory budget.  This entry point needs no
// allocation at all: its scratch is a file-scope device array compiled into
// the library, which every GPU that loads the library holds until the
// process exits.
//
// The scratch holds one partial maximum per 128-row block plus the final
// maximum, so a call is limited to FA_QUANT_NOALLOC_MAX_BLOCKS blocks
// (B * H * ceil(N / 128)); larger calls are rejected with
// FA_ERR_SCRATCH_LIMIT before anything is launched.  Every partial a call
// reads was written earlier in the same call, so nothing has to be cleared:
// a block whose input load timed out writes +inf (and the library's error
// word is set, reported by fa_check_device_error), never leaves an earlier
// call's value in place.  But all calls share the one array, so two calls
// that overlap on the GPU (different streams, or different host threads on
// one device) race and may produce wrong scales.  Serialise them.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"
#include "quant_fp8.h"

namespace {

constexpr int kScratchFloats = FA_QUANT_NOALLOC_MAX_BLOCKS + 64;  // partials + final max slot
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};
bool g_supported[kMaxDevices] = {};

// Once per device, with that device current: check the architecture and look
// up the device address of the scratch array (in host code the symbol itself
// is only a host-side stand-in and must never be passed to a kernel).
fa_status scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    g_supported[dev] = (major == 10 && minor == 3);
    if (!g_supported[dev]) return FA_ERR_UNSUPPORTED;
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_quant_fp8_per_tensor_noalloc(const float* x, void* x8, float* descale, int64_t B,
                                                     int64_t H, int64_t N, int64_t d,
                                                     const int8_t* hadamard_signs, cudaStream_t stream) {
  if (B < 0 || H < 0 || N < 0 || d < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) return FA_OK;
  const int64_t nblk = (N + 127) / 128;
  if (N > ((int64_t)1 << 31) - 128) return FA_ERR_UNSUPPORTED;
  if (B * H > FA_QUANT_NOALLOC_MAX_BLOCKS || B * H * nblk > FA_QUANT_NOALLOC_MAX_BLOCKS)
    return FA_ERR_SCRATCH_LIMIT;
  if (!x || !x8 || !descale) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x8) & 15u) ||
      (reinterpret_cast<uintptr_t>(descale) & 3u))
    return FA_ERR_INVALID_ARG;

  fa::QuantLaunch L;
  std::memset(&L, 0, sizeof(L));
  if (hadamard_signs) {
    for (int64_t i = 0; i < d; ++i) {
      const int8_t sgn = hadamard_signs[i];
      if (sgn != 1 && sgn != -1) return FA_ERR_INVALID_ARG;
      if (sgn < 0) L.signs.w[i >> 5] |= 1u << (i & 31);
    }
    L.rot = 1;
    L.rinv = (float)(1.0 / std::sqrt((double)d));
  } else {
    L.rot = 0;
    L.rinv = 1.0f;
  }

  int dev = 0;
  int* err = nullptr;
  fa_status st = fa::internal_device_setup(&dev, &err);
  if (st != FA_OK) return st;
  float* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != FA_OK) return st;
  if ((st = fa::internal_encode_quant_map(&L.map, x, B * H, N, d)) != FA_OK) return st;

  L.x = x;
  L.x8 = static_cast<uint8_t*>(x8);
  L.descale = descale;
  L.amax_ws = nullptr;
  L.BH = (int)(B * H);
  L.N = (int)N;
  L.d = (int)d;
  L.nblk = (int)nblk;
  L.per_tensor = 1;
  L.err = err;
  L.drop_pos = fa::internal_take_quant_inject();
  L.stream = stream;
  return fa::launch_quant_per_tensor_partials(L, scratch, scratch + FA_QUANT_NOALLOC_MAX_BLOCKS) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}
