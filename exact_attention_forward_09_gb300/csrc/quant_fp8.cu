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
// Arithmetic.  y is the rotated row in fp32: sign flip, then the in-place
// Walsh-Hadamard butterfly with strides 1, 2, 4, ... (a + b, a - b), every
// element seeing the same sequence of fp32 additions whatever lane holds it.
// The block scale is s = amax(y) / 448 in fp32 (1 for an all-zero block) and
// the 1/sqrt(d) factor is folded into the stored descale.  The code is the
// E4M3 value nearest to the exact quotient y / s (ties to even, saturated at
// 448): one rounding, from the real number.  It is decided exactly without a
// division: with r = RN(1/s), the products y * RN(r (1 + 2^-20)) and
// y * RN(r (1 - 2^-20)) bracket y / s strictly, so when both convert to the
// same code that code is the answer; otherwise y / s lies next to the one
// E4M3 midpoint m between the two codes, and the sign of y - m s -- exact
// from a single fused multiply-add, the FMA residual of the Handbook of
// Floating-Point Arithmetic (Muller et al.) -- picks the side, a zero residual
// being a tie.  That happens for about one element in 2^15.
//
// Kernel organisation (persistent, one CTA per SM).  A load warp streams the
// input through a ring of shared-memory slots with TMA (each slot is half a
// 128-row block: 32-float x 64-row boxes, 128-byte swizzle, rows past N read
// as zero), with full / empty mbarriers; a group of warps takes a block in
// one pass (two or three groups on alternate blocks).  A row is spread over 4 lanes
// (lane / 8 picks the quarter, lane % 8 the row; 8 or 16 rows per warp),
// chosen so that the 8 lanes of each shared-memory phase read 8 different
// rows and the swizzle puts them in different banks; at d = 128 each lane
// holds a whole row instead (32 rows per warp, 12 warps; 8 with the rotary
// embedding, whose angle tables take shared memory too),
// so that no stage of the butterfly crosses lanes, and 8 consecutive lanes
// are again 8 rows in different banks.  The rotated rows stay in registers: each warp frees its
// slot as soon as it has read it, takes the block maximum across its group's warps
// through a predicate-AND barrier (which also lets a warp that gave up stop
// the others), and encodes from registers.  HBM-bound: 4 bytes read and 1
// written per element.
#include <climits>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "quant_fp8.h"

namespace fa {
namespace {

template <int D, int LPR_ = 4, bool ROPE_ = false>
struct QCfg {
  // Lanes per row: 1 at d = 128, 4 otherwise (the launch picks).  One lane
  // per row keeps every stage of the butterfly inside a lane (with a row
  // over 4 lanes the two stages that cross lanes took about a third of the
  // kernel's time, measured: 51.8 -> 37.5 us at B=4 H=16 N=4096); its
  // 128-register rows leave 12 warps per SM, which also carry the plain
  // modes a little faster (block scales 31.4-32.8 -> 30.7 us, per tensor
  // 56.9 -> 52.9 us), and with the angle tables staged in shared memory
  // (below) also the rotary embedding without the rotation (rope half
  // 54 -> 48 us, interleaved unchanged).
  static constexpr int LPR = (D == 128) ? LPR_ : 4;
  // Rotary embedding with staged angle tables (d = 64 and 128): the CTA
  // takes a contiguous range of blocks in position-major order (the heads of
  // one 128-row position block next to each other), so one copy of the
  // block's cos and sin rows in shared memory serves every head of its range
  // at that position, read with the same 128-byte swizzle as x.  Loaded per
  // lane from global memory instead, the tables took about half of each
  // call, a chain of dependent loads per row (B=4 H=16 N=4096, d = 128:
  // rope + rotation 82 -> 56 us, rope alone 99 -> 48 us; d = 64, B=8 H=32
  // N=2048: 103 -> 66 and 93 -> 58 us).  d = 256's tables (128 KB) do not
  // fit beside the ring, and it keeps the per-lane loads.
  static constexpr bool TBL = ROPE_ && D != 256;
  static constexpr int TBL_BOXES = D / 2 / 32;                     // 32-float boxes per table row
  static constexpr int TBL_TAB_BYTES = TBL ? TBL_BOXES * 128 * 128 : 0;  // one table, 128 rows
  static constexpr int TBL_BYTES = 2 * TBL_TAB_BYTES;            // cos and sin
  static constexpr int RPW = 32 / LPR;           // rows of a warp's row set
  // Warps per CTA.  With 4 lanes per row the rotation and the exact rounding
  // are latency-bound chains per row, so the warps in flight matter: d = 64
  // runs 32 warps of 64 registers (measured 13% faster with the rotation
  // than 16 warps); d = 256 runs 16 warps (its rows need 128 registers).
  // d = 128 with one row per lane (128 independent elements each) runs 12
  // in three groups of 4 (168 registers; 8 warps of 254 were 17% slower).
  // With staged tables and one lane per row, 8 warps in two groups (the
  // tables take the third group's ring).
  static constexpr int NW = (D == 64) ? 32 : (LPR == 1) ? (TBL ? 8 : 12) : 16;
  static constexpr int THREADS = 32 * NW;
  // Two (one row per lane: three) groups work on alternate blocks, each with
  // its own ring and barrier, so that one group's wait for its block maximum
  // overlaps the other groups' work (d = 256: one group; its rows do not fit
  // twice).
  static constexpr int NG = (D == 256) ? 1 : (LPR == 1 && !TBL) ? 3 : 2;
  static constexpr int WG = NW / NG;             // warps per group
  static constexpr int RS = 128 / (RPW * WG);    // row sets per warp and block
  static_assert(RS == 1 || RS == 2, "a group covers a 128-row block");
  static constexpr int E = D / LPR;              // elements of a row per lane
  static constexpr int G = E < 32 ? E : 32;      // contiguous run of a lane's elements
  static constexpr int BOXES = D / 32;           // 32-float boxes per row
  static constexpr int SLOT_ROWS = 64;           // half a block per slot
  static constexpr int BOX_BYTES = SLOT_ROWS * 128;
  static constexpr int SLOT_BYTES = BOXES * BOX_BYTES;
  // warps that read one slot: every warp of the group (two row sets: both
  // halves of each block) or the warps covering one half
  static constexpr int READERS = (RS == 2) ? WG : SLOT_ROWS / RPW;
  static constexpr int MASKW = (E / 32 > 2) ? E / 32 : 2;  // sign-bit words of a lane's elements
  // Slots per group.  With one row set per warp, a warp reads one half of
  // each block, so each slot must serve one half only and the count is even:
  // position q goes to slot q % NSG and to half q % 2.  (An odd count would
  // let a slot alternate between the halves, and a half running a block
  // ahead could wait on a slot two phases ahead of its last fill, which an
  // mbarrier's phase parity cannot tell from the previous phase.)  With two
  // row sets every warp of a group reads both halves, in order, so any
  // count works.
  static constexpr int NSG_RAW = (196608 - TBL_BYTES) / SLOT_BYTES / NG;
  static constexpr int NSG_CAP = NSG_RAW > 8 ? 8 : NSG_RAW;
  static constexpr int NSG = (RS == 1) ? (NSG_CAP & ~1) : NSG_CAP;
  static_assert(NSG >= 2 && (RS == 2 || NSG % 2 == 0), "ring too shallow or odd");
  static constexpr int NSLOT = NG * NSG;
  // ring, tables, barriers, alignment
  static constexpr int SMEM_BYTES = NSLOT * SLOT_BYTES + TBL_BYTES + 1024 + 1024;
};

template <int NS>
struct QShared {
  uint64_t full[NS];
  uint64_t empty[NS];
  float red[64];       // [group][block parity][warp of group]; MODE 1: [warp]
  int last_pos[NS];
  uint64_t tbl_full;   // staged tables: one completion per table phase
  int tbl_cnt;         // staged tables: warps that have left their table phases, in all
  int tbl_issued;      // staged tables: last table phase issued
  int abort_flag;
  int first_bad;       // first block iteration (of the CTA) some warp could not finish
};

struct QuantParams {
  uint8_t* x8;
  float* descale;
  float* ws;          // MODE 1: one float (atomic max); MODE 2: the tensor maximum; MODE 3: per-block maxima
  int* err;
  const float* rcos;
  const float* rsin;
  SignBits sg;
  int N, nblk, total;  // rows per head, blocks per head, blocks in all
  int rot;
  int x8_vec32;        // x8 is 32-byte aligned
  float rinv;
  int rope;
  int drop_pos;
};

// Atomic add on a shared-memory int, acquire-release at CTA scope (the
// staged tables' phase count): returns the old value.
__device__ __forceinline__ int atom_add_acq_rel_cta(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(v)
               : "memory");
  return old;
}

// Index within the row of a lane's local element e (quarter p of the row).
template <int D, int LPR>
__device__ __forceinline__ int elem_of(int e, int p) {
  if constexpr (QCfg<D, LPR>::LPR == 1) {
    return e;
  } else {
    constexpr int G = QCfg<D, LPR>::G;
    return (e & (G - 1)) + G * p + 128 * (e >> 5);
  }
}

__device__ __forceinline__ uint32_t cvt_e4m3x4(float2 lo, float2 hi) {
  uint16_t a, b;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(a) : "f"(lo.y), "f"(lo.x));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(b) : "f"(hi.y), "f"(hi.x));
  return (uint32_t)a | ((uint32_t)b << 16);
}

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)code));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}

// The bracketing codes of four values differ: settle each differing byte by
// the sign of y - m s (m the E4M3 midpoint between the two candidates).
__device__ __noinline__ uint32_t settle4(float y0, float y1, float y2, float y3, uint32_t chi, uint32_t clo, float s) {
  const float y[4] = {y0, y1, y2, y3};
  uint32_t out = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t ch = (chi >> (8 * b)) & 0xffu, cl = (clo >> (8 * b)) & 0xffu;
    uint32_t c = ch;
    if (ch != cl) {
      const float m = 0.5f * (fabsf(e4m3_value(ch)) + fabsf(e4m3_value(cl)));
      const float rem = fmaf(-m, s, fabsf(y[b]));
      c = rem > 0.0f ? ch : (rem < 0.0f ? cl : ((ch & 1u) ? cl : ch));
    }
    out |= c << (8 * b);
  }
  return out;
}

// Four codes of y / s; rh, rl bracket 1/s from above and below.
__device__ __forceinline__ uint32_t encode4(const float* v, float2 rh, float2 rl, float s) {
  const float2 a = make_float2(v[0], v[1]), b = make_float2(v[2], v[3]);
  const uint32_t ch = cvt_e4m3x4(mul2(a, rh), mul2(b, rh));
  const uint32_t cl = cvt_e4m3x4(mul2(a, rl), mul2(b, rl));
  if (ch == cl) return ch;
  return settle4(v[0], v[1], v[2], v[3], ch, cl, s);
}

// ld(t, col): the four table entries col .. col + 3 of this lane's row, of
// the cos (t = 0) or sin (t = 1) table.
template <int D, int LPR, class Ld>
__device__ __forceinline__ void rope_row(float (&v)[QCfg<D, LPR>::E], int p, const Ld& ld, int mode) {
  constexpr int E = QCfg<D, LPR>::E;
  if (mode == 1) {
    // pairs (2i, 2i+1): adjacent elements of one lane, angle elem / 2
#pragma unroll
    for (int e0 = 0; e0 < E; e0 += 8) {
      const int a0 = elem_of<D, LPR>(e0, p) >> 1;
      const float4 C = ld(0, a0);
      const float4 S = ld(1, a0);
      const float cv[4] = {C.x, C.y, C.z, C.w}, sv[4] = {S.x, S.y, S.z, S.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x = v[e0 + 2 * k], y = v[e0 + 2 * k + 1];
        v[e0 + 2 * k] = __fsub_rn(__fmul_rn(x, cv[k]), __fmul_rn(y, sv[k]));
        v[e0 + 2 * k + 1] = __fadd_rn(__fmul_rn(x, sv[k]), __fmul_rn(y, cv[k]));
      }
    }
  } else if (mode == 2) {
    if constexpr (QCfg<D, LPR>::LPR == 1) {
      // pairs (i, i + D/2): both in this lane
#pragma unroll
      for (int e0 = 0; e0 < D / 2; e0 += 4) {
        const float4 C = ld(0, e0);
        const float4 S = ld(1, e0);
        const float cv[4] = {C.x, C.y, C.z, C.w}, sv[4] = {S.x, S.y, S.z, S.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x = v[e0 + k], y = v[e0 + k + D / 2];
          v[e0 + k] = __fsub_rn(__fmul_rn(x, cv[k]), __fmul_rn(y, sv[k]));
          v[e0 + k + D / 2] = __fadd_rn(__fmul_rn(x, sv[k]), __fmul_rn(y, cv[k]));
        }
      }
    } else if constexpr (D == 256) {
      // pairs (i, i + 128): local elements e and e + 32 of one lane
#pragma unroll
      for (int e0 = 0; e0 < 32; e0 += 4) {
        const int a0 = elem_of<D, LPR>(e0, p);
        const float4 C = ld(0, a0);
        const float4 S = ld(1, a0);
        const float cv[4] = {C.x, C.y, C.z, C.w}, sv[4] = {S.x, S.y, S.z, S.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x = v[e0 + k], y = v[e0 + k + 32];
          v[e0 + k] = __fsub_rn(__fmul_rn(x, cv[k]), __fmul_rn(y, sv[k]));
          v[e0 + k + 32] = __fadd_rn(__fmul_rn(x, sv[k]), __fmul_rn(y, cv[k]));
        }
      }
    } else {
      // pairs (i, i + D/2): quarters p and p ^ 2 of the row, lanes 16 apart
      const bool first = (p & 2) == 0;
#pragma unroll
      for (int e0 = 0; e0 < E; e0 += 4) {
        const int a0 = elem_of<D, LPR>(e0, p & 1);
        const float4 C = ld(0, a0);
        const float4 S = ld(1, a0);
        const float cv[4] = {C.x, C.y, C.z, C.w}, sv[4] = {S.x, S.y, S.z, S.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float o = __shfl_xor_sync(0xffffffffu, v[e0 + k], 16);
          const float x = first ? v[e0 + k] : o, y = first ? o : v[e0 + k];
          v[e0 + k] = first ? __fsub_rn(__fmul_rn(x, cv[k]), __fmul_rn(y, sv[k]))
                            : __fadd_rn(__fmul_rn(x, sv[k]), __fmul_rn(y, cv[k]));
        }
      }
    }
  }
}

// Sign flip and Walsh-Hadamard butterfly of a row, held by one lane or
// spread over the 4 lanes lane % 8 + 8 * {0, 1, 2, 3}; strides in ascending
// order.
template <int D, int LPR>
__device__ __forceinline__ void rotate_row(float (&v)[QCfg<D, LPR>::E], int p,
                                           const uint32_t (&smask)[QCfg<D, LPR>::MASKW]) {
  constexpr int E = QCfg<D, LPR>::E, G = QCfg<D, LPR>::G;
#pragma unroll
  for (int e = 0; e < E; ++e)
    v[e] = __uint_as_float(__float_as_uint(v[e]) ^ ((smask[e >> 5] << (31 - (e & 31))) & 0x80000000u));
  if constexpr (QCfg<D, LPR>::LPR == 1) {
    // every stride inside the lane: 1 scalar, then 2 .. D/2 in packed pairs
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float a = v[e], b = v[e + 1];
      v[e] = __fadd_rn(a, b);
      v[e + 1] = __fsub_rn(a, b);
    }
#pragma unroll
    for (int h = 2; h < E; h <<= 1) {
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        if (!(e & h)) {
          const float2 a = make_float2(v[e], v[e + 1]), b = make_float2(v[e + h], v[e + h + 1]);
          const float2 s = add2(a, b), d = sub2(a, b);
          v[e] = s.x; v[e + 1] = s.y;
          v[e + h] = d.x; v[e + h + 1] = d.y;
        }
      }
    }
  } else {
    // stride 1 (inside a lane, scalar)
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float a = v[e], b = v[e + 1];
      v[e] = __fadd_rn(a, b);
      v[e + 1] = __fsub_rn(a, b);
    }
    // strides 2 .. G/2 (inside a lane, packed pairs)
#pragma unroll
    for (int h = 2; h < G; h <<= 1) {
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        if (!(e & h)) {
          const float2 a = make_float2(v[e], v[e + 1]), b = make_float2(v[e + h], v[e + h + 1]);
          const float2 s = add2(a, b), d = sub2(a, b);
          v[e] = s.x; v[e + 1] = s.y;
          v[e + h] = d.x; v[e + h + 1] = d.y;
        }
      }
    }
    // strides G and 2G: the other quarters of the row (lanes 8 and 16 apart);
    // the lower index takes a + b, the upper b' - a' as RN(partner - own)
#pragma unroll
    for (int m = 8; m <= 16; m <<= 1) {
      const bool upper = (p & (m >> 3)) != 0;
      const float2 sg2 = make_float2(upper ? -1.0f : 1.0f, upper ? -1.0f : 1.0f);
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, v[e], m), __shfl_xor_sync(0xffffffffu, v[e + 1], m));
        const float2 r = fma2(make_float2(v[e], v[e + 1]), sg2, o);
        v[e] = r.x; v[e + 1] = r.y;
      }
    }
    if constexpr (D == 256) {
      // stride 128: local elements e and e + 32
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const float2 a = make_float2(v[e], v[e + 1]), b = make_float2(v[e + 32], v[e + 33]);
        const float2 s = add2(a, b), d = sub2(a, b);
        v[e] = s.x; v[e + 1] = s.y;
        v[e + 32] = d.x; v[e + 33] = d.y;
      }
    }
  }
}

// MODE 0: per-block scale.  MODE 1: per-tensor maximum into *ws (one atomic
// max per CTA).  MODE 2: per-tensor encode with the maximum in *ws.
// MODE 3: per-block maxima to ws[block] (no atomics).
template <int D, int MODE, bool ROPE, int LPR>
__global__ void __launch_bounds__(QCfg<D, LPR, ROPE>::THREADS, 1)
    quant_e4m3_kernel(const __grid_constant__ CUtensorMap map, const __grid_constant__ CUtensorMap map_cos,
                      const __grid_constant__ CUtensorMap map_sin, const QuantParams prm) {
  using C = QCfg<D, LPR, ROPE>;
  constexpr int E = C::E, RS = C::RS, NSG = C::NSG;
  static_assert(C::G == QCfg<D, LPR>::G && C::E == QCfg<D, LPR>::E, "the row helpers use the same lane layout");
  extern __shared__ __align__(1024) uint8_t qsmem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsmem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tbl = ring + C::NSLOT * C::SLOT_BYTES;  // staged tables: cos boxes, then sin boxes
  QShared<C::NSLOT>* sh = reinterpret_cast<QShared<C::NSLOT>*>(tbl + C::TBL_BYTES);
  volatile int* abort_flag = &sh->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (int)gridDim.x;
  const int grp = warp / C::WG;     // group of this warp
  const int wg = warp % C::WG;      // warp within the group
  const int p = (C::LPR == 1) ? 0 : lane >> 3;       // quarter of the row held by this lane
  const int rl = (C::LPR == 1) ? lane : lane & 7;    // row within the warp's row set

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], C::READERS);  // the warps that read a slot's rows
      sh->last_pos[s] = -1;
    }
    mbar_init(&sh->tbl_full, 1);
    sh->tbl_cnt = 0;
    sh->tbl_issued = -1;
    sh->abort_flag = 0;
    sh->first_bad = INT_MAX;
    fence_barrier_init();
  }
  __syncthreads();

  // Block of this CTA's iteration `it` (-1: none left), its head and its
  // 128-row block within the head; the returned index is bh * nblk + blk.
  // Without staged tables the CTAs stride over the blocks head by head
  // (b = blockIdx.x + it * G); with them each CTA takes the contiguous range
  // [t_start, t_end) of the position-major order b' = blk * BH + bh.
  const int nblk_ = prm.nblk, total_ = prm.total, BH = total_ / (nblk_ > 0 ? nblk_ : 1);
  const long long t_start = (long long)blockIdx.x * total_ / G;
  const long long t_end = (long long)(blockIdx.x + 1) * total_ / G;
  auto block_of = [&](int it, int& bh, int& blk) -> int {
    if constexpr (C::TBL) {
      const long long bp = t_start + it;
      if (bp >= t_end) return -1;
      blk = (int)(bp / BH);
      bh = (int)(bp - (long long)blk * BH);
      return bh * nblk_ + blk;
    } else {
      const int b = blockIdx.x + it * G;
      if (b >= total_) return -1;
      bh = b / nblk_;
      blk = b - bh * nblk_;
      return b;
    }
  };

  // Staged tables: phase k holds the cos and sin rows of position block
  // blk_first + k (rows past N read as 0).  Every warp passes through every
  // phase of the CTA in order, waiting for each table (so the barrier's
  // parity never skips a phase) and counting itself out when it moves on;
  // the warp whose count completes phase k issues phase k + 1 into the same
  // buffer, so a table is replaced only after every warp is done with it.
  const int blk_first = C::TBL ? (int)(t_start / BH) : 0;
  const int nphase = C::TBL ? (int)((t_end - 1) / BH) - blk_first + 1 : 0;
  auto tbl_issue = [&](int k) {
    mbar_arrive_expect_tx(&sh->tbl_full, C::TBL_BYTES);
    const int row0 = (blk_first + k) * 128;
#pragma unroll
    for (int bx = 0; bx < C::TBL_BOXES; ++bx) {
      tma_load_3d(tbl + bx * 16384, &map_cos, &sh->tbl_full, 32 * bx, row0, 0);
      tma_load_3d(tbl + C::TBL_TAB_BYTES + bx * 16384, &map_sin, &sh->tbl_full, 32 * bx, row0, 0);
    }
    sh->tbl_issued = k;
  };
  if (C::TBL && threadIdx.x == 0) {
    tma_prefetch_desc(&map_cos);
    tma_prefetch_desc(&map_sin);
    tbl_issue(0);
  }
  int tk = -1;  // table phase this warp holds
  // hold phase k: count out of the phases before it and wait for each table
  auto tbl_to = [&](int k) -> bool {
    bool okk = true;
    while (tk < k) {
      if (tk >= 0) {
        __syncwarp();
        if (lane == 0) {
          const int old = atom_add_acq_rel_cta(&sh->tbl_cnt, 1);
          if (old == C::NW * (tk + 1) - 1 && tk + 1 < nphase && !*abort_flag) {
            fence_proxy_async_smem();
            tbl_issue(tk + 1);
          }
        }
      }
      ++tk;
      okk = __all_sync(0xffffffffu, mbar_wait(&sh->tbl_full, (uint32_t)(tk & 1), abort_flag, prm.err)) && okk;
    }
    return okk;
  };

  // Block iteration `it` of this CTA is block_of(it); group g takes
  // it = g, g + NG, g + 2 NG, ...  Its j-th block fills group positions 2j
  // (rows 0..63) and 2j + 1 (rows 64..127) of the group's ring of NSG slots.
  // Row set k of this warp: half hk, row r_slot within the half.
  constexpr int WPH = C::SLOT_ROWS / C::RPW;   // warps covering one half block
  auto half_of = [&](int k) -> int { return (RS == 2) ? k : wg / WPH; };
  const int r_slot = (wg % WPH) * C::RPW + rl;
  const int swz = r_slot & 7;                   // the 128-byte swizzle's row key
  uint8_t* gring = ring + grp * NSG * C::SLOT_BYTES;
  uint64_t* gfull = &sh->full[grp * NSG];
  uint64_t* gempty = &sh->empty[grp * NSG];
  int* glast = &sh->last_pos[grp * NSG];

  // Loads: lane 0 of the group's first warp keeps the group's ring full,
  // issuing group position q once the slot's previous position was released.
  int issued = 0;
  bool more = true;
  const bool issuer = (wg == 0 && lane == 0);
  auto issue_upto = [&](int limit) -> bool {
    bool ok = true;
    if (issuer) {
      for (; more && issued < limit; ++issued) {
        const int q = issued;
        const int it = C::NG * (q >> 1) + grp;
        int bh, blk;
        if (block_of(it, bh, blk) < 0) { more = false; break; }
        const int slot = q % NSG;
        if (!mbar_wait(&gempty[slot], (uint32_t)(((q / NSG) & 1) ^ 1), abort_flag, prm.err)) {
          ok = false;
          break;
        }
        // test hook: this position is never filled, so its consumers' wait runs out
        if (q == prm.drop_pos && blockIdx.x == 0 && grp == 0) continue;
        const int row0 = blk * 128 + (q & 1) * C::SLOT_ROWS;
        if (row0 >= prm.N) {
          mbar_arrive(&gfull[slot]);  // nothing to load: rows past N are zeros
        } else {
          mbar_arrive_expect_tx(&gfull[slot], C::SLOT_BYTES);
          uint8_t* dst = gring + slot * C::SLOT_BYTES;
#pragma unroll
          for (int k = 0; k < C::BOXES; ++k) tma_load_3d(dst + k * C::BOX_BYTES, &map, &gfull[slot], 32 * k, row0, bh);
        }
        glast[slot] = q;
      }
    }
    return ok;
  };
  if (issuer) tma_prefetch_desc(&map);

  // sign bits of this lane's elements (selected, not indexed, so that the
  // parameter block stays out of local memory)
  uint32_t smask[C::MASKW] = {};
  if (prm.rot) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t w = prm.sg.w[k];
      if constexpr (C::LPR == 1) {
        if (k < C::MASKW) smask[k] = w;
      } else if constexpr (D == 64) {
        if (k == (p >> 1)) smask[0] = (w >> (16 * (p & 1))) & 0xffffu;
      } else {
        if (k == p) smask[0] = w;
        if (D == 256 && k == p + 4) smask[1] = w;
      }
    }
  }
  float s_t = 1.0f;  // MODE 2: the tensor's scale
  if constexpr (MODE == 2) {
    const float am = *prm.ws;
    s_t = (am > 0.0f) ? __fdiv_rn(am, 448.0f) : 1.0f;
  }
  float cta_max = 0.0f;  // MODE 1
  const int N = prm.N;

  for (int j = 0;; ++j) {
    const int it = C::NG * j + grp;
    int bh, blk;
    const int b = block_of(it, bh, blk);
    if (b < 0) break;
    bool ok = __shfl_sync(0xffffffffu, (int)issue_upto(2 * j + NSG), 0) != 0;
    if constexpr (C::TBL) ok = tbl_to(blk - blk_first) && ok;
    float v[RS][E];
    float am = 0.0f;
#pragma unroll
    for (int k = 0; k < RS; ++k) {
      const int hk = half_of(k);
      const int pos = 2 * j + hk;
      const int slot = pos % NSG;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&gfull[slot], (uint32_t)((pos / NSG) & 1), abort_flag, prm.err));
      if (ok) {
        const uint8_t* src = gring + slot * C::SLOT_BYTES + r_slot * 128;
#pragma unroll
        for (int e = 0; e < E; e += 4) {
          const int i = elem_of<D, LPR>(e, p);
          const int ch = (i & 31) >> 2;
          const float4 t = *reinterpret_cast<const float4*>(src + (i >> 5) * C::BOX_BYTES + ((ch ^ swz) << 4));
          v[k][e] = t.x; v[k][e + 1] = t.y; v[k][e + 2] = t.z; v[k][e + 3] = t.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&gempty[slot]);
        // refill the slot as soon as the group has read it (a failure here
        // shows up at the next block's issue)
        (void)__shfl_sync(0xffffffffu, (int)issue_upto(2 * j + NSG + hk + 1), 0);
      }
    }
    if (ok) {
#pragma unroll
      for (int k = 0; k < RS; ++k) {
        const int n = blk * 128 + half_of(k) * C::SLOT_ROWS + r_slot;
        if (n >= N) {
#pragma unroll
          for (int e = 0; e < E; ++e) v[k][e] = 0.0f;
        }
        if constexpr (C::TBL) {
          // row r of the staged block: 16-byte chunk c of each 128-byte box
          // row at position c ^ (r % 8)
          const uint8_t* trow = tbl + (half_of(k) * C::SLOT_ROWS + r_slot) * 128;
          auto ld = [&](int t, int col) -> float4 {
            return *reinterpret_cast<const float4*>(trow + t * C::TBL_TAB_BYTES + (col >> 5) * 16384 +
                                                    ((((col & 31) >> 2) ^ swz) << 4));
          };
          rope_row<D, LPR>(v[k], p, ld, prm.rope);
        } else if constexpr (ROPE) {
          const size_t nr = (size_t)(n < N ? n : N - 1) * (D / 2);
          const float* rc = prm.rcos + nr;
          const float* rs = prm.rsin + nr;
          auto ld = [&](int t, int col) -> float4 {
            return __ldg(reinterpret_cast<const float4*>((t ? rs : rc) + col));
          };
          rope_row<D, LPR>(v[k], p, ld, prm.rope);
        }
        if (prm.rot) rotate_row<D, LPR>(v[k], p, smask);
#pragma unroll
        for (int e = 0; e < E; e += 2) am = max3f(am, fabsf(v[k][e]), fabsf(v[k][e + 1]));
      }
    }

    float s = 1.0f;
    if constexpr (MODE == 1) {
      if (!ok) {
        if (lane == 0) atomicMin(&sh->first_bad, it);
        break;
      }
      cta_max = fmaxf(cta_max, am);
      continue;
    } else if constexpr (MODE == 2) {
      if (!ok) {
        if (lane == 0) atomicMin(&sh->first_bad, it);
        break;
      }
      s = s_t;
    } else {
      // block maximum over the group's warps; the barrier also ends the loop
      // for every warp of the group as soon as one of them could not read
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, m));
      float* red = &sh->red[0] + (grp * 2 + (j & 1)) * C::WG;
      if (lane == 0) red[wg] = am;
      if (!bar_and(1 + grp, 32 * C::WG, ok)) {
        if (lane == 0) atomicMin(&sh->first_bad, it);
        break;
      }
      float bm = red[lane & (C::WG - 1)];
#pragma unroll
      for (int m = C::WG / 2; m >= 1; m >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, m));
      if constexpr (MODE == 3) {
        if (wg == 0 && lane == 0) prm.ws[b] = bm;
        continue;
      }
      s = (bm > 0.0f) ? __fdiv_rn(bm, 448.0f) : 1.0f;
    }
    // encode: a scale too small for its reciprocal to stay finite is
    // handled with y and s both scaled by 2^64 (exact)
    float se = s;
    if (s < 0x1p-64f) {
      se = s * 0x1p64f;
#pragma unroll
      for (int k = 0; k < RS; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) v[k][e] *= 0x1p64f;
    }
    const float r = __frcp_rn(se);
    const float rh = __fmul_rn(r, 0x1.00001p0f), rl_ = __fmul_rn(r, 0x1.ffffep-1f);
    const float2 rh2 = make_float2(rh, rh), rl2 = make_float2(rl_, rl_);
#pragma unroll
    for (int k = 0; k < RS; ++k) {
      const int n = blk * 128 + half_of(k) * C::SLOT_ROWS + r_slot;
      if constexpr (C::LPR == 1) {
        // a whole row per lane: 32 codes at a time, stored as they are made
        uint8_t* row = prm.x8 + ((size_t)bh * N + (n < N ? n : 0)) * D;
#pragma unroll
        for (int jj = 0; jj < E / 32; ++jj) {
          uint32_t w8[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) w8[q] = encode4(&v[k][32 * jj + 4 * q], rh2, rl2, se);
          if (n < N) {
            if (prm.x8_vec32) {
              st_global_v8(row + 32 * jj, w8);
            } else {
              *reinterpret_cast<uint4*>(row + 32 * jj) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
              *reinterpret_cast<uint4*>(row + 32 * jj + 16) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
            }
          }
        }
      } else {
        uint32_t words[E / 4];
#pragma unroll
        for (int q = 0; q < E / 4; ++q) words[q] = encode4(&v[k][4 * q], rh2, rl2, se);
        if (n < N) {
          uint8_t* row = prm.x8 + ((size_t)bh * N + n) * D;
#pragma unroll
          for (int jj = 0; jj < E / 16; ++jj)
            *reinterpret_cast<uint4*>(row + elem_of<D, LPR>(16 * jj, p)) =
                make_uint4(words[4 * jj], words[4 * jj + 1], words[4 * jj + 2], words[4 * jj + 3]);
        }
      }
    }
    if (wg == 0 && lane == 0) prm.descale[b] = __fmul_rn(s, prm.rinv);
  }
  // staged tables: pass through the phases still ahead (counting out of
  // each, which the other warps may be waiting for), up to the last one
  if constexpr (C::TBL) (void)tbl_to(nphase - 1);
  // never leave with copies in flight: after a timeout, each issuer waits
  // (bounded) for the last fill of every slot of its group that was filled
  if (issuer && *abort_flag) {
    for (int sl = 0; sl < NSG; ++sl) {
      const int q = glast[sl];
      if (q < 0) continue;
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&gfull[sl], (uint32_t)((q / NSG) & 1)) && globaltimer() - t0 < FA_WAIT_LIMIT_NS) {
      }
    }
  }
  // the CTA's maximum (MODE 1) and, after a timeout, marks on every block
  // from the first one some warp could not finish, so that no caller reads
  // a stale or unwritten scale without the error word being set
  __syncthreads();
  // and for the table load in flight, if one was issued and not waited for
  if (C::TBL && threadIdx.x == 0 && *abort_flag && sh->tbl_issued >= 0) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&sh->tbl_full, (uint32_t)(sh->tbl_issued & 1)) && globaltimer() - t0 < FA_WAIT_LIMIT_NS) {
    }
  }
  if constexpr (MODE == 1) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) cta_max = fmaxf(cta_max, __shfl_xor_sync(0xffffffffu, cta_max, m));
    if (lane == 0) sh->red[warp] = cta_max;
    __syncthreads();
    if (threadIdx.x == 0) {
      float mx = 0.0f;
      for (int w = 0; w < C::NW; ++w) mx = fmaxf(mx, sh->red[w]);
      if (sh->first_bad != INT_MAX) mx = INFINITY;
      atomicMax(reinterpret_cast<int*>(prm.ws), __float_as_int(mx));
    }
  } else {
    if (threadIdx.x == 0 && sh->first_bad != INT_MAX) {
      for (int it = sh->first_bad;; ++it) {
        int bh, blk;
        const int bb = block_of(it, bh, blk);
        if (bb < 0) break;
        if constexpr (MODE == 3) prm.ws[bb] = INFINITY;
        else prm.descale[bb] = __int_as_float(0x7fc00000);
      }
    }
  }
}

int sm_count_cached() {
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (sms[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    sms[dev] = v;
  }
  return sms[dev];
}

template <int D, int MODE, bool ROPE, int LPR>
cudaError_t launch_one(const QuantLaunch& L, float* ws, int drop_pos) {
  using C = QCfg<D, LPR, ROPE>;
  auto kern = quant_e4m3_kernel<D, MODE, ROPE, LPR>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  QuantParams prm;
  prm.x8 = L.x8;
  prm.descale = L.descale;
  prm.ws = ws;
  prm.err = L.err;
  prm.rcos = L.rope_cos;
  prm.rsin = L.rope_sin;
  prm.sg = L.signs;
  prm.N = L.N;
  prm.nblk = L.nblk;
  prm.total = L.BH * L.nblk;
  prm.rot = L.rot;
  prm.x8_vec32 = (reinterpret_cast<uintptr_t>(L.x8) & 31u) == 0;
  prm.rinv = L.rinv;
  prm.rope = L.rope;
  prm.drop_pos = drop_pos;
  const int sms = sm_count_cached();
  const int grid = prm.total < sms ? prm.total : sms;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, L.stream>>>(L.map, L.map_cos, L.map_sin, prm);
  return cudaGetLastError();
}

template <int D, int MODE, int LPR>
cudaError_t launch_rope(const QuantLaunch& L, float* ws, int drop_pos) {
  return L.rope ? launch_one<D, MODE, true, LPR>(L, ws, drop_pos) : launch_one<D, MODE, false, LPR>(L, ws, drop_pos);
}

// one lane per row at d = 128, 4 otherwise
template <int D, int MODE>
cudaError_t launch_mode(const QuantLaunch& L, float* ws, int drop_pos) {
  return launch_rope<D, MODE, (D == 128) ? 1 : 4>(L, ws, drop_pos);
}

template <int D>
cudaError_t launch_quant_d(const QuantLaunch& L) {
  if (!L.per_tensor) return launch_mode<D, 0>(L, nullptr, L.drop_pos);
  cudaError_t e = cudaMemsetAsync(L.amax_ws, 0, sizeof(float), L.stream);
  if (e != cudaSuccess) return e;
  e = launch_mode<D, 1>(L, L.amax_ws, L.drop_pos);
  if (e != cudaSuccess) return e;
  return launch_mode<D, 2>(L, L.amax_ws, -1);
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
cudaError_t launch_quant_partials_d(const QuantLaunch& L, float* partials, float* amax_out) {
  cudaError_t e = launch_mode<D, 3>(L, partials, L.drop_pos);
  if (e != cudaSuccess) return e;
  reduce_max_kernel<<<1, 1024, 0, L.stream>>>(partials, L.BH * L.nblk, amax_out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_mode<D, 2>(L, amax_out, -1);
}

}  // namespace

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
