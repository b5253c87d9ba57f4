// attn_bwd.cu -- attention backward (dQ, dK, dV) for sm_103a: tcgen05 MMAs
// with TMEM accumulators, TMA tile loads, mbarrier pipelines.
//
// What it computes, for the loss sum(dO * O) of O = softmax(scale Q K^T) V
// (the pages list dQ, dK, dV among the paths to cover and compare the
// backward's speed with FA2: "FlashAttention-3: async pipelines on Hopper",
// sections "correctness validation must cover asynchronous boundaries" and
// "how to read the paper's performance numbers"; the gradient itself is the
// derivative of the definition in wmrh.cn FlashAttention V3 article, sec. 1.1):
//   P_ij  = exp(scale q_i.k_j - LSE_i)       (LSE from the forward pass)
//   dP_ij = dO_i . v_j,   D_i = dO_i . O_i  (= sum_j P_ij dP_ij)
//   dS_ij = P_ij (dP_ij - D_i)
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
// Like the forward, P is recomputed from the scores and the saved LSE, one
// tile at a time, and never stored in global memory.
//
// Organisation.  One CTA per (key/value head, 128-key tile): dK and dV of
// those keys stay in TMEM (lane = key) for the whole run while the CTA walks
// the 64-query tiles of every query head of the group.  Per query tile the
// MMA warp computes S^T = K Q^T and dP^T = V dO^T into TMEM; the compute
// warpgroup (one thread per key) turns a row of each into P and dS (bf16 /
// f16), written back to TMEM (dS also to shared memory); the MMA warp then
// accumulates dV += P^T dO and dK += dS^T Q with the left operand read from
// TMEM, and computes dQ^T = K^T dS^T for the tile, which a second warpgroup
// (one thread per head-dim column) stages in shared memory and adds to an
// fp32 dQ accumulator in global memory with TMA tensor reduce-adds (d = 64
// uses 128-query steps and a row-major dQ tile; see BwdCfg).  Shared-memory
// bandwidth is the scarce resource of this kernel (the tensor core reads its
// shared-memory operands through it), so nothing that can stay in TMEM or
// registers goes through it.
// S^T / dP^T of tile t+1 are issued as soon as tile t's rows are read out,
// so the tensor core runs them while the compute warpgroup works on tile t.
// A preprocessing kernel forms D and clears the dQ accumulator; a last
// kernel scales it and converts it to the element type.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "attn_bwd.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBK = 128;  // keys per CTA (TMEM lanes of S^T, dP^T, dK, dV)
constexpr int kRec = 64;  // query rows per LSE / D record
constexpr int kSmemCap = 232448;

// d = 128: 64-query steps; dK + dV take 256 TMEM columns, so dQ is formed
// transposed (dQ^T = K^T dS^T, M = d) and dS also goes to TMEM for dK.
// d = 64: 128-query steps (S^T, dP^T with N = 128); dQ = dS K has M = 128
// queries, so it comes out row-major per thread; dK reads dS from shared
// memory (no TMEM left for it).
template <int ELEM, int D, bool CAUSAL = false>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "the backward kernel covers head dimensions 64 and 128");
  static constexpr int BQ = (D == 64) ? 128 : 64;  // queries per step
  static constexpr int NCH = D / 64;               // 128-byte column panels per row
  static constexpr int KV_PANEL = kBK * 128;       // one panel of a K or V tile (= one dS panel)
  static constexpr int Q_PANEL = BQ * 128;         // one panel of a Q or dO tile
  static constexpr int KV_BYTES = NCH * KV_PANEL;
  static constexpr int QT_BYTES = NCH * Q_PANEL;
  static constexpr int NST = 3;                    // Q/dO stages
  static constexpr int STAGE_BYTES = 2 * QT_BYTES; // Q, then dO
  static constexpr int REC = BQ / kRec;            // LSE / D records per step
  static constexpr int VEC_FLOATS = REC * 2 * kRec;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_ST = OFF_V + KV_BYTES;
  static constexpr int OFF_DS = OFF_ST + NST * STAGE_BYTES;   // dS [key][query], BQ / 64 panels
  static constexpr int OFF_VEC = OFF_DS + kBK * BQ * 2;       // per stage: REC x (-LSE log2 e [64], -D [64])
  // the dQ tile (BQ rows x D fp32) staged for the tensor reduce-add, in
  // 32-column boxes with the 128-byte swizzle
  static constexpr int DQ_STAGE_BYTES = BQ * D * 4;
  static constexpr int OFF_DQST = (OFF_VEC + NST * VEC_FLOATS * 4 + 1023) / 1024 * 1024;  // swizzled boxes: 1024-aligned
  static_assert(OFF_DS % 1024 == 0 && OFF_DQST % 1024 == 0 && (BQ * 128) % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(OFF_ST % 1024 == 0 && 2 * KV_BYTES <= NST * STAGE_BYTES, "dK / dV staging in the stage area");
  static constexpr int OFF_BAR = OFF_DQST + DQ_STAGE_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
  static_assert(SMEM_BYTES <= kSmemCap, "shared memory budget");
  static constexpr bool DS_TMEM = (D == 128);      // dS in TMEM as dK's left operand
  static constexpr uint32_t COL_DV = 0;
  static constexpr uint32_t COL_DK = D;
  static constexpr uint32_t COL_S = 2 * D;
  static constexpr uint32_t COL_DP = 2 * D + BQ;
  static constexpr uint32_t COL_DQ = 2 * D + 2 * BQ;    // dQ^T (d = 128) or dQ (d = 64): 64 columns
  static constexpr uint32_t COL_P = COL_DQ + 64;        // P, 16-bit pairs: BQ / 2 columns
  static constexpr uint32_t COL_DSM = COL_P + BQ / 2;   // dS likewise (d = 128 only)
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert((DS_TMEM ? COL_DSM + BQ / 2 : COL_DSM) <= TMEM_COLS, "TMEM budget");
  static constexpr uint32_t FMT = (ELEM == 0) ? 1u : 0u;  // bf16 = 1, f16 = 0
  static constexpr uint32_t IDESC_S = instr_desc(FMT, FMT, 0, 0, kBK, BQ);  // S^T, dP^T
  static constexpr uint32_t IDESC_KV = instr_desc(FMT, FMT, 0, 1, kBK, D);  // dV, dK
  // dQ^T (M = d = 128, N = 64 queries) or dQ (M = 128 queries, N = d = 64)
  static constexpr uint32_t IDESC_DQ = instr_desc(FMT, FMT, 1, 1, 128, 64);
  // compute warpgroups (thread = key), each taking HALF_Q of a step's BQ
  // query columns in pieces of PIECE: two warpgroups with 32-column pieces,
  // or four with 16-column pieces for non-causal d = 64, whose 128-query
  // steps are bound by this work (more warps per sub-partition, few live
  // registers; the causal instance measured slower that way); then the dQ
  // warpgroup (thread = head-dim column for d = 128, query row for d = 64),
  // the load warp and the MMA warp
  static constexpr int NCWG = (D == 64 && !CAUSAL) ? 4 : 2;
  static constexpr int COMPUTE_WARPS = 4 * NCWG;
  static constexpr int HALF_Q = BQ / NCWG;   // query columns per compute warpgroup
  static constexpr int PIECE = (NCWG == 4) ? 16 : 32;
  static constexpr int NSUB = HALF_Q / PIECE;  // pieces per warpgroup and step
  static_assert(NSUB >= 1 && HALF_Q % PIECE == 0, "whole pieces");
  static constexpr int DQ_WARP0 = COMPUTE_WARPS;
  static constexpr int LOAD_WARP = DQ_WARP0 + 4;
  static constexpr int MMA_WARP = LOAD_WARP + 1;
  static constexpr int THREADS = 32 * (MMA_WARP + 1);
};

struct BwdBars {
  uint64_t kv_full;
  uint64_t st_full[4];   // NST <= 4
  uint64_t st_empty[4];
  uint64_t s_full;
  uint64_t s_free;
  uint64_t p_full;
  uint64_t p_free;
  uint64_t dq_full;
  uint64_t dq_free;
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// 32 lanes x 32 bit, 16 consecutive columns (thread i: lane quarter base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[W]) {
  if constexpr (W == 32) tmem_ld32(taddr, r);
  else tmem_ld16(taddr, r);
}
template <int W>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[W]) {
  if constexpr (W == 16) tmem_st16(taddr, r);
  else tmem_st8(taddr, r);
}

// Tiled 3-D shared -> global store through a tensor map (box layout as the
// map's swizzle mode), tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* ssrc, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(ssrc)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

template <int ELEM>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (ELEM == 0) return pack_bf16x2(lo, hi);
  else return pack_f16x2(lo, hi);
}

// Bounded spin on a barrier phase with no abort bookkeeping (teardown only).
__device__ __forceinline__ void settle(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < FA_WAIT_LIMIT_NS) {
  }
}

template <int ELEM, int D, bool CAUSAL>
__global__ void __launch_bounds__(BwdCfg<ELEM, D, CAUSAL>::THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv, const BwdParams prm) {
  using C = BwdCfg<ELEM, D, CAUSAL>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::OFF_BAR);
  volatile int* abort_flag = &bars->abort_flag;
  float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Nq = prm.Nq;
  const int Nk = prm.Nk;
  const int nkt = (Nk + kBK - 1) / kBK;
  const int nqt = (Nq + C::BQ - 1) / C::BQ;
  const int nrec = prm.nrec;  // LSE / D records per query head
  const int grp = prm.Hq / prm.Hkv;
  const int koff = Nk - Nq;  // causal: key j visible to query i iff j <= i + koff

  // CTA -> (key/value head, key tile).  Causal: key-tile-major, so the tiles
  // with the most visible queries (the first ones) start first.
  int bkv, kt;
  if constexpr (CAUSAL) {
    kt = (int)blockIdx.x / prm.BHkv;
    bkv = (int)blockIdx.x % prm.BHkv;
  } else {
    bkv = (int)blockIdx.x / nkt;
    kt = (int)blockIdx.x % nkt;
  }
  const int k0 = kt * kBK;
  const int bq_head0 = (bkv / prm.Hkv) * prm.Hq + (bkv % prm.Hkv) * grp;  // first query head (b*Hq + h)
  int qt0 = 0;  // first query tile that sees a key of this tile
  if constexpr (CAUSAL) {
    const int first = k0 - koff;
    qt0 = first > 0 ? first / C::BQ : 0;
  }
  const int per_head = nqt > qt0 ? nqt - qt0 : 0;
  const int T = grp * per_head;  // steps of this CTA
  auto step_of = [&](int t, int& bhq, int& q0) {
    bhq = bq_head0 + t / per_head;
    q0 = (qt0 + t % per_head) * C::BQ;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->st_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 32 * C::COMPUTE_WARPS);
    mbar_init(&bars->p_full, 32 * C::COMPUTE_WARPS);
    mbar_init(&bars->p_free, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 128);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------------------ load --
    // Lane 0 issues every copy: K and V once, then per step the Q and dO
    // tiles and the tile's 64 log2-scaled LSE values and 64 D values (one
    // contiguous 512-byte record prepared by the preprocessing kernel), all
    // counted on the stage's barrier.
    if (T > 0 && lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::KV_BYTES);
      for (int ch = 0; ch < C::NCH; ++ch) {
        tma_load_3d(smem + C::OFF_K + ch * C::KV_PANEL, &tm_k, &bars->kv_full, ch * 64, k0, bkv);
        tma_load_3d(smem + C::OFF_V + ch * C::KV_PANEL, &tm_v, &bars->kv_full, ch * 64, k0, bkv);
      }
      int t = 0;
      for (; t < T; ++t) {
        const int s = t % C::NST;
        if (t >= C::NST &&
            !mbar_wait(&bars->st_empty[s], (uint32_t)(((t / C::NST) - 1) & 1), abort_flag, prm.err))
          break;
        int bhq, q0;
        step_of(t, bhq, q0);
        // failure-injection hook (tests only): this stage is never filled,
        // so the waits on it run out and the kernel aborts
        if (t == prm.drop_step && blockIdx.x == 0) continue;
        mbar_arrive_expect_tx(&bars->st_full[s], 2 * C::QT_BYTES + C::VEC_FLOATS * 4);
        uint8_t* st = smem + C::OFF_ST + s * C::STAGE_BYTES;
        for (int ch = 0; ch < C::NCH; ++ch) {
          tma_load_3d(st + ch * C::Q_PANEL, &tm_q, &bars->st_full[s], ch * 64, q0, bhq);
          tma_load_3d(st + C::QT_BYTES + ch * C::Q_PANEL, &tm_do, &bars->st_full[s], ch * 64, q0, bhq);
        }
        bulk_load(vec + s * C::VEC_FLOATS, prm.vecs + ((size_t)bhq * nrec + q0 / kRec) * (2 * kRec),
                  C::VEC_FLOATS * 4, &bars->st_full[s]);
      }
      // never leave with copies in flight: the K/V tile and each stage's last fill
      settle(&bars->kv_full, 0);
      for (int i = 0; i < C::NST && i < t; ++i) {
        const int tl = t - 1 - i;
        settle(&bars->st_full[tl % C::NST], (uint32_t)((tl / C::NST) & 1));
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------- MMA --
    // Warp-converged issue loop; one elected lane issues each MMA / commit.
    if (T > 0) {
      auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, prm.err));
      };
      const uint32_t k_s = smem_u32(smem + C::OFF_K);
      const uint32_t v_s = smem_u32(smem + C::OFF_V);
      const uint32_t st_s = smem_u32(smem + C::OFF_ST);
      // K-major views (rows of 128 bytes, 8-row groups 1024 bytes apart)
      const uint64_t k_kdesc = smem_desc(k_s, 16, 1024, 2);
      const uint64_t v_kdesc = smem_desc(v_s, 16, 1024, 2);
      const uint64_t st_kdesc = smem_desc(st_s, 16, 1024, 2);
      // MN-major views: the next 64 columns of the MN dimension one panel on
      const uint64_t st_mdesc = smem_desc(st_s, C::Q_PANEL, 1024, 2);   // Q, dO as [K = query][N = d]
      const uint64_t k_mdesc = smem_desc(k_s, C::KV_PANEL, 1024, 2);    // K as [K = key][MN = d]
      const uint64_t ds_mdesc = smem_desc(smem_u32(smem + C::OFF_DS), C::KV_PANEL, 1024, 2);  // dS [K = key][MN = query]

      const uint64_t ds_kdesc = smem_desc(smem_u32(smem + C::OFF_DS), 16, 1024, 2);  // dS [M = key][K = query]
      // S^T = K Q^T (is_dp: dP^T = V dO^T) from stage s; K = d in steps of 16
      auto issue_st = [&](int s, bool is_dp) {
        const uint64_t a0 = is_dp ? v_kdesc : k_kdesc;
        const uint32_t b_off = s * C::STAGE_BYTES + (is_dp ? C::QT_BYTES : 0);
        const uint32_t d_tmem = tmem + (is_dp ? C::COL_DP : C::COL_S);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int ch = ks / 4, in_ch = (ks % 4) * 32;
          const uint64_t a = a0 + (uint64_t)((ch * C::KV_PANEL + in_ch) >> 4);
          const uint64_t b = st_kdesc + (uint64_t)((b_off + ch * C::Q_PANEL + in_ch) >> 4);
          mma_ss_elect<0>(d_tmem, a, b, C::IDESC_S, ks > 0 ? 1u : 0u);
        }
      };
      // dV += P^T dO  and  dK += dS^T Q  over the BQ queries of stage s;
      // P^T from TMEM (16 queries = 8 columns per step), dS^T from TMEM
      // (d = 128) or from shared memory (d = 64)
      auto issue_kv = [&](int s, bool acc) {
#pragma unroll
        for (int ks = 0; ks < C::BQ / 16; ++ks) {
          const uint64_t b = st_mdesc + (uint64_t)((s * C::STAGE_BYTES + C::QT_BYTES + ks * 2048) >> 4);
          mma_ts_elect<0>(tmem + C::COL_DV, tmem + C::COL_P + ks * 8, b, C::IDESC_KV, (acc || ks > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < C::BQ / 16; ++ks) {
          const uint64_t b = st_mdesc + (uint64_t)((s * C::STAGE_BYTES + ks * 2048) >> 4);
          if constexpr (C::DS_TMEM) {
            mma_ts_elect<0>(tmem + C::COL_DK, tmem + C::COL_DSM + ks * 8, b, C::IDESC_KV, (acc || ks > 0) ? 1u : 0u);
          } else {
            const uint64_t a = ds_kdesc + (uint64_t)(((ks / 4) * C::KV_PANEL + (ks % 4) * 32) >> 4);
            mma_ss_elect<0>(tmem + C::COL_DK, a, b, C::IDESC_KV, (acc || ks > 0) ? 1u : 0u);
          }
        }
      };
      // d = 128: dQ^T (d x queries) = K^T dS^T; d = 64: dQ (queries x d) =
      // dS K; both over the kBK keys, operands MN-major in shared memory
      auto issue_dq = [&]() {
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const uint64_t kk = k_mdesc + (uint64_t)((ks * 2048) >> 4);
          const uint64_t dd = ds_mdesc + (uint64_t)((ks * 2048) >> 4);
          if constexpr (D == 128) mma_ss_elect<0>(tmem + C::COL_DQ, kk, dd, C::IDESC_DQ, ks > 0 ? 1u : 0u);
          else mma_ss_elect<0>(tmem + C::COL_DQ, dd, kk, C::IDESC_DQ, ks > 0 ? 1u : 0u);
        }
      };

      bool ok = warp_wait(&bars->kv_full, 0) && warp_wait(&bars->st_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_st(0, false);
        issue_st(0, true);
        mma_commit_elect(&bars->s_full);
      }
      for (int t = 0; t < T && ok; ++t) {
        const int s = t % C::NST;
        if (t + 1 < T) {
          // the next tile's S^T and dP^T, once this tile's rows are read out
          const int s1 = (t + 1) % C::NST;
          ok = warp_wait(&bars->st_full[s1], (uint32_t)(((t + 1) / C::NST) & 1)) &&
               warp_wait(&bars->s_free, (uint32_t)(t & 1));
          if (!ok) break;
          tc_fence_after();
          issue_st(s1, false);
          issue_st(s1, true);
          mma_commit_elect(&bars->s_full);
        }
        ok = warp_wait(&bars->p_full, (uint32_t)(t & 1));
        if (!ok) break;
        tc_fence_after();
        issue_kv(s, t > 0);
        mma_commit_elect(&bars->st_empty[s]);  // last reads of this stage's Q and dO
        if (t >= 1) {
          ok = warp_wait(&bars->dq_free, (uint32_t)((t - 1) & 1));
          if (!ok) break;
          tc_fence_after();
        }
        issue_dq();
        mma_commit_elect(&bars->dq_full);
        mma_commit_elect(&bars->p_free);  // last reads of P and dS
      }
      if (ok) mma_commit_elect(&bars->acc_full);
      // every MMA issued here has completed before TMEM is freed
      mma_commit_elect(&bars->drain);
      settle(&bars->drain, 0);
    }
    __syncwarp();
  } else if (warp < C::COMPUTE_WARPS) {
    // --------------------------------------------------------- compute --
    // Warpgroup g handles query columns [g * HALF_Q, (g + 1) * HALF_Q) of
    // each step, in pieces of PIECE columns; thread r of a warpgroup owns key r (TMEM
    // lane r).
    const int cg = warp / 4;
    const int r = threadIdx.x & 127;
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const int key = k0 + r;
    const int cb = cg * C::HALF_Q;
    const float2 sl2 = make_float2(prm.scale_log2, prm.scale_log2);
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int s = t % C::NST;
      int bhq, q0;
      step_of(t, bhq, q0);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full, (uint32_t)(t & 1), abort_flag, prm.err) &&
                                       mbar_wait(&bars->st_full[s], (uint32_t)((t / C::NST) & 1), abort_flag,
                                                 prm.err));
      if (!ok) break;
      tc_fence_after();
      // causal: columns c < lim (relative to cb) are keys past the query's
      // last visible key
      int lim = 0;
      bool need_mask = false;
      if constexpr (CAUSAL) {
        lim = key - koff - q0 - cb;
        need_mask = (k0 + kBK - 1 - koff - q0 - cb) > 0;  // same for the whole warpgroup
      }
      constexpr int PW = C::PIECE;
#pragma unroll
      for (int sub = 0; sub < C::NSUB; ++sub) {
        const int c0 = cb + PW * sub;  // first query column of this piece
        uint32_t sr[PW], dr[PW];
        tmem_ld_cols<PW>(tmem + lane_addr + C::COL_S + c0, sr);
        tmem_ld_cols<PW>(tmem + lane_addr + C::COL_DP + c0, dr);
        tmem_wait_ld();
        if (sub == C::NSUB - 1) {
          tc_fence_before();
          mbar_arrive(&bars->s_free);  // this step's rows are read out
        }
        // the piece's -LSE * log2(e) and -D values (record c0 / 64)
        const float* nl2 = vec + s * C::VEC_FLOATS + (c0 / kRec) * (2 * kRec) + (c0 % kRec);
        const float* nd = nl2 + kRec;
        uint32_t pp[PW / 2], dd[PW / 2];
#pragma unroll
        for (int i = 0; i < PW; i += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(nl2 + i);
          const float4 d4 = *reinterpret_cast<const float4*>(nd + i);
          // P = 2^(s * scale * log2 e - LSE * log2 e), in pairs
          const float2 x01 = fma2(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), sl2,
                                  make_float2(l4.x, l4.y));
          const float2 x23 = fma2(make_float2(__uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3])), sl2,
                                  make_float2(l4.z, l4.w));
          float p0 = ex2(x01.x), p1 = ex2(x01.y), p2 = ex2(x23.x), p3 = ex2(x23.y);
          if (CAUSAL && need_mask) {
            const int c = PW * sub + i;
            p0 = (c < lim) ? 0.0f : p0;
            p1 = (c + 1 < lim) ? 0.0f : p1;
            p2 = (c + 2 < lim) ? 0.0f : p2;
            p3 = (c + 3 < lim) ? 0.0f : p3;
          }
          // dS = P (dP - D)
          const float2 g01 = add2(make_float2(__uint_as_float(dr[i]), __uint_as_float(dr[i + 1])),
                                  make_float2(d4.x, d4.y));
          const float2 g23 = add2(make_float2(__uint_as_float(dr[i + 2]), __uint_as_float(dr[i + 3])),
                                  make_float2(d4.z, d4.w));
          const float2 s01 = mul2(make_float2(p0, p1), g01);
          const float2 s23 = mul2(make_float2(p2, p3), g23);
          pp[i / 2] = pack2<ELEM>(p0, p1);
          pp[i / 2 + 1] = pack2<ELEM>(p2, p3);
          dd[i / 2] = pack2<ELEM>(s01.x, s01.y);
          dd[i / 2 + 1] = pack2<ELEM>(s23.x, s23.y);
        }
        // P and dS of the previous step have been consumed (checked once,
        // before this step's first store)
        if (sub == 0 && t > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_free, (uint32_t)((t - 1) & 1), abort_flag, prm.err));
          if (!ok) break;
          tc_fence_after();
        }
        // P (and for d = 128 dS) into TMEM, 16-bit pairs: left operands of
        // dV (and dK) ...
        tmem_st_cols<PW / 2>(tmem + lane_addr + C::COL_P + c0 / 2, pp);
        if constexpr (C::DS_TMEM) tmem_st_cols<PW / 2>(tmem + lane_addr + C::COL_DSM + c0 / 2, dd);
        // ... and dS into row r of shared memory ([key][query], 64-query
        // panels, 128-byte swizzle: 16-byte chunk c of a row at c ^ (r % 8))
#pragma unroll
        for (int ch = 0; ch < PW / 8; ++ch) {
          const int c8 = c0 / 8 + ch;  // 8-query chunk index within the step
          uint8_t* row = smem + C::OFF_DS + (c8 / 8) * C::KV_PANEL + r * 128;
          *reinterpret_cast<uint4*>(row + (((c8 % 8) ^ (r & 7)) * 16)) =
              make_uint4(dd[4 * ch], dd[4 * ch + 1], dd[4 * ch + 2], dd[4 * ch + 3]);
        }
      }
      if (!ok) break;
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    // epilogue: warpgroup 0 stores dV, warpgroup 1 scale * dK (any further
    // compute warpgroups are done).  Each thread
    // converts its key's row and writes it into the (now idle) Q/dO stage
    // area as 64-column panels with the 128-byte swizzle; one thread then
    // stores the panels with TMA (rows past Nk are clipped).  The four warps
    // of a warpgroup decide together whether to go on, so none of them
    // waits at the named barrier for a warp that gave up.
    bool have = ok;
    if (ok && T > 0) {
      have = __all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, abort_flag, prm.err));
      if (have) tc_fence_after();
    }
    if (cg < 2 && bar_and(2 + cg, 128, have)) {
      const uint32_t col = cg ? C::COL_DK : C::COL_DV;
      const float mult = cg ? prm.scale : 1.0f;
      uint8_t* stg = smem + C::OFF_ST + cg * C::KV_BYTES;  // kBK rows x D, NCH panels
#pragma unroll 1
      for (int h = 0; h < D / 64; ++h) {
        uint32_t a[32], b[32];
        if (T > 0) {
          tmem_ld32(tmem + lane_addr + col + h * 64, a);
          tmem_ld32(tmem + lane_addr + col + h * 64 + 32, b);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = b[i] = 0u;
        }
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          w[i] = pack2<ELEM>(__uint_as_float(a[2 * i]) * mult, __uint_as_float(a[2 * i + 1]) * mult);
          w[16 + i] = pack2<ELEM>(__uint_as_float(b[2 * i]) * mult, __uint_as_float(b[2 * i + 1]) * mult);
        }
        uint8_t* row = stg + h * C::KV_PANEL + r * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<uint4*>(row + ((i ^ (r & 7)) * 16)) = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
      fence_proxy_async_smem();
      bar_sync_n(2 + cg, 128);
      if (r == 0) {
        const CUtensorMap* map = cg ? &tm_dk : &tm_dv;
        for (int h = 0; h < D / 64; ++h) tma_store_3d(map, stg + h * C::KV_PANEL, h * 64, k0, bkv);
        bulk_commit_group();
        bulk_wait_all();  // the panels are read and the rows written before the CTA exits
      }
    }
  } else if (warp < C::LOAD_WARP) {
    // ------------------------------------------------------------- dQ --
    // d = 128: thread c holds column c of the dQ^T tile (TMEM lane c) and
    // adds it to the fp32 accumulator: per query row, a warp adds 32
    // consecutive floats.  d = 64: thread r holds query row r of the dQ
    // tile; the tile is staged in shared memory (two 32-column boxes,
    // 128-byte swizzle, so the row-per-thread writes are conflict-free) and
    // added by two TMA tensor reduce-adds (rows past Nq are clipped).
    const int c = threadIdx.x - 32 * C::DQ_WARP0;
    const uint32_t lane_addr = (uint32_t)((warp - C::DQ_WARP0) * 32) << 16;
    if constexpr (D == 128) {
      // column c of the dQ^T tile = column c of the dQ tile: element (q, c)
      // goes to box c / 32, row q, float c % 32 (chunk (c % 32) / 4 at
      // position chunk ^ (q % 8)); a warp writes one whole 128-byte row
      uint8_t* stg = smem + C::OFF_DQST;
      if (c == 0) tma_prefetch_desc(&tm_dq);
      const int box = c / 32, ch = (c % 32) / 4, within = (c % 4) * 4;
      for (int t = 0; t < T; ++t) {
        int bhq, q0;
        step_of(t, bhq, q0);
        const bool w_ok =
            __all_sync(0xffffffffu, mbar_wait(&bars->dq_full, (uint32_t)(t & 1), abort_flag, prm.err));
        uint32_t a[32], b[32];
        if (w_ok) {
          tc_fence_after();
          tmem_ld32(tmem + lane_addr + C::COL_DQ, a);
          tmem_ld32(tmem + lane_addr + C::COL_DQ + 32, b);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&bars->dq_free);
        }
        if (c == 0 && t > 0) bulk_wait_read_all();
        if (!bar_and(1, 128, w_ok)) break;
        uint8_t* base = stg + box * (C::BQ * 128) + within;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          *reinterpret_cast<uint32_t*>(base + q * 128 + ((ch ^ (q & 7)) * 16)) = a[q];
          *reinterpret_cast<uint32_t*>(base + (q + 32) * 128 + ((ch ^ (q & 7)) * 16)) = b[q];
        }
        fence_proxy_async_smem();
        bar_sync_n(1, 128);
        if (c == 0) {
#pragma unroll
          for (int bx = 0; bx < D / 32; ++bx) tma_reduce_add_3d(&tm_dq, stg + bx * (C::BQ * 128), 32 * bx, q0, bhq);
          bulk_commit_group();
        }
      }
      if (c == 0) bulk_wait_all();
    } else {
      uint8_t* stg = smem + C::OFF_DQST;
      if (c == 0) tma_prefetch_desc(&tm_dq);
      for (int t = 0; t < T; ++t) {
        int bhq, q0;
        step_of(t, bhq, q0);
        const bool w_ok =
            __all_sync(0xffffffffu, mbar_wait(&bars->dq_full, (uint32_t)(t & 1), abort_flag, prm.err));
        uint32_t a[32], b[32];
        if (w_ok) {
          tc_fence_after();
          tmem_ld32(tmem + lane_addr + C::COL_DQ, a);
          tmem_ld32(tmem + lane_addr + C::COL_DQ + 32, b);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&bars->dq_free);
        }
        // the staging tile is free once the previous reduce has read it
        if (c == 0 && t > 0) bulk_wait_read_all();
        if (!bar_and(1, 128, w_ok)) break;
        // row c: box 0 holds columns 0-31, box 1 columns 32-63; 16-byte
        // chunk k of a row at position k ^ (row % 8)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int pos = ((k ^ (c & 7)) * 16);
          *reinterpret_cast<uint4*>(stg + c * 128 + pos) = make_uint4(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3]);
          *reinterpret_cast<uint4*>(stg + C::BQ * 128 + c * 128 + pos) =
              make_uint4(b[4 * k], b[4 * k + 1], b[4 * k + 2], b[4 * k + 3]);
        }
        fence_proxy_async_smem();
        bar_sync_n(1, 128);
        if (c == 0) {
          tma_reduce_add_3d(&tm_dq, stg, 0, q0, bhq);
          tma_reduce_add_3d(&tm_dq, stg + C::BQ * 128, 32, q0, bhq);
          bulk_commit_group();
        }
      }
      if (c == 0) bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------- small kernels --

// One warp per query row, padded to nrec 64-row records per head: the row's
// record entries (-LSE * log2 e, -D) and a cleared dq_acc row.
template <int D, bool F16>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const void* __restrict__ o, const void* __restrict__ dout,
                                                       const float* __restrict__ lse, float* __restrict__ vecs,
                                                       float* __restrict__ dq_acc, long long prow_total, int nq,
                                                       int nrec) {
  const long long prow = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (prow >= prow_total) return;
  const long long bhq = prow / ((long long)nrec * kRec);
  const int qp = (int)(prow % ((long long)nrec * kRec));  // row within the head, padded
  float* rec = vecs + (bhq * nrec + qp / kRec) * (2 * kRec) + (qp % kRec);
  if (qp >= nq) {
    if (lane == 0) {
      rec[0] = -INFINITY;
      rec[kRec] = 0.0f;
    }
    return;
  }
  const long long row = bhq * nq + qp;
  constexpr int EPL = D / 32;  // elements per lane
  const uint16_t* op = reinterpret_cast<const uint16_t*>(o) + row * D + lane * EPL;
  const uint16_t* dp = reinterpret_cast<const uint16_t*>(dout) + row * D + lane * EPL;
  uint16_t ov[EPL], dv[EPL];
  if constexpr (EPL == 8) {
    *reinterpret_cast<uint4*>(ov) = *reinterpret_cast<const uint4*>(op);
    *reinterpret_cast<uint4*>(dv) = *reinterpret_cast<const uint4*>(dp);
  } else if constexpr (EPL == 4) {
    *reinterpret_cast<uint2*>(ov) = *reinterpret_cast<const uint2*>(op);
    *reinterpret_cast<uint2*>(dv) = *reinterpret_cast<const uint2*>(dp);
  } else {
    *reinterpret_cast<uint32_t*>(ov) = *reinterpret_cast<const uint32_t*>(op);
    *reinterpret_cast<uint32_t*>(dv) = *reinterpret_cast<const uint32_t*>(dp);
  }
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    float a, b;
    if constexpr (F16) {
      a = __half2float(__ushort_as_half(ov[i]));
      b = __half2float(__ushort_as_half(dv[i]));
    } else {
      a = __bfloat162float(__ushort_as_bfloat16(ov[i]));
      b = __bfloat162float(__ushort_as_bfloat16(dv[i]));
    }
    acc = fmaf(a, b, acc);
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) {
    const float l = lse[row];
    rec[0] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;  // a row with no key: P = 0
    rec[kRec] = -acc;
  }
  float* z = dq_acc + row * D + lane * EPL;
  if constexpr (EPL == 2) {
    *reinterpret_cast<float2*>(z) = make_float2(0.0f, 0.0f);
  } else {
#pragma unroll
    for (int i = 0; i < EPL / 4; ++i) reinterpret_cast<float4*>(z)[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
}

template <bool F16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ acc, void* __restrict__ dq,
                                                             float scale, long long n8) {
  const float4* a4 = reinterpret_cast<const float4*>(acc);
  uint4* o = reinterpret_cast<uint4*>(dq);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const float4 x = a4[2 * i], y = a4[2 * i + 1];
    uint4 r;
    if constexpr (F16) {
      r.x = pack_f16x2(x.x * scale, x.y * scale);
      r.y = pack_f16x2(x.z * scale, x.w * scale);
      r.z = pack_f16x2(y.x * scale, y.y * scale);
      r.w = pack_f16x2(y.z * scale, y.w * scale);
    } else {
      r.x = pack_bf16x2(x.x * scale, x.y * scale);
      r.y = pack_bf16x2(x.z * scale, x.w * scale);
      r.z = pack_bf16x2(y.x * scale, y.y * scale);
      r.w = pack_bf16x2(y.z * scale, y.w * scale);
    }
    o[i] = r;
  }
}

__global__ void __launch_bounds__(256) zero_fill_kernel(uint4* __restrict__ p, long long n16) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (long long)gridDim.x * blockDim.x)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// grid for a grid-stride loop over n items: at most 8 blocks of 256 per SM
unsigned stride_grid(long long n) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long b = (n + 255) / 256;
  const long long cap = 8LL * sms;
  if (b > cap) b = cap;
  return (unsigned)(b < 1 ? 1 : b);
}

}  // namespace

template <int ELEM, int D, bool CAUSAL>
cudaError_t launch_attn_bwd(const BwdLaunch& L) {
  using C = BwdCfg<ELEM, D, CAUSAL>;
  auto kern = attn_bwd_kernel<ELEM, D, CAUSAL>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  const long long nkt = (L.prm.Nk + kBK - 1) / kBK;
  const long long ctas = (long long)L.prm.BHkv * nkt;
  kern<<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, L.stream>>>(L.q, L.dout, L.k, L.v, L.dq_acc, L.dk, L.dv,
                                                               L.prm);
  return cudaGetLastError();
}

template cudaError_t launch_attn_bwd<0, 128, false>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<0, 128, true>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<1, 128, false>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<1, 128, true>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<0, 64, false>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<0, 64, true>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<1, 64, false>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<1, 64, true>(const BwdLaunch&);

// Query rows per step of the kernel for head dimension d (the Q / dO TMA
// box height) and the 64-row LSE / D records it needs per query head.
int bwd_step_rows(int d) { return d == 64 ? BwdCfg<0, 64>::BQ : BwdCfg<0, 128>::BQ; }
long long bwd_records_per_head(long long nq, int d) {
  const long long bq = bwd_step_rows(d);
  return (nq + bq - 1) / bq * (bq / kRec);
}

cudaError_t launch_bwd_prep(const void* o, const void* dout, const float* lse, float* vecs, float* dq_acc,
                            long long bhq, int nq, int nrec, int d, bool f16, cudaStream_t stream) {
  const long long prows = bhq * nrec * kRec;
  const unsigned blocks = (unsigned)((prows + 7) / 8);
  if (d == 64) {
    if (f16) bwd_prep_kernel<64, true><<<blocks, 256, 0, stream>>>(o, dout, lse, vecs, dq_acc, prows, nq, nrec);
    else bwd_prep_kernel<64, false><<<blocks, 256, 0, stream>>>(o, dout, lse, vecs, dq_acc, prows, nq, nrec);
  } else if (d == 128) {
    if (f16) bwd_prep_kernel<128, true><<<blocks, 256, 0, stream>>>(o, dout, lse, vecs, dq_acc, prows, nq, nrec);
    else bwd_prep_kernel<128, false><<<blocks, 256, 0, stream>>>(o, dout, lse, vecs, dq_acc, prows, nq, nrec);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_convert(const float* dq_acc, void* dq, float scale, long long elems, bool f16,
                                  cudaStream_t stream) {
  const long long n8 = elems / 8;
  const unsigned g = stride_grid(n8);
  if (f16) bwd_dq_convert_kernel<true><<<g, 256, 0, stream>>>(dq_acc, dq, scale, n8);
  else bwd_dq_convert_kernel<false><<<g, 256, 0, stream>>>(dq_acc, dq, scale, n8);
  return cudaGetLastError();
}

cudaError_t launch_zero_fill(void* p, long long bytes, cudaStream_t stream) {
  const long long n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  zero_fill_kernel<<<stride_grid(n16), 256, 0, stream>>>(reinterpret_cast<uint4*>(p), n16);
  return cudaGetLastError();
}

}  // namespace fa
