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
// f16) in shared memory; the MMA warp then accumulates dV += P^T dO and
// dK += dS^T Q and computes dQ^T = K^T dS^T for the tile, which a second
// warpgroup (one thread per head-dim column) moves through shared memory and
// adds to an fp32 dQ accumulator in global memory with a bulk reduce-add.
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
constexpr int kBQ = 64;   // queries per step
constexpr int kSmemCap = 232448;

template <int ELEM, int D>
struct BwdCfg {
  static_assert(D == 128, "the backward kernel covers head dimension 128");
  static constexpr int NCH = D / 64;               // 128-byte column panels per row
  static constexpr int KV_PANEL = kBK * 128;       // one panel of a K or V tile
  static constexpr int Q_PANEL = kBQ * 128;        // one panel of a Q or dO tile
  static constexpr int KV_BYTES = NCH * KV_PANEL;
  static constexpr int QT_BYTES = NCH * Q_PANEL;
  static constexpr int NST = 3;                    // Q/dO stages
  static constexpr int STAGE_BYTES = 2 * QT_BYTES; // Q, then dO
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_ST = OFF_V + KV_BYTES;
  static constexpr int OFF_P = OFF_ST + NST * STAGE_BYTES;
  static constexpr int OFF_DS = OFF_P + kBK * kBQ * 2;
  static constexpr int OFF_DQ = OFF_DS + kBK * kBQ * 2;   // dQ tile staging, fp32 [kBQ][D]
  static constexpr int OFF_VEC = OFF_DQ + kBQ * D * 4;    // per stage: log2-scaled LSE[kBQ], D[kBQ]
  static constexpr int OFF_BAR = OFF_VEC + NST * 2 * kBQ * 4;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
  static_assert(SMEM_BYTES <= kSmemCap, "shared memory budget");
  static constexpr uint32_t COL_DV = 0;
  static constexpr uint32_t COL_DK = D;
  static constexpr uint32_t COL_S = 2 * D;
  static constexpr uint32_t COL_DP = 2 * D + kBQ;
  static constexpr uint32_t COL_DQ = 2 * D + 2 * kBQ;  // two buffers of kBQ columns
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_DQ + 2 * kBQ <= TMEM_COLS, "TMEM budget");
  static constexpr uint32_t FMT = (ELEM == 0) ? 1u : 0u;  // bf16 = 1, f16 = 0
  static constexpr uint32_t IDESC_S = instr_desc(FMT, FMT, 0, 0, kBK, kBQ);  // S^T, dP^T
  static constexpr uint32_t IDESC_KV = instr_desc(FMT, FMT, 0, 1, kBK, D);   // dV, dK
  static constexpr uint32_t IDESC_DQ = instr_desc(FMT, FMT, 1, 1, D, kBQ);   // dQ^T
  static constexpr int DQ_WARP0 = 4;  // warps 0-3: compute (thread = key); 4-7: dQ (thread = column)
  static constexpr int LOAD_WARP = 8;
  static constexpr int MMA_WARP = 9;
  static constexpr int THREADS = 320;
};

struct BwdBars {
  uint64_t kv_full;
  uint64_t st_full[3];
  uint64_t st_empty[3];
  uint64_t s_full;
  uint64_t s_free;
  uint64_t p_full;
  uint64_t p_free;
  uint64_t dq_full[2];
  uint64_t dq_free[2];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

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
__global__ void __launch_bounds__(320, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const BwdParams prm) {
  using C = BwdCfg<ELEM, D>;
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
  const int nqt = (Nq + kBQ - 1) / kBQ;
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
    qt0 = first > 0 ? first / kBQ : 0;
  }
  const int per_head = nqt > qt0 ? nqt - qt0 : 0;
  const int T = grp * per_head;  // steps of this CTA
  auto step_of = [&](int t, int& bhq, int& q0) {
    bhq = bq_head0 + t / per_head;
    q0 = (qt0 + t % per_head) * kBQ;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bars->st_full[s], 32);
      mbar_init(&bars->st_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 128);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->p_free, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->dq_full[b], 1);
      mbar_init(&bars->dq_free[b], 128);
    }
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
    // Lane 0 issues the TMA copies; all lanes stage the per-row LSE (scaled
    // to log2 units) and D of each query tile, and all arrive on the stage.
    if (T > 0) {
      bool ok = true;
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(&bars->kv_full, 2 * C::KV_BYTES);
        for (int ch = 0; ch < C::NCH; ++ch) {
          tma_load_3d(smem + C::OFF_K + ch * C::KV_PANEL, &tm_k, &bars->kv_full, ch * 64, k0, bkv);
          tma_load_3d(smem + C::OFF_V + ch * C::KV_PANEL, &tm_v, &bars->kv_full, ch * 64, k0, bkv);
        }
      }
      int t = 0;
      for (; t < T; ++t) {
        const int s = t % C::NST;
        if (t >= C::NST) {
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&bars->st_empty[s], (uint32_t)(((t / C::NST) - 1) & 1), abort_flag, prm.err));
          if (!ok) break;
        }
        int bhq, q0;
        step_of(t, bhq, q0);
        float* l2s = vec + s * 2 * kBQ;
        float* drs = l2s + kBQ;
        for (int e = lane; e < kBQ; e += 32) {
          const int i = q0 + e;
          float l2 = INFINITY, dr = 0.0f;  // rows past Nq: P = 0
          if (i < Nq) {
            const float l = prm.lse[(size_t)bhq * Nq + i];
            l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;  // a row with no key: P = 0
            dr = prm.drow[(size_t)bhq * Nq + i];
          }
          l2s[e] = l2;
          drs[e] = dr;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->st_full[s], 2 * C::QT_BYTES);
          uint8_t* st = smem + C::OFF_ST + s * C::STAGE_BYTES;
          for (int ch = 0; ch < C::NCH; ++ch) {
            tma_load_3d(st + ch * C::Q_PANEL, &tm_q, &bars->st_full[s], ch * 64, q0, bhq);
            tma_load_3d(st + C::QT_BYTES + ch * C::Q_PANEL, &tm_do, &bars->st_full[s], ch * 64, q0, bhq);
          }
        } else {
          mbar_arrive(&bars->st_full[s]);
        }
      }
      // never leave with copies in flight: the K/V tile and each stage's last fill
      if (lane == 0) {
        settle(&bars->kv_full, 0);
        for (int i = 0; i < C::NST && i < t; ++i) {
          const int tl = t - 1 - i;
          settle(&bars->st_full[tl % C::NST], (uint32_t)((tl / C::NST) & 1));
        }
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
      const uint64_t p_kdesc = smem_desc(smem_u32(smem + C::OFF_P), 16, 1024, 2);
      const uint64_t ds_kdesc = smem_desc(smem_u32(smem + C::OFF_DS), 16, 1024, 2);
      // MN-major views: the next 64 columns of the MN dimension one panel on
      const uint64_t st_mdesc = smem_desc(st_s, C::Q_PANEL, 1024, 2);   // Q, dO as [K = query][N = d]
      const uint64_t k_mdesc = smem_desc(k_s, C::KV_PANEL, 1024, 2);    // K as [K = key][M = d]
      const uint64_t ds_mdesc = smem_desc(smem_u32(smem + C::OFF_DS), C::KV_PANEL, 1024, 2);  // dS [K = key][N = query]

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
      // dV += P^T dO  and  dK += dS^T Q  over the kBQ queries of stage s
      auto issue_kv = [&](int s, bool acc) {
#pragma unroll
        for (int ks = 0; ks < kBQ / 16; ++ks) {
          const uint64_t a = p_kdesc + (uint64_t)((ks * 32) >> 4);
          const uint64_t b = st_mdesc + (uint64_t)((s * C::STAGE_BYTES + C::QT_BYTES + ks * 2048) >> 4);
          mma_ss_elect<0>(tmem + C::COL_DV, a, b, C::IDESC_KV, (acc || ks > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < kBQ / 16; ++ks) {
          const uint64_t a = ds_kdesc + (uint64_t)((ks * 32) >> 4);
          const uint64_t b = st_mdesc + (uint64_t)((s * C::STAGE_BYTES + ks * 2048) >> 4);
          mma_ss_elect<0>(tmem + C::COL_DK, a, b, C::IDESC_KV, (acc || ks > 0) ? 1u : 0u);
        }
      };
      // dQ^T (d x queries) = K^T dS^T over the kBK keys, into buffer bq
      auto issue_dq = [&](int bq) {
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const uint64_t a = k_mdesc + (uint64_t)((ks * 2048) >> 4);
          const uint64_t b = ds_mdesc + (uint64_t)((ks * 2048) >> 4);
          mma_ss_elect<0>(tmem + C::COL_DQ + bq * kBQ, a, b, C::IDESC_DQ, ks > 0 ? 1u : 0u);
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
        const int bq = t & 1;
        if (t >= 2) {
          ok = warp_wait(&bars->dq_free[bq], (uint32_t)(((t >> 1) - 1) & 1));
          if (!ok) break;
          tc_fence_after();
        }
        issue_dq(bq);
        mma_commit_elect(&bars->dq_full[bq]);
        mma_commit_elect(&bars->p_free);  // last reads of P and dS
      }
      if (ok) mma_commit_elect(&bars->acc_full);
      // every MMA issued here has completed before TMEM is freed
      mma_commit_elect(&bars->drain);
      settle(&bars->drain, 0);
    }
    __syncwarp();
  } else if (warp < C::DQ_WARP0) {
    // --------------------------------------------------------- compute --
    const int r = threadIdx.x;                       // key within the tile = TMEM lane
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
    const int key = k0 + r;
    const float sl2 = prm.scale_log2;
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
      uint32_t sa[32], sb[32], pa[32], pb[32];
      tmem_ld32(tmem + lane_addr + C::COL_S, sa);
      tmem_ld32(tmem + lane_addr + C::COL_S + 32, sb);
      tmem_ld32(tmem + lane_addr + C::COL_DP, pa);
      tmem_ld32(tmem + lane_addr + C::COL_DP + 32, pb);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->s_free);

      const float* l2s = vec + s * 2 * kBQ;
      const float* drs = l2s + kBQ;
      // causal: columns c < lim are keys past the query's last visible key
      int lim = 0;
      bool need_mask = false;
      if constexpr (CAUSAL) {
        lim = key - koff - q0;
        need_mask = (k0 + kBK - 1 - koff - q0) > 0;  // same for the whole CTA step
      }
      uint32_t pp[32], dd[32];
      auto half = [&](const uint32_t(&sr)[32], const uint32_t(&dr)[32], int cb) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(l2s + cb + i);
          const float4 d4 = *reinterpret_cast<const float4*>(drs + cb + i);
          const float la[4] = {l4.x, l4.y, l4.z, l4.w};
          const float da[4] = {d4.x, d4.y, d4.z, d4.w};
          float pv[4], dv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float p = ex2(fmaf(__uint_as_float(sr[i + u]), sl2, -la[u]));
            if (CAUSAL && need_mask) p = (cb + i + u < lim) ? 0.0f : p;
            pv[u] = p;
            dv[u] = p * (__uint_as_float(dr[i + u]) - da[u]);
          }
          pp[(cb + i) / 2] = pack2<ELEM>(pv[0], pv[1]);
          pp[(cb + i) / 2 + 1] = pack2<ELEM>(pv[2], pv[3]);
          dd[(cb + i) / 2] = pack2<ELEM>(dv[0], dv[1]);
          dd[(cb + i) / 2 + 1] = pack2<ELEM>(dv[2], dv[3]);
        }
      };
      half(sa, pa, 0);
      half(sb, pb, 32);

      // P and dS of the previous step have been consumed
      if (t > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_free, (uint32_t)((t - 1) & 1), abort_flag, prm.err));
        if (!ok) break;
        tc_fence_after();
      }
      // row r of P and dS, 128-byte swizzle: 16-byte chunk c at c ^ (r % 8)
      uint8_t* prow = smem + C::OFF_P + r * 128;
      uint8_t* drow = smem + C::OFF_DS + r * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const int pc = (ch ^ (r & 7)) * 16;
        *reinterpret_cast<uint4*>(prow + pc) = make_uint4(pp[4 * ch], pp[4 * ch + 1], pp[4 * ch + 2], pp[4 * ch + 3]);
        *reinterpret_cast<uint4*>(drow + pc) = make_uint4(dd[4 * ch], dd[4 * ch + 1], dd[4 * ch + 2], dd[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->p_full);
    }
    // epilogue: dV and scale * dK rows of this tile's keys
    if (ok && T > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, abort_flag, prm.err));
      if (ok) tc_fence_after();
    }
    if (ok) {
      const bool store = key < Nk;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which ? C::COL_DK : C::COL_DV;
        const float mult = which ? prm.scale : 1.0f;
        uint8_t* dst = reinterpret_cast<uint8_t*>(which ? prm.dk : prm.dv) + ((size_t)bkv * Nk + key) * D * 2;
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
          if (store) {
            uint4* o = reinterpret_cast<uint4*>(dst + h * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
      }
    }
  } else if (warp < C::LOAD_WARP) {
    // ------------------------------------------------------------- dQ --
    // Thread c holds column c of the dQ^T tile (TMEM lane c); it writes the
    // tile row-major into shared memory, then one thread adds the tile's
    // valid rows to the fp32 accumulator with a bulk reduce-add.
    const int c = threadIdx.x - 32 * C::DQ_WARP0;
    const uint32_t lane_addr = (uint32_t)((warp - C::DQ_WARP0) * 32) << 16;
    float* stg = reinterpret_cast<float*>(smem + C::OFF_DQ);
    for (int t = 0; t < T; ++t) {
      const int bq = t & 1;
      int bhq, q0;
      step_of(t, bhq, q0);
      const bool w_ok =
          __all_sync(0xffffffffu, mbar_wait(&bars->dq_full[bq], (uint32_t)((t >> 1) & 1), abort_flag, prm.err));
      uint32_t a[32], b[32];
      if (w_ok) {
        tc_fence_after();
        tmem_ld32(tmem + lane_addr + C::COL_DQ + bq * kBQ, a);
        tmem_ld32(tmem + lane_addr + C::COL_DQ + bq * kBQ + 32, b);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->dq_free[bq]);
      }
      // the staging tile is free once the previous reduce has read it
      if (c == 0 && t > 0) bulk_wait_read_all();
      if (!bar_and(1, 128, w_ok)) break;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        stg[q * D + c] = __uint_as_float(a[q]);
        stg[(q + 32) * D + c] = __uint_as_float(b[q]);
      }
      fence_proxy_async_smem();
      bar_sync_n(1, 128);
      if (c == 0) {
        const int rows = Nq - q0 < kBQ ? Nq - q0 : kBQ;
        bulk_reduce_add_f32(prm.dq_acc + ((size_t)bhq * Nq + q0) * D, stg, (uint32_t)(rows * D * 4));
        bulk_commit_group();
      }
    }
    if (c == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------- small kernels --

template <int D, bool F16>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const void* __restrict__ o, const void* __restrict__ dout,
                                                       float* __restrict__ drow, float* __restrict__ dq_acc,
                                                       long long rows) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
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
  if (lane == 0) drow[row] = acc;
  float4* z = reinterpret_cast<float4*>(dq_acc + row * D + lane * EPL);
#pragma unroll
  for (int i = 0; i < (EPL + 3) / 4; ++i) {
    if (EPL >= 4) z[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  if constexpr (EPL == 2) *reinterpret_cast<float2*>(dq_acc + row * D + lane * 2) = make_float2(0.0f, 0.0f);
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
  using C = BwdCfg<ELEM, D>;
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
  kern<<<(unsigned)ctas, C::THREADS, C::SMEM_BYTES, L.stream>>>(L.q, L.dout, L.k, L.v, L.prm);
  return cudaGetLastError();
}

template cudaError_t launch_attn_bwd<0, 128, false>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<0, 128, true>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<1, 128, false>(const BwdLaunch&);
template cudaError_t launch_attn_bwd<1, 128, true>(const BwdLaunch&);

cudaError_t launch_bwd_prep(const void* o, const void* dout, float* drow, float* dq_acc, long long rows, int d,
                            bool f16, cudaStream_t stream) {
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  if (d == 64) {
    if (f16) bwd_prep_kernel<64, true><<<blocks, 256, 0, stream>>>(o, dout, drow, dq_acc, rows);
    else bwd_prep_kernel<64, false><<<blocks, 256, 0, stream>>>(o, dout, drow, dq_acc, rows);
  } else if (d == 128) {
    if (f16) bwd_prep_kernel<128, true><<<blocks, 256, 0, stream>>>(o, dout, drow, dq_acc, rows);
    else bwd_prep_kernel<128, false><<<blocks, 256, 0, stream>>>(o, dout, drow, dq_acc, rows);
  } else if (d == 256) {
    if (f16) bwd_prep_kernel<256, true><<<blocks, 256, 0, stream>>>(o, dout, drow, dq_acc, rows);
    else bwd_prep_kernel<256, false><<<blocks, 256, 0, stream>>>(o, dout, drow, dq_acc, rows);
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
