// attn_fwd.cuh -- fused exact attention forward for sm_103a (tcgen05 + TMEM +
// TMA), one template for BF16 / FP16 / FP8-E4M3 operands.
//
// What it computes (per query row i of head (b,h)):
//   S_ij = scale * q_i . k_j  (FP8: times the Q-block and K-block descales),
//   O_i  = sum_j softmax_j(S_i.) v_j,   LSE_i = ln sum_j exp(S_ij),
// by the online-softmax recurrence over 128-key tiles: running maximum m,
// running sum l and an fp32 accumulator o that is rescaled by exp(m_old -
// m_new) whenever m moves, O = o / l at the end (wmrh.cn FlashAttention V3
// article, sec. 2.1; "FlashAttention-3: async pipelines on Hopper", section
// "Online Softmax is still the core of exact merging").  The N x N scores
// live only in tensor memory, one 128 x 128 tile at a time.
//
// CTA organisation (warp-specialised roles, chosen for Blackwell rather than
// the Hopper producer / consumer-warpgroup split of the pages):
//   * load warp    one thread issues TMA copies: the Q tile(s) once, then K
//                  and V tiles through an NS-slot shared-memory ring with
//                  full/empty mbarriers ("FlashAttention-3: async pipelines
//                  on Hopper", section "first overlap: producer and consumer
//                  in parallel": stage = j mod s, two states per stage).
//   * MMA warp     runs in step; one elected lane issues every tcgen05.mma:
//                  S = Q K^T into TMEM, then O += P V with P read from TMEM;
//                  it also allocates TMEM.
//   * softmax      one warpgroup per Q tile, one thread per query row: reads
//                  S from TMEM, masks, takes the row max, rescales O in TMEM
//                  when the max moved by more than TAU (exact: o, l, m stay
//                  consistent), writes P back into TMEM over S, keeps l; at
//                  the end divides by l and stores O and LSE.
// With two Q tiles per CTA (d <= 128) the MMA warp interleaves the two
// tiles, so the tensor core works on one tile's GEMMs while the other tile's
// softmax runs (the Blackwell form of the pages' ping-pong of two consumer
// warpgroups, section "second overlap").  With one Q tile (d = 256) S is
// double-buffered in TMEM and Q K_{j+1}^T runs during softmax j (the pages'
// intra-warpgroup two-stage pipeline, section "third overlap").
// Causal: key tiles above the diagonal are never loaded or multiplied; the
// diagonal tile is masked (section "why causal shapes are harder to
// schedule").
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "fa.h"
#include "ptx.cuh"

namespace fa {

enum ElemKind : int { kBF16 = 0, kFP16 = 1, kE4M3 = 2 };

constexpr int kBM = 128;  // query rows per Q tile (= TMEM lanes)
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kSmemLimit = 232448;

// Variants (compile-time bits; 0 is the kernel the library ships).  Each
// bit turns one design choice back into a simpler form, or tries an
// alternative, for ablation builds that time what the choice is worth.
enum : int {
  kVarSplitSoftmax = 1,    // two softmax warpgroups per Q tile, 64 key columns each (measured slower)
  kVarEagerRescale = 2,    // rescale O whenever a row maximum rises (no lazy threshold)
  kVarWholeP = 4,          // hand P to the MMA warp in one piece instead of two halves
  kVarOneTile = 8,         // one Q tile per CTA (S double-buffered) also for d <= 128
  kVarNoSteal = 16,        // no work stealing: every CTA runs only the unit it was launched with
  kVarSepP = 32,           // P in its own tensor-memory columns (d = 64, two Q tiles): Q K^T(j+1) may
                           // start once the softmax has read S(j)
  kVarPoly = 64,           // a share of P's exponentials by a polynomial on the FMA pipe (measured slower)
  kVarEarlyQK = 128,       // two Q tiles, P over S: the part of the next Q K^T whose S columns P does not
                           // use is issued when the first half of P arrives, the rest after the second half
                           // (measured slower: an MMA with N = 64 runs at 2/3 of the N = 128 rate)
  kVarDirectStore = 256,   // O written by each lane to its own row with vector stores (no staging in
                           // shared memory, no bulk tensor copy; all ring slots kept)
};

template <int ELEM, int D, bool CAUSAL, int VAR = 0>
struct AttnCfg {
  static constexpr int ES = (ELEM == kE4M3) ? 1 : 2;           // bytes per element
  static constexpr int MMA_KIND = (ELEM == kE4M3) ? 1 : 0;     // kind::f16 or kind::f8f6f4
  static constexpr int ROW_BYTES = D * ES;
  static_assert(ROW_BYTES % 128 == 0, "rows must be a multiple of the 128-byte swizzle span");
  static constexpr int CH_ELEMS = 128 / ES;                    // elements per 128-byte chunk
  static constexpr int NCH = ROW_BYTES / 128;                  // chunks per row
  static constexpr int CHUNK_BYTES = 128 * 128;                // 128 rows x 128 bytes
  static constexpr int NQT = (D <= 128 && !(VAR & kVarOneTile)) ? 2 : 1;  // Q tiles per CTA
  // Softmax warpgroups per Q tile: with two, each thread owns 64 of a row's
  // 128 key columns and the two halves of a row exchange their maxima
  // through shared memory (double-buffered on the tile count).
  static constexpr int CSPLIT = (NQT == 2 && (VAR & kVarSplitSoftmax)) ? 2 : 1;
  static constexpr int SCOLS = kBN / CSPLIT;                   // key columns per softmax thread
  static constexpr int XCH_BYTES = (CSPLIT == 2) ? 2 * 2 * 2 * 128 * 4 : 0;  // [parity][tile][part][row]
  static constexpr int TILE_BYTES = kBN * ROW_BYTES;           // one K or V tile
  static constexpr int SLOT_BYTES = TILE_BYTES < 32768 ? TILE_BYTES : 32768;
  static constexpr int SPT = TILE_BYTES / SLOT_BYTES;          // ring slots per tile
  static constexpr int SLOT_CH = SLOT_BYTES / CHUNK_BYTES;     // chunks per slot
  static constexpr int SLOT_D = SLOT_CH * CH_ELEMS;            // head-dim columns per slot
  static constexpr int Q_BYTES = NQT * kBM * ROW_BYTES;
  // Epilogue: each softmax warp converts 64 columns of its 32 rows of O at a
  // time into a 4 KB staging box (128-byte rows, 128-byte swizzle) and one
  // lane writes the box to global memory with a bulk tensor copy, so that the
  // O writes are whole lines, asynchronous, and cost the warps one shared
  // memory pass instead of scattered 32-byte stores to 32 rows per
  // instruction.  At d = 128 (16-bit) the boxes take one of the five ring
  // slots (measured: mid +2%, long causal +1%, N = 512 +11%, N = 16384 -0.3%);
  // d = 256 (one Q tile, four softmax warps) keeps its five slots and stores
  // directly (with the boxes and four slots it was 2.5% slower).
  static constexpr bool EPI_TMA = (CSPLIT == 1) && (D <= 128) && !(VAR & kVarDirectStore);
  static constexpr int EPI_BOX_COLS = 64;
  static constexpr int EPI_WARP_BYTES = 32 * EPI_BOX_COLS * 2;
  static constexpr int EPI_BYTES = EPI_TMA ? 4 * NQT * EPI_WARP_BYTES : 0;
  static constexpr int NS_MAX = (kSmemLimit - 1024 - 1024 - XCH_BYTES - EPI_BYTES - Q_BYTES) / SLOT_BYTES;
  static constexpr int NS = NS_MAX > 8 ? 8 : NS_MAX;           // ring depth
  static_assert(NS >= 2 * SPT, "ring too shallow");
  static constexpr int KSTEP = 32 / ES;                        // MMA K per instruction (32 bytes)
  static constexpr int KSTEPS_QK = D / KSTEP;
  static constexpr int KSTEPS_PV = kBN / KSTEP;
  static_assert(KSTEPS_PV % 2 == 0, "P is handed over in two halves of the key tile");
  static constexpr int P_COLS = kBN * ES / 4;                  // TMEM columns of P per row
  // P of key half h starts at column h * P_HALF_OFF of the S/P buffer: right
  // after the first half normally; with the split softmax at column 64, the
  // first column of the S columns its own warps read, so that no part's P
  // lands on S columns the other part has still to read.
  static constexpr int P_HALF_OFF = (CSPLIT == 2) ? 64 : P_COLS / 2;
  static constexpr uint32_t TMEM_COLS = 512;
  // Separate P (two Q tiles, when S, P and O of both fit): S_t at 128 t,
  // P_t after both S buffers, O_t after both P buffers.  Otherwise P is
  // written over S (same columns).
  static constexpr bool SEPP = (VAR & kVarSepP) && NQT == 2 && CSPLIT == 1 &&
                               2 * (kBN + P_COLS + D) <= (int)TMEM_COLS;
  static constexpr uint32_t S_COL0 = 0;                        // S buffers at 0 and 128
  static constexpr uint32_t P_COL0 = SEPP ? 2 * kBN : 0;       // P buffers (SEPP) or P over S
  static constexpr uint32_t O_COL0 = SEPP ? 2 * kBN + 2 * P_COLS : 256;  // O accumulators
  static_assert(O_COL0 + NQT * D <= TMEM_COLS, "TMEM budget");
  static constexpr int SOFTMAX_WARPS = 4 * NQT * CSPLIT;
  static constexpr int MMA_WARP = SOFTMAX_WARPS;
  static constexpr int LOAD_WARP = SOFTMAX_WARPS + 1;
  // Two Q tiles: a third, control warpgroup (MMA warp, load warp, two idle
  // warps) so that registers can move between whole warpgroups: launched
  // at LAUNCH_REGS, the control warpgroup drops to CTRL_REGS and the softmax
  // warpgroups rise to SOFTMAX_REGS (their sum stays within the launch
  // total).  One Q tile: 6 warps, no reallocation needed.  The 16-bit
  // kernels' warp-wide MMA loop spills below ~100 registers and their
  // softmax fits in 200 (measured fastest of 72/216, 88/208, 104/200); the
  // FP8 softmax is the tighter side and keeps 216.
  static constexpr bool REALLOC = (NQT == 2 && CSPLIT == 1);
  static constexpr int THREADS = REALLOC ? 32 * (SOFTMAX_WARPS + 4) : 32 * (SOFTMAX_WARPS + 2);
  // Split softmax: 18 warps (16 softmax, MMA, load), up to 5 per
  // sub-partition, so at most 96 registers each, without reallocation.
  static constexpr int LAUNCH_REGS = (CSPLIT == 2) ? 96 : 168;
  static constexpr int CTRL_REGS = (CSPLIT == 2) ? 96 : (ELEM == kE4M3) ? 72 : 104;
  static constexpr int SOFTMAX_REGS = (CSPLIT == 2) ? 96 : (ELEM == kE4M3) ? 216 : 200;
  static_assert(!REALLOC || 128 * CTRL_REGS + SOFTMAX_WARPS * 32 * SOFTMAX_REGS <= THREADS * LAUNCH_REGS,
                "register split exceeds the launch budget");
  // lazy-rescale threshold (log2 units): p <= 2^TAU against the running max.
  // FP8 takes the largest TAU its P range allows (below): each rescale reads
  // and writes all of O in TMEM on the softmax's own chain, and at TAU = 2
  // rescales cost FP8 about 12% (measured).
  static constexpr float TAU = (VAR & kVarEagerRescale) ? 0.0f : (ELEM == kE4M3) ? 3.8f : 8.0f;
  // Exponentials of P: POLY of every 8 pairs by the FMA-pipe polynomial
  // (ex2_poly2, degree POLY_DEG), the rest by MUFU ex2.  Off in the shipped
  // kernels: the softmax of a tile is a chain of dependent steps, not a
  // saturated special-function unit, and every 1/8 of the exponentials moved
  // onto the FMA pipe lengthened it (5-10% slower per 1/8, measured on
  // bf16 d = 64 / 128 and FP8).  fp16 P (11-bit significand) would take the
  // degree-4 polynomial.
  static constexpr int POLY = !(VAR & kVarPoly) ? 0 : (ELEM == kE4M3) ? 3 : (D <= 64) ? 3 : 1;
  static constexpr int POLY_DEG = (ELEM == kFP16) ? 4 : 3;
  static constexpr bool poly_pair(int k) { return ((k % 8 + 1) * POLY) / 8 > ((k % 8) * POLY) / 8; }
  // FP8: P is stored as p * 2^5 * (s_Vj / max_j s_Vj) <= 2^5 * 2^TAU < 446,
  // inside the E4M3 range (448).  The scale sets where small p reach E4M3's
  // subnormals (p below 2^-11); 2^5 against 2^6 left the O error of the FP8
  // workloads unchanged (measured) and lets TAU rise from 2.8 to 3.8.
  static constexpr float P8_SCALE = 32.0f;
  // short units' masked tiles without the per-score select (see the softmax)
  static constexpr bool MASK_NOSEL = (ELEM != kE4M3) && (D == 128 || CAUSAL);
  static_assert(ELEM != kE4M3 || TAU <= 3.807f, "FP8 P would leave the E4M3 range: 32 * 2^TAU must stay <= 448");
  static constexpr uint32_t A_FMT = (ELEM == kBF16) ? 1u : 0u;  // bf16=1, f16=0, e4m3=0
  static constexpr uint32_t IDESC_QK = instr_desc(A_FMT, A_FMT, 0, 0, 128, kBN);
  // Early Q K^T: keys QK_SPLIT.. of the next tile land on S columns that P
  // (written over S from column 0) never uses.
  static constexpr bool EARLY_QK = (VAR & kVarEarlyQK) && NQT == 2 && CSPLIT == 1 && !SEPP && !(VAR & kVarWholeP);
  static constexpr int QK_SPLIT = P_COLS;
  static_assert(!EARLY_QK || (QK_SPLIT % 16 == 0 && QK_SPLIT < kBN), "MMA N must be a multiple of 16");
  static constexpr uint32_t IDESC_QK_LO = instr_desc(A_FMT, A_FMT, 0, 0, 128, QK_SPLIT);
  static constexpr uint32_t IDESC_QK_HI = instr_desc(A_FMT, A_FMT, 0, 0, 128, kBN - QK_SPLIT);
  static constexpr uint32_t IDESC_PV = instr_desc(A_FMT, A_FMT, 0, 1, 128, SLOT_D);
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = Q_BYTES;
  static constexpr int OFF_XCH = OFF_RING + NS * SLOT_BYTES;
  static constexpr int OFF_EPI = OFF_XCH + XCH_BYTES;
  static_assert(OFF_EPI % 1024 == 0, "the 128-byte swizzle of the staging boxes needs 1024-byte alignment");
  static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 1024 + 1024;  // + barriers + alignment slack
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory budget");
};

struct AttnParams {
  void* o;              // [BH, N, D] bf16 / f16 (FP8 path: bf16)
  float* lse;           // [BH, N]
  const float* q_ds;    // FP8 only: [BH, nblk]
  const float* k_ds;
  const float* v_ds;
  int* err;             // device error word
  int N;                // query rows per head (Nq)
  int Nk;               // keys per head
  int BH;               // batch x query heads
  int Hq, Hkv;          // query heads, key/value heads (Hq % Hkv == 0)
  int nblk;             // ceil(Nq / 128): Q descale blocks per head
  int nblk_k;           // ceil(Nk / 128): K/V descale blocks per head
  float scale_log2;     // scale * log2(e)
  int drop_pos;         // test hook: ring position CTA 0 never fills (-1: none)
  // Units [0, pair_units) hold NQT Q tiles each; when pair_units is below
  // the number of such groups, each remaining group is run as NQT units of
  // one Q tile (shorter units for a last, partial wave of SMs).
  int pair_units;
  int o_vec32;          // 1: o is 32-byte aligned (rows are stored 32 bytes at a time)
  // Row r of a head sits at sequence position r % q_period (q_period = N,
  // or Nq when the query heads of a key/value group are packed into one
  // head of g * Nq rows); causal masks use that position.
  int q_period;
  // Causal unit order: heads are taken head_chunk at a time (chunks in
  // head order), and within a chunk the units with the most key tiles come
  // first (longest processing time first).  head_chunk = BH: one chunk.
  int head_chunk;
  // Split-KV: splits > 1 divides each row's key tiles into runs of
  // split_tiles; a unit then covers one run and writes O normalised over its
  // keys (fp32) to o_part[split][bh][row][d] and its LSE to
  // lse_part[split][bh][row], for a separate combine.
  int splits;
  int split_tiles;
  float* o_part;
  float* lse_part;
};

// Barriers in shared memory.
template <int NS>
struct Bars {
  uint64_t q_full;
  uint64_t q_empty;
  uint64_t full[NS];
  uint64_t empty[NS];
  uint64_t s_full[2];
  uint64_t s_free[2];     // separate P: the softmax has read S (the next Q K^T may overwrite it)
  uint64_t p_free[2];     // separate P: P V done (P buffer free, O stable)
  uint64_t p_full[2][2];  // [S/P buffer][half of the key tile]
  uint64_t o_ready[2];
  uint64_t o_full[2];
  uint64_t drain;
  uint64_t clc_bar;        // response of the work-stealing request
  uint64_t unit_full[2];   // queue of next-unit ids (load warp -> others)
  uint64_t unit_empty[2];
  alignas(16) uint32_t clc_resp[4];
  alignas(16) int unit_q[2][8];  // decoded units: {bh (-1: none), kvh, q_base, Jt0 | Jt1 << 16, split, tb, active mask}
  uint32_t tmem_base;
  int abort_flag;
};

// Number of key tiles a Q tile starting at row q0 visits.  Causal masks are
// aligned at the bottom right: key j is visible to query i iff
// j <= i + off with off = Nk - Nq (off = 0 for equal lengths).
template <bool CAUSAL>
__device__ __forceinline__ int kv_tiles_for(int q0, int nkv, int off) {
  if constexpr (CAUSAL) {
    const int last_key = q0 + kBM - 1 + off;  // last key any row of the tile sees
    if (last_key < 0) return 0;
    const int tiles = last_key / kBN + 1;
    return tiles < nkv ? tiles : nkv;
  } else {
    return nkv;
  }
}

// The ring carries K and V tiles in the order the MMA warp consumes them:
//   two Q tiles : K0 V0 K1 V1 ...            (S(j+1) is issued after PV(j))
//   one Q tile  : K0 K1 V0 K2 V1 K3 V2 ...   (S(j+2) is issued after PV(j))

// SPLIT: the split-KV instance: rows may be packed (causal positions modulo
// q_period) and, when prm.splits > 1, units cover runs of key tiles and
// write fp32 partial results.  Without it every row is its own position and
// a unit covers the whole key range.
// Multiplies this thread's OCOLS columns of O in TMEM by alpha.  Taken only
// when a row maximum of the warp rose past the lazy threshold, so it is kept
// out of line: its registers then do not weigh on the softmax's main path
// (measured +1.3% at N = 16384 bf16, neutral elsewhere).
template <int OCOLS>
__device__ __noinline__ void rescale_o_cols(uint32_t o_addr, float alpha) {
#pragma unroll 1
  for (int c0 = 0; c0 < OCOLS; c0 += 32) {
    uint32_t u[32];
    tmem_ld32(o_addr + c0, u);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
    tmem_st32(o_addr + c0, u);
  }
  tmem_wait_st();
}

template <int ELEM, int D, bool CAUSAL, bool SPLIT, int VAR = 0>
__global__ void __launch_bounds__(AttnCfg<ELEM, D, CAUSAL, VAR>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const AttnParams prm) {
  using C = AttnCfg<ELEM, D, CAUSAL, VAR>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars<C::NS>* bars = reinterpret_cast<Bars<C::NS>*>(smem + C::OFF_BAR);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = prm.N;                     // query rows
  const int Nk = prm.Nk;                   // keys
  const int nkv = (Nk + kBN - 1) / kBN;
  const int qgroup = prm.Hq / prm.Hkv;     // query heads per key/value head
  const int n_groups = (N + C::NQT * kBM - 1) / (C::NQT * kBM);
  const int koff = Nk - N;                 // causal diagonal offset (unpacked rows)
  const int S = SPLIT ? prm.splits : 1;  // key splits
  const int U_groups = prm.BH * n_groups * S;  // (head, group of NQT Q tiles, key split)
  // work units: every group, or pair_units groups and the rest as single Q tiles
  const int U = U_groups + (C::NQT - 1) * (U_groups - prm.pair_units);
  const int G = (int)gridDim.x;

  // Work units are launched one CTA each, in this order: non-causal,
  // head-major (the Q-tile groups of a head are adjacent, their K/V re-read
  // from L2); causal, group-major with the heaviest groups (most key tiles)
  // first (longest-processing-time-first).  A CTA that is about to finish
  // its unit takes over the next not-yet-started CTA's unit through cluster
  // launch control, so units flow to whichever SM frees up first and the
  // next unit's loads overlap the current unit's tail.  The load warp makes
  // the request and passes the unit id to the other roles through a
  // two-slot queue in shared memory.
  (void)G;
  struct Unit {
    int bh, kvh, q_base, J;
    int Jt[2];
    bool active[2];
    int split, tb;  // key split and its first key tile
  };
  auto decode = [&](int u) -> Unit {
    Unit w;
    int group;
    w.split = SPLIT ? u % S : 0;
    int v = SPLIT ? u / S : u;
    int single = -1;  // which Q tile of its group a single-tile unit runs
    if (!CAUSAL && !SPLIT && C::NQT == 2 && v >= prm.pair_units) {
      const int x = v - prm.pair_units;
      v = prm.pair_units + x / 2;
      single = x % 2;
    }
    if constexpr (CAUSAL) {
      // heaviest groups first within chunks of head_chunk heads (chunks in
      // head order), so that the K/V of the heads in flight stay in L2
      const int per_chunk = prm.head_chunk * n_groups;
      const int c = v / per_chunk;
      const int idx = v - c * per_chunk;
      const int heads_here = min(prm.head_chunk, prm.BH - c * prm.head_chunk);
      group = n_groups - 1 - idx / heads_here;
      w.bh = c * prm.head_chunk + idx % heads_here;
    } else {
      w.bh = v / n_groups;
      group = v % n_groups;
    }
    w.q_base = group * (C::NQT * kBM) + (single > 0 ? kBM : 0);
    w.tb = SPLIT ? w.split * prm.split_tiles : 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int q0 = w.q_base + t * kBM;
      w.active[t] = (t < C::NQT) && (q0 < N) && (single < 0 || t == 0);
      int tiles = 0;
      if (w.active[t]) {
        if constexpr (CAUSAL && SPLIT) {
          // last key any row of the tile sees, from the largest position
          // among its rows (rows of several packed heads: the last one)
          const int q1 = min(q0 + kBM, N) - 1;
          const int P = prm.q_period;
          const int maxpos = (q1 / P != q0 / P) ? P - 1 : q1 % P;
          tiles = kv_tiles_for<CAUSAL>(maxpos - (kBM - 1), nkv, Nk - P);
        } else if constexpr (CAUSAL) {
          tiles = kv_tiles_for<CAUSAL>(q0, nkv, koff);
        } else {
          tiles = nkv;
        }
      }
      if constexpr (SPLIT) {
        // this split's run of key tiles
        tiles -= w.tb;
        tiles = tiles < 0 ? 0 : (tiles > prm.split_tiles ? prm.split_tiles : tiles);
      }
      w.Jt[t] = tiles;
    }
    w.J = w.Jt[0] > w.Jt[1] ? w.Jt[0] : w.Jt[1];
    w.kvh = (w.bh / prm.Hq) * prm.Hkv + (w.bh % prm.Hq) / qgroup;
    return w;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], 128);
      mbar_init(&bars->p_free[t], 1);
      mbar_init(&bars->p_full[t][0], 128);
      mbar_init(&bars->p_full[t][1], 128);
      mbar_init(&bars->o_ready[t], 1);
      mbar_init(&bars->o_full[t], 1);
    }
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->clc_bar, 1);
    for (int q = 0; q < 2; ++q) {
      mbar_init(&bars->unit_full[q], 1);
      mbar_init(&bars->unit_empty[q], 1 + C::SOFTMAX_WARPS);
    }
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

  // Unit number r of this CTA from the queue (the load warp decodes each
  // unit once and publishes it; bh < 0 means no more units), then release
  // the slot.  `arrive` is done by one lane per warp.
  auto fetch_unit = [&](int r, bool arrive, bool& okr) -> Unit {
    Unit w;
    const int slot = r & 1;
    okr = mbar_wait(&bars->unit_full[slot], (uint32_t)((r >> 1) & 1), abort_flag, prm.err);
    volatile int* qv = reinterpret_cast<volatile int*>(&bars->unit_q[slot][0]);
    const int4 v = make_int4(qv[0], qv[1], qv[2], qv[3]);
    w.split = SPLIT ? qv[4] : 0;
    w.tb = SPLIT ? qv[5] : 0;
    const int act = qv[6];
    if (arrive) mbar_arrive(&bars->unit_empty[slot]);
    w.bh = okr ? v.x : -1;
    w.kvh = v.y;
    w.q_base = v.z;
    w.Jt[0] = v.w & 0xffff;
    w.Jt[1] = (v.w >> 16) & 0xffff;
    w.J = w.Jt[0] > w.Jt[1] ? w.Jt[0] : w.Jt[1];
    w.active[0] = (act & 1) != 0;
    w.active[1] = (act & 2) != 0;
    return w;
  };
  // the load warp's side: publish unit r (u < 0: no more units)
  auto publish_unit = [&](int r, int u) -> bool {
    const int slot = r & 1;
    if (r >= 2 && !mbar_wait(&bars->unit_empty[slot], (uint32_t)(((r - 2) >> 1) & 1), abort_flag, prm.err))
      return false;
    int4 v = make_int4(-1, 0, 0, 0);
    int split = 0, tb = 0, act = 0;
    if (u >= 0) {
      const Unit w = decode(u);
      v = make_int4(w.bh, w.kvh, w.q_base, w.Jt[0] | (w.Jt[1] << 16));
      split = w.split;
      tb = w.tb;
      act = (w.active[0] ? 1 : 0) | (w.active[1] ? 2 : 0);
    }
    volatile int* qv = reinterpret_cast<volatile int*>(&bars->unit_q[slot][0]);
    qv[0] = v.x;
    qv[1] = v.y;
    qv[2] = v.z;
    qv[3] = v.w;
    qv[4] = split;
    qv[5] = tb;
    qv[6] = act;
    mbar_arrive(&bars->unit_full[slot]);
    return true;
  };

  if (warp >= C::SOFTMAX_WARPS) {
    // control warpgroup: give registers to the softmax warpgroups
    if constexpr (C::REALLOC) regs_dec<C::CTRL_REGS>();
  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------------------ load --
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_kv = policy_evict_last();
      const uint64_t pol_q = policy_evict_first();
      int pos = 0;     // ring position (continues across units)
      int k = 0;       // units loaded by this CTA
      int n_req = 0;   // work-stealing requests made
      bool more = true;
      bool ok = true;
      int u = (int)blockIdx.x;
      ok = publish_unit(0, u);
      for (int r = 0; ok && u >= 0; ++r) {
        const Unit w = decode(u);
        if (w.J > 0) {  // (a unit whose rows see no key needs no loads)
        // the Q buffer is free once the previous unit's last Q K^T finished
        if (k > 0 && !mbar_wait(&bars->q_empty, (uint32_t)((k - 1) & 1), abort_flag, prm.err)) { ok = false; break; }
        uint32_t qbytes = 0;
        for (int t = 0; t < C::NQT; ++t) qbytes += w.Jt[t] > 0 ? (uint32_t)(kBM * C::ROW_BYTES) : 0u;
        mbar_arrive_expect_tx(&bars->q_full, qbytes);
        for (int t = 0; t < C::NQT; ++t) {
          if (w.Jt[t] == 0) continue;
          for (int ch = 0; ch < C::NCH; ++ch)
            tma_load_3d_hint(smem + C::OFF_Q + (t * C::NCH + ch) * C::CHUNK_BYTES, &tm_q, &bars->q_full,
                             ch * C::CH_ELEMS, w.q_base + t * kBM, w.bh, pol_q);
        }
        // one K or V tile (SPT ring slots) into the ring
        auto load_tile = [&](bool is_v, int j) {
          const CUtensorMap* map = is_v ? &tm_v : &tm_k;
          for (int sp = 0; sp < C::SPT && ok; ++sp, ++pos) {
            const int slot = pos % C::NS;
            const uint32_t ph = (uint32_t)((pos / C::NS) & 1);
            if (!mbar_wait(&bars->empty[slot], ph ^ 1u, abort_flag, prm.err)) { ok = false; break; }
            // failure-injection hook (tests only): this slot is never filled,
            // so the MMA warp's wait on it runs out and the kernel aborts
            if (pos == prm.drop_pos && blockIdx.x == 0) continue;
            mbar_arrive_expect_tx(&bars->full[slot], C::SLOT_BYTES);
            for (int ch = 0; ch < C::SLOT_CH; ++ch)
              tma_load_3d_hint(smem + C::OFF_RING + slot * C::SLOT_BYTES + ch * C::CHUNK_BYTES, map,
                               &bars->full[slot], (sp * C::SLOT_CH + ch) * C::CH_ELEMS, (w.tb + j) * kBN, w.kvh,
                               pol_kv);
          }
        };
        if constexpr (C::NQT == 2) {
          for (int j = 0; j < w.J && ok; ++j) {
            load_tile(false, j);
            load_tile(true, j);
          }
        } else {
          for (int j = 0; j < w.J && j < 2 && ok; ++j) load_tile(false, j);
          for (int j = 0; j < w.J && ok; ++j) {
            load_tile(true, j);
            if (j + 2 < w.J) load_tile(false, j + 2);
          }
        }
        ++k;
        }
        if (!ok) break;
        // every load of this unit is issued: claim the next unit
        int nu = -1;
        if (more && !(VAR & kVarNoSteal)) {
          mbar_arrive_expect_tx(&bars->clc_bar, 16);
          clc_try_cancel(bars->clc_resp, &bars->clc_bar);
          if (!mbar_wait(&bars->clc_bar, (uint32_t)(n_req & 1), abort_flag, prm.err)) { ok = false; break; }
          ++n_req;
          nu = clc_query_x(bars->clc_resp);
          if (nu < 0 || nu >= U) { nu = -1; more = false; }
        }
        // publish it as unit r+1 (its slot is reused once the others read unit r-1)
        if (!publish_unit(r + 1, nu)) {
          ok = false;
          break;
        }
        u = nu;
      }
      // Never leave with copies in flight: wait (bounded) for the last fill
      // of every slot that was used, and for the last Q tile.
      const int used = pos < C::NS ? pos : C::NS;
      for (int i = 0; i < used; ++i) {
        const int p_last = pos - 1 - i;
        const int slot = p_last % C::NS;
        const uint32_t ph = (uint32_t)((p_last / C::NS) & 1);
        uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&bars->full[slot], ph) && globaltimer() - t0 < FA_WAIT_LIMIT_NS) {
        }
      }
      if (k > 0) {
        uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&bars->q_full, (uint32_t)((k - 1) & 1)) && globaltimer() - t0 < FA_WAIT_LIMIT_NS) {
        }
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------- MMA --
    // The whole warp runs the issuing loop in step, so that its counters,
    // ring positions and descriptors are warp-uniform; each tcgen05.mma and
    // commit is issued by one elected lane.  A single diverged lane running
    // the same loop spends nearly a 128x128x16 step's tensor time on issuing
    // each MMA, so every wait and commit beside them starves the pipe.
    {
      const uint32_t q_s = smem_u32(smem + C::OFF_Q);
      const uint32_t ring_s = smem_u32(smem + C::OFF_RING);
      int pos = 0;          // ring position of the next item to consume
      int k = 0;            // units processed
      int pc[2] = {0, 0};   // two Q tiles: P handshakes consumed per tile
      int nqk[2] = {0, 0};  // separate P: Q K^T issued per tile (s_free phase of the previous one)
      int g = 0;            // one Q tile: S/P iterations so far (buffer = g & 1)
      bool ok = true;
      // every lane waits; the outcome is made uniform across the warp
      auto warp_wait = [&](uint64_t* bar, uint32_t parity, volatile int* af, int* ew) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, af, ew));
      };

      // wait for a whole tile (SPT slots) at the current ring position
      auto wait_tile = [&](int p) -> bool {
        for (int sp = 0; sp < C::SPT; ++sp) {
          const int slot = (p + sp) % C::NS;
          if (!warp_wait(&bars->full[slot], (uint32_t)(((p + sp) / C::NS) & 1), abort_flag, prm.err))
            return false;
        }
        tc_fence_after();
        return true;
      };
      auto release_tile = [&](int p) {
        for (int sp = 0; sp < C::SPT; ++sp) mma_commit_elect(&bars->empty[(p + sp) % C::NS]);
      };
      // S_buf = Q_t K^T for the K tile at ring position p
      // Descriptors are built once and advanced per K step by adding the
      // step's byte offset >> 4 to the start-address field (bits 0..13; all
      // shared addresses are below 256 KB, so the field cannot overflow):
      // the issuing thread then spends a single add per operand per MMA.
      const uint64_t q_desc0 = smem_desc(q_s, 16, 1024, 2);                 // Q tiles, K-major
      const uint64_t ring_k_desc0 = smem_desc(ring_s, 16, 1024, 2);         // K slots, K-major
      const uint64_t ring_v_desc0 = smem_desc(ring_s, C::CHUNK_BYTES, 1024, 2);  // V slots, MN-major
      auto slot_of = [&](int p) -> uint32_t { return (uint32_t)(p % C::NS); };
      // S_buf = Q_t K^T for the K tile at ring position p; part 0: all keys,
      // part 1: keys 0 .. QK_SPLIT-1, part 2: keys QK_SPLIT .. kBN-1
      auto issue_qk = [&](int t, int buf, int p, int part = 0) {
        const int key0 = (part == 2) ? C::QK_SPLIT : 0;
        const uint32_t idesc = (part == 0) ? C::IDESC_QK : (part == 1) ? C::IDESC_QK_LO : C::IDESC_QK_HI;
        const uint32_t d_tmem = tmem + C::S_COL0 + buf * kBN + key0;
        const uint64_t a0 = q_desc0 + (uint64_t)((t * C::NCH * C::CHUNK_BYTES) >> 4);
        uint64_t b0[C::SPT];
#pragma unroll
        for (int sp = 0; sp < C::SPT; ++sp)
          b0[sp] = ring_k_desc0 + (uint64_t)((slot_of(p + sp) * C::SLOT_BYTES + key0 * 128) >> 4);
#pragma unroll
        for (int ks = 0; ks < C::KSTEPS_QK; ++ks) {
          const int byte_k = ks * 32;                         // byte offset along the row
          const int ch = byte_k / 128;
          const int in_ch = byte_k % 128;
          const int sp = ch / C::SLOT_CH;                     // which slot of the tile
          const int ch_in_slot = ch % C::SLOT_CH;
          const uint64_t a = a0 + (uint64_t)((ch * C::CHUNK_BYTES + in_ch) >> 4);
          const uint64_t b = b0[sp] + (uint64_t)((ch_in_slot * C::CHUNK_BYTES + in_ch) >> 4);
          mma_ss_elect<C::MMA_KIND>(d_tmem, a, b, idesc, ks > 0 ? 1u : 0u);
        }
      };
      // O_t (+)= P_buf V for half h of the keys of the V tile at ring position p
      auto issue_pv = [&](int t, int buf, int p, bool acc, int h) {
        const uint32_t p_tmem = tmem + C::P_COL0 + buf * (C::SEPP ? C::P_COLS : kBN);
#pragma unroll
        for (int sp = 0; sp < C::SPT; ++sp) {
          const uint32_t d_tmem = tmem + C::O_COL0 + t * D + sp * C::SLOT_D;
          const uint64_t v0 = ring_v_desc0 + (uint64_t)((slot_of(p + sp) * C::SLOT_BYTES) >> 4);
#pragma unroll
          for (int ks = h * (C::KSTEPS_PV / 2); ks < (h + 1) * (C::KSTEPS_PV / 2); ++ks) {
            // keys ks*KSTEP .. +KSTEP-1 are KSTEP/8 groups of 8 rows (1024 B each)
            const uint64_t b = v0 + (uint64_t)((ks * (C::KSTEP / 8) * 1024) >> 4);
            const uint32_t p_col = (uint32_t)(h * C::P_HALF_OFF + (ks - h * (C::KSTEPS_PV / 2)) * 8);
            mma_ts_elect<C::MMA_KIND>(d_tmem, p_tmem + p_col, b, C::IDESC_PV, (acc || ks > 0) ? 1u : 0u);
          }
        }
      };

      for (int r = 0; ok; ++r) {
        const Unit w = fetch_unit(r, lane == 0, ok);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok || w.bh < 0) break;
        if (w.J > 0) {  // (a unit whose rows see no key needs no MMA)
        ok = warp_wait(&bars->q_full, (uint32_t)(k & 1), abort_flag, prm.err);
        if (!ok) break;
        tc_fence_after();
        // the Q buffer is released after this unit's last Q K^T
        int qk_left = w.Jt[0] + w.Jt[1];
        auto qk_issued = [&]() {
          if (--qk_left == 0) mma_commit_elect(&bars->q_empty);
        };
        if constexpr (C::NQT == 2 && C::SEPP) {
          // Separate P: S_t(j+1) is computed as soon as the softmax has read
          // S_t(j) (s_free), while it still works on P_t(j); P V_t(j) then
          // follows from the P buffer.  p_free tells the softmax that P V_t(j)
          // is done (O stable, P buffer free); the unit's last P V commits
          // o_full instead.
          auto qk_next = [&](int t, int p) -> bool {
            if (nqk[t] > 0) {
              if (!warp_wait(&bars->s_free[t], (uint32_t)((nqk[t] - 1) & 1), abort_flag, prm.err)) return false;
              tc_fence_after();
            }
            issue_qk(t, t, p);
            mma_commit_elect(&bars->s_full[t]);
            qk_issued();
            ++nqk[t];
            return true;
          };
          ok = wait_tile(pos);
          if (!ok) break;
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (ok && w.Jt[t] > 0) ok = qk_next(t, pos);
          if (!ok) break;
          release_tile(pos);
          pos += C::SPT;
          for (int j = 0; j < w.J && ok; ++j) {
            const int pv_pos = pos;            // V_j
            const int k_pos = pos + C::SPT;    // K_{j+1}
            if (j + 1 < w.J) {
              ok = wait_tile(k_pos);
              if (!ok) break;
#pragma unroll
              for (int t = 0; t < 2; ++t)
                if (ok && j + 1 < w.Jt[t]) ok = qk_next(t, k_pos);
              if (!ok) break;
            }
            ok = wait_tile(pv_pos);
            if (!ok) break;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (!ok) break;
              if (j >= w.Jt[t]) continue;
#pragma unroll
              for (int h = 0; h < 2 && ok; ++h) {
                ok = warp_wait(&bars->p_full[t][h], (uint32_t)(pc[t] & 1), abort_flag, prm.err);
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, t, pv_pos, j > 0, h);
              }
              ++pc[t];
              if (!ok) break;
              mma_commit_elect(j + 1 < w.Jt[t] ? &bars->p_free[t] : &bars->o_full[t]);
            }
            if (!ok) break;
            release_tile(pv_pos);
            pos += C::SPT;
            if (j + 1 < w.J) {
              release_tile(k_pos);
              pos += C::SPT;
            }
          }
        } else if constexpr (C::NQT == 2) {
          // prologue: S_t(0) for both tiles
          ok = wait_tile(pos);
          if (!ok) break;
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (w.Jt[t] > 0) {
              issue_qk(t, t, pos);
              mma_commit_elect(&bars->s_full[t]);
              qk_issued();
            }
          release_tile(pos);
          pos += C::SPT;
          for (int j = 0; j < w.J && ok; ++j) {
            const int pv_pos = pos;            // V_j
            const int k_pos = pos + C::SPT;    // K_{j+1}
            bool v_ready = false, k_ready = false;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (!ok) break;
              if (j >= w.Jt[t]) continue;
              if (!v_ready) { ok = wait_tile(pv_pos); v_ready = true; if (!ok) break; }
              // P arrives in two halves of the key tile: the first half's
              // MMAs run while the softmax still writes the second
#pragma unroll
              for (int h = 0; h < 2 && ok; ++h) {
                ok = warp_wait(&bars->p_full[t][h], (uint32_t)(pc[t] & 1), abort_flag, prm.err);
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, t, pv_pos, j > 0, h);
                if (C::EARLY_QK && h == 0 && j + 1 < w.Jt[t]) {
                  // the softmax has read all of S(j): the S columns that P
                  // does not use can take their part of S(j+1) now
                  if (!k_ready) { ok = wait_tile(k_pos); k_ready = true; if (!ok) break; }
                  issue_qk(t, t, k_pos, 2);
                }
              }
              ++pc[t];
              if (!ok) break;
              if (j + 1 < w.Jt[t]) {
                if (!k_ready) { ok = wait_tile(k_pos); k_ready = true; if (!ok) break; }
                issue_qk(t, t, k_pos, C::EARLY_QK ? 1 : 0);
                mma_commit_elect(&bars->s_full[t]);
                qk_issued();
              } else {
                mma_commit_elect(&bars->o_full[t]);
              }
            }
            if (!ok) break;
            release_tile(pv_pos);
            pos += C::SPT;
            if (j + 1 < w.J) {
              release_tile(k_pos);
              pos += C::SPT;
            }
          }
        } else {
          // one Q tile, S double-buffered: S(0), S(1), then PV(j), S(j+2);
          // buffers alternate on the running iteration count g
          const int Jn = w.Jt[0];
          for (int j = 0; j < 2 && j < Jn && ok; ++j) {
            ok = wait_tile(pos);
            if (!ok) break;
            issue_qk(0, (g + j) & 1, pos);
            mma_commit_elect(&bars->s_full[(g + j) & 1]);
            qk_issued();
            release_tile(pos);
            pos += C::SPT;
          }
          for (int j = 0; j < Jn && ok; ++j) {
            const int gj = g + j;
            const int b = gj & 1;
            ok = wait_tile(pos);  // V_j
            if (!ok) break;
#pragma unroll
            for (int h = 0; h < 2 && ok; ++h) {
              ok = warp_wait(&bars->p_full[b][h], (uint32_t)((gj >> 1) & 1), abort_flag, prm.err);
              if (!ok) break;
              tc_fence_after();
              issue_pv(0, b, pos, j > 0, h);
            }
            if (!ok) break;
            mma_commit_elect(&bars->o_ready[b]);
            release_tile(pos);
            pos += C::SPT;
            if (j + 2 < Jn) {
              ok = wait_tile(pos);  // K_{j+2}
              if (!ok) break;
              issue_qk(0, b, pos);
              mma_commit_elect(&bars->s_full[b]);
              qk_issued();
              release_tile(pos);
              pos += C::SPT;
            }
          }
          if (ok) mma_commit_elect(&bars->o_full[0]);
          g += Jn;
        }
        ++k;
        }
      }
      // drain: every MMA issued by this thread has completed before TMEM is freed
      mma_commit_elect(&bars->drain);
      uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&bars->drain, 0) && globaltimer() - t0 < FA_WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  }
  // (any further warps of the control warpgroup have no role)
  } else {
    // --------------------------------------------------------- softmax --
    if constexpr (C::REALLOC) regs_inc<C::SOFTMAX_REGS>();
    constexpr int NCOL = C::SCOLS;                  // key columns of a tile per thread
    const int t = warp / (4 * C::CSPLIT);           // Q tile of this warp
    const int part = (warp / 4) % C::CSPLIT;        // which NCOL key columns (split softmax)
    const int cbase = part * NCOL;                  // first of them within a key tile
    const int wq = warp % 4;                        // TMEM lane quarter
    const int r_in = wq * 32 + lane;                // row within the tile
    const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
    // Split softmax: the two warps holding the two column parts of the same
    // 32 rows meet at their own named barrier (1..8), always through the
    // predicate-AND form, so that a warp that gave up never leaves its
    // partner waiting; row maxima and row sums cross through shared memory
    // (slot parity alternates with the tile count, so a slot is rewritten
    // only after the partner has passed the next barrier).
    const uint32_t pair_bar = 1u + (uint32_t)(t * 4 + wq);
    float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);
    auto xslot = [&](int parity, int prt) -> float* { return xch + ((parity * 2 + t) * 2 + prt) * 128 + r_in; };
    const bool neg = prm.scale_log2 < 0.0f;
    const float mask_val = neg ? INFINITY : -INFINITY;
    int sc = 0;               // two Q tiles: S handshakes consumed (this tile)
    int g = 0;                // one Q tile: running iteration count
    int oc = 0;               // units finished by this tile (o_full phases)
    int pv_seen = 0;          // one Q tile: PV completions consumed (global iteration order)
    int xc = 0;               // split softmax: exchanges made (slot parity)
    int pfw = 0;              // separate P: p_free phases consumed (this tile)
    bool ok = true;

    for (int rr = 0; ok; ++rr) {
      bool okr = true;
      const Unit w = fetch_unit(rr, lane == 0, okr);
      okr = __all_sync(0xffffffffu, okr);
      // the two column parts of a row agree on going on, so that neither
      // waits at their barrier for a partner that has left
      if constexpr (C::CSPLIT == 2) okr = bar_and(pair_bar, 64, okr);
      if (!okr) { ok = false; break; }
      if (w.bh < 0) break;
      do {  // one unit (skipped when this tile lies beyond N)
      if (!(t == 0 ? w.active[0] : w.active[1])) break;
      const int bh = w.bh;
      const int q0 = w.q_base + t * kBM;
      const int row = q0 + r_in;
      const int Jn = (t == 0) ? w.Jt[0] : w.Jt[1];
      // output columns of this thread: all D, or its part's half
      constexpr int OCOLS = D / C::CSPLIT;
      const int ocol0 = part * OCOLS;
      if (Jn == 0) {
        // no row of this tile sees a key of this unit (causal, Nq > Nk, or a
        // key split beyond the tile's last key): O = 0, LSE = -inf
        if (row < N) {
          if (SPLIT && S > 1) {
            const size_t pr = ((size_t)w.split * prm.BH + bh) * N + row;
            float4* dst = reinterpret_cast<float4*>(prm.o_part + pr * D + ocol0);
#pragma unroll 1
            for (int i = 0; i < OCOLS / 4; ++i) dst[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (part == 0) prm.lse_part[pr] = -INFINITY;
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(prm.o) +
                                                  (((size_t)bh * N + row) * D + ocol0) * 2);
#pragma unroll 1
            for (int i = 0; i < OCOLS / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            if (part == 0) prm.lse[(size_t)bh * N + row] = -INFINITY;
          }
        }
        break;
      }

      // last key this row sees (keys beyond it are masked)
      // and the smallest last-visible key among the tile's rows (causal)
      int last_col = Nk - 1, first_last = q0 + koff;
      if constexpr (CAUSAL && SPLIT) {
        // packed rows: position = row % q_period
        const int P = prm.q_period;
        last_col = min(Nk - 1, row % P + (Nk - P));
        first_last = (min(q0 + kBM, N) - 1) / P != q0 / P ? Nk - P : q0 % P + (Nk - P);
      } else if constexpr (CAUSAL) {
        last_col = min(Nk - 1, row + koff);
      }
      float m_run = -INFINITY;  // reference maximum, log2 units
      float l_run = 0.0f;       // row sum over this thread's key columns
      float v_mult = 1.0f;      // FP8: max_j s_Vj / P8_SCALE
      const int bh_blk = bh * prm.nblk;          // Q descale blocks of this head
      const int kv_blk = w.kvh * prm.nblk_k;     // K/V descale blocks
      float qds = 1.0f, vmax = 1.0f;
      if constexpr (ELEM == kE4M3) {
        qds = prm.q_ds[bh_blk + q0 / kBM];
        // max of the head's V-block descales: lanes take strided blocks
        vmax = 0.0f;
        for (int b = lane; b < prm.nblk_k; b += 32) vmax = fmaxf(vmax, prm.v_ds[kv_blk + b]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
        if (!(vmax > 0.0f)) vmax = 1.0f;
        v_mult = vmax / C::P8_SCALE;
      }
      // FP8 per-tile factors, prepared one tile ahead so that neither the
      // descale loads nor the log / reciprocal sit between S and P.  The
      // single-part softmax forms them for 32 key tiles at once, one tile per
      // lane, and each tile takes its three by a shuffle after P of the tile
      // before has been handed over (measured 3-4% faster than forming them
      // per tile); the split softmax loads tile j+1's descales when S(j)
      // arrives and forms its factors after P(j).
      //   f_k:   q-block descale x k-block descale (multiplies the scale)
      //   f_lpv: log2 of P~'s V-block factor 2^5 * s_Vj / max s_V
      //   f_inv: that factor's reciprocal (undoes it in the row sum)
      float f_k = 1.0f, f_lpv = 0.0f, f_inv = 1.0f;
      float kd_next = 1.0f, vd_next = 1.0f;
      auto fp8_factors = [&](float kd, float vd) {
        f_k = qds * kd;
        const float pv = C::P8_SCALE * (vd / vmax);
        f_lpv = lg2(pv);
        f_inv = 1.0f / pv;
      };
      // single-part softmax: the factors of 32 key tiles at a time, one
      // tile per lane, handed to each tile by a shuffle
      float b_fk = 1.0f, b_lpv = 0.0f, b_inv = 1.0f;
      auto fp8_batch = [&](int jb0) {
        const int jb = jb0 + lane;
        if (jb < Jn) {
          const float kd = prm.k_ds[kv_blk + w.tb + jb], vd = prm.v_ds[kv_blk + w.tb + jb];
          b_fk = qds * kd;
          const float pv = C::P8_SCALE * (vd / vmax);
          b_lpv = lg2(pv);
          b_inv = 1.0f / pv;
        }
      };
      auto fp8_take = [&](int jt) {
        f_k = __shfl_sync(0xffffffffu, b_fk, jt & 31);
        f_lpv = __shfl_sync(0xffffffffu, b_lpv, jt & 31);
        f_inv = __shfl_sync(0xffffffffu, b_inv, jt & 31);
      };
      if constexpr (ELEM == kE4M3) {
        if constexpr (C::CSPLIT == 1) {
          if (Jn > 0) {
            fp8_batch(0);
            fp8_take(0);
          }
        } else {
          if (Jn > 0) fp8_factors(prm.k_ds[kv_blk + w.tb], prm.v_ds[kv_blk + w.tb]);
        }
      }
      // one Q tile: consume o_ready completions up to (and including) the PV
      // of global iteration x on buffer x & 1 (they complete in order)
      auto consume_o = [&](int x) -> bool {
        while (pv_seen <= x) {
          // PV(pv_seen) ran on buffer pv_seen & 1, as that buffer's
          // (pv_seen >> 1)-th completion (one counter, no indexed array)
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_ready[pv_seen & 1], (uint32_t)((pv_seen >> 1) & 1),
                                                 abort_flag, prm.err)))
            return false;
          ++pv_seen;
        }
        return true;
      };


      for (int j = 0; j < Jn && ok; ++j) {
        const int gj = g + j;
        const int buf = (C::NQT == 2) ? t : (gj & 1);
        const uint32_t ph = (C::NQT == 2) ? (uint32_t)(sc & 1) : (uint32_t)((gj >> 1) & 1);
        const bool okw = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[buf], ph, abort_flag, prm.err));
        ++sc;
        if constexpr (C::CSPLIT == 2) {
          // ---- split softmax: this thread's 64 key columns of the tile, read
          // from TMEM twice (once for the row maximum, once for P), 32 at a
          // time, so that few registers are live
          const uint32_t s_addr = tmem + lane_addr + C::S_COL0 + buf * kBN;
          float cj = prm.scale_log2;   // scale of this tile (log2 units)
          const int col0 = (w.tb + j) * kBN;
          const bool need_mask = (col0 + kBN > Nk) || (CAUSAL && col0 + kBN - 1 > first_last);
          const int lim = last_col - col0 - cbase;   // this part's columns c > lim are masked
          float mx = mask_val;
          if (okw) {
            tc_fence_after();
            uint32_t ua[32], ub[32];
            tmem_ld32(s_addr + cbase, ua);
            tmem_ld32(s_addr + cbase + 32, ub);
            tmem_wait_ld();
            if constexpr (ELEM == kE4M3) {
              cj *= f_k;
              if (j + 1 < Jn) {
                kd_next = prm.k_ds[kv_blk + w.tb + j + 1];
                vd_next = prm.v_ds[kv_blk + w.tb + j + 1];
              }
            }
            auto sv = [&](int c) -> float {
              const float x = __uint_as_float(c < 32 ? ua[c] : ub[c - 32]);
              return (need_mask && c > lim) ? mask_val : x;
            };
            // row max (min for a negative scale): eight chains of 3-input max
            float r8[8];
            if (!neg) {
#pragma unroll
              for (int i = 0; i < 8; ++i) r8[i] = fmaxf(sv(i), sv(8 + i));
#pragma unroll
              for (int c = 16; c < 64; c += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) r8[i] = max3f(r8[i], sv(c + i), sv(c + 8 + i));
              mx = max3f(max3f(r8[0], r8[1], r8[2]), max3f(r8[3], r8[4], r8[5]), fmaxf(r8[6], r8[7]));
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) r8[i] = fminf(sv(i), sv(8 + i));
#pragma unroll
              for (int c = 16; c < 64; c += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) r8[i] = min3f(r8[i], sv(c + i), sv(c + 8 + i));
              mx = min3f(min3f(r8[0], r8[1], r8[2]), min3f(r8[3], r8[4], r8[5]), fminf(r8[6], r8[7]));
            }
          }
          // the whole row's maximum: exchange with the other column part
          if (okw) *xslot(xc & 1, part) = mx;
          if (!bar_and(pair_bar, 64, okw)) { ok = false; break; }
          {
            const float other = *xslot(xc & 1, part ^ 1);
            mx = neg ? fminf(mx, other) : fmaxf(mx, other);
          }
          ++xc;
          // a row whose keys in this tile are all masked keeps -inf (for a
          // zero scale mx * cj would be inf * 0 = NaN)
          const float mx2 = (mx == mask_val) ? -INFINITY : mx * cj;
          float alpha = 1.0f;
          const bool move = (mx2 > m_run + C::TAU) || (m_run == -INFINITY && mx2 != -INFINITY);
          if (move) {
            alpha = ex2(m_run - mx2);  // 0 on the first tile
            m_run = mx2;
          }
          l_run *= alpha;
          // rescale this part's half of O when any row of the warp moved
          if (j > 0 && __any_sync(0xffffffffu, move)) {
            const uint32_t o_addr = tmem + lane_addr + C::O_COL0 + t * D + ocol0;
#pragma unroll 1
            for (int c0 = 0; c0 < OCOLS; c0 += 32) {
              uint32_t u[32];
              tmem_ld32(o_addr + c0, u);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
              tmem_st32(o_addr + c0, u);
            }
            tmem_wait_st();
          }
          // P = 2^(s*cj - m), 32 keys at a time, into this part's P columns
          // (which start at the first S column it reads, so a chunk of P only
          // overwrites S this thread has already read)
          const float2 cj2 = make_float2(cj, cj);
          const float lpv = f_lpv, inv_pv = f_inv;
          const float2 nm2 = make_float2(lpv - m_run, lpv - m_run);
          float2 acc[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
          const uint32_t p_addr = s_addr + (uint32_t)(part * C::P_HALF_OFF);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t u[32];
            tmem_ld32(s_addr + cbase + 32 * q, u);
            tmem_wait_ld();
            auto p_pair = [&](int c) -> float2 {   // c: column within this chunk
              const float2 x = fma2(make_float2(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), cj2, nm2);
              float2 p = make_float2(ex2(x.x), ex2(x.y));
              if (need_mask) {
                p.x = (32 * q + c > lim) ? 0.0f : p.x;
                p.y = (32 * q + c + 1 > lim) ? 0.0f : p.y;
              }
              return p;
            };
            if constexpr (ELEM == kE4M3) {
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float2 a = p_pair(4 * i), b = p_pair(4 * i + 2);
                acc[(2 * i) & 3] = add2(acc[(2 * i) & 3], a);
                acc[(2 * i + 1) & 3] = add2(acc[(2 * i + 1) & 3], b);
                pk[i] = pack_e4m3x4(a.x, a.y, b.x, b.y);
              }
              tmem_st8(p_addr + q * 8, pk);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float2 a = p_pair(h * 16 + 2 * i);
                  acc[i & 3] = add2(acc[i & 3], a);
                  pk[i] = (ELEM == kBF16) ? pack_bf16x2(a.x, a.y) : pack_f16x2(a.x, a.y);
                }
                tmem_st8(p_addr + q * 16 + h * 8, pk);
              }
            }
          }
          {
            const float2 tt = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
            l_run += (ELEM == kE4M3) ? (tt.x + tt.y) * inv_pv : (tt.x + tt.y);
          }
          tmem_wait_st();
          tc_fence_before();
          // this part's keys are half `part` of the tile
          mbar_arrive(&bars->p_full[buf][part]);
          if constexpr (ELEM == kE4M3) {
            if (j + 1 < Jn) fp8_factors(kd_next, vd_next);
          }
        } else {
        if (!okw) { ok = false; break; }
        if constexpr (C::NQT == 1) {
          tc_fence_after();
          // PV(gj-2) was issued before S(gj), so it has completed: consume
          // its o_ready phase to keep at most one pending per buffer
          if (gj >= 2 && !consume_o(gj - 2)) { ok = false; break; }
        }
        const uint32_t s_addr = tmem + lane_addr + C::S_COL0 + buf * kBN;
        // where P goes: over S, or (separate P) this tile's P buffer
        const uint32_t p_base = C::SEPP ? tmem + lane_addr + C::P_COL0 + t * C::P_COLS : s_addr;
        float s[NCOL];
        float cj = prm.scale_log2;   // scale of this tile (log2 units)
        const int col0 = (w.tb + j) * kBN;
        const bool need_mask = (col0 + kBN > Nk) || (CAUSAL && col0 + kBN - 1 > first_last);
        float mx = mask_val;
        if (okw) {
          if constexpr (C::NQT == 2) tc_fence_after();
          {
            uint32_t u[32];
#pragma unroll
            for (int c4 = 0; c4 < NCOL / 32; ++c4) {
              tmem_ld32(s_addr + cbase + c4 * 32, u);
#pragma unroll
              for (int i = 0; i < 32; ++i) s[c4 * 32 + i] = __uint_as_float(u[i]);
            }
            tmem_wait_ld();
          }
          if constexpr (C::SEPP) {
            // S is in registers: the next Q K^T may overwrite it
            tc_fence_before();
            mbar_arrive(&bars->s_free[t]);
          }
          if constexpr (ELEM == kE4M3) cj *= f_k;
          if (need_mask) {
            const int lim = last_col - col0 - cbase;
#pragma unroll
            for (int c = 0; c < NCOL; ++c) {
              s[c] = (c > lim) ? mask_val : s[c];
            }
          }
          // row max (min for a negative scale) of this thread's columns:
          // eight chains of 3-input max
          float r8[8];
          if (!neg) {
#pragma unroll
            for (int i = 0; i < 8; ++i) r8[i] = fmaxf(s[i], s[8 + i]);
#pragma unroll
            for (int c = 16; c < NCOL; c += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) r8[i] = max3f(r8[i], s[c + i], s[c + 8 + i]);
            mx = max3f(max3f(r8[0], r8[1], r8[2]), max3f(r8[3], r8[4], r8[5]), fmaxf(r8[6], r8[7]));
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) r8[i] = fminf(s[i], s[8 + i]);
#pragma unroll
            for (int c = 16; c < NCOL; c += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) r8[i] = min3f(r8[i], s[c + i], s[c + 8 + i]);
            mx = min3f(min3f(r8[0], r8[1], r8[2]), min3f(r8[3], r8[4], r8[5]), fminf(r8[6], r8[7]));
          }
        }
        // a row whose keys in this tile are all masked keeps -inf (for a zero
        // scale mx * cj would be inf * 0 = NaN)
        const float mx2 = (mx == mask_val) ? -INFINITY : mx * cj;
        float alpha = 1.0f;
        // (a row that has seen no key yet keeps m = -inf until it does)
        const bool move = (mx2 > m_run + C::TAU) || (m_run == -INFINITY && mx2 != -INFINITY);
        if (move) {
          alpha = ex2(m_run - mx2);  // 0 on the first tile
          m_run = mx2;
        }
        l_run *= alpha;
        if constexpr (C::SEPP) {
          // P V of the previous tile must be done before O is rescaled and
          // the P buffer rewritten
          if (j > 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->p_free[t], (uint32_t)(pfw & 1), abort_flag, prm.err))) {
              ok = false;
              break;
            }
            ++pfw;
            tc_fence_after();
          }
        }
        // rescale O (this thread's output columns) when any row of the warp
        // moved (never on the first tile)
        if (j > 0 && __any_sync(0xffffffffu, move)) {
          if constexpr (C::NQT == 1) {
            // O holds PV(gj-1): wait for it
            if (!consume_o(gj - 1)) { ok = false; break; }
            tc_fence_after();
          }
          rescale_o_cols<OCOLS>(tmem + lane_addr + C::O_COL0 + t * D + ocol0, alpha);
        }
        // P = 2^(s*cj - m) and the row sum (four packed pairs of chains),
        // packed and written back over S a quarter (32 keys) at a time, so
        // the stores overlap the rest and few registers are live at once.
        const float2 cj2 = make_float2(cj, cj);
        // FP8: the V-block factor of p~ is folded into the exponent
        // (2^(x - m + f_lpv)); the row sum is rescaled once per tile (f_inv)
        const float lpv = f_lpv, inv_pv = f_inv;
        // masked scores are already -inf (+inf for a negative scale) and give
        // 2^-inf = 0 where the masked tile takes the select-free form (below);
        // there a row with no visible key yet (m = -inf) takes 0 in place of
        // -m, so that they do not meet -m = +inf
        float2 nm2 = make_float2(lpv - m_run, lpv - m_run);
        if (C::MASK_NOSEL && need_mask && m_run == -INFINITY) nm2 = make_float2(0.0f, 0.0f);
        float2 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
        auto p_pair = [&](int c, bool masked_tile, bool poly) -> float2 {
          const float2 x = fma2(make_float2(s[c], s[c + 1]), cj2, nm2);
          float2 p = poly ? ex2_poly2<C::POLY_DEG>(x) : make_float2(ex2(x.x), ex2(x.y));
          if (masked_tile) {
            p.x = (s[c] == mask_val) ? 0.0f : p.x;
            p.y = (s[c + 1] == mask_val) ? 0.0f : p.y;
          }
          return p;
        };
        // quarters (32 keys) of the tile held by this thread; P of quarter
        // Q sits in TMEM columns Q * 32 * ES / 4 .. of the S/P buffer
        constexpr int NQ = NCOL / 32;
        auto emit = [&](bool masked_tile) {
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            const int qq = part * NQ + q;   // quarter within the tile
            if (C::CSPLIT == 1 && !(VAR & kVarWholeP) && q == 2) {
              // keys 0..63 of P are in TMEM: let their MMAs start
              tmem_wait_st();
              tc_fence_before();
              mbar_arrive(&bars->p_full[buf][0]);
            }
            if constexpr (ELEM == kE4M3) {
              uint32_t u[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int c = q * 32 + 4 * i;
                const float2 a = p_pair(c, masked_tile, C::poly_pair(2 * i));
                const float2 b = p_pair(c + 2, masked_tile, C::poly_pair(2 * i + 1));
                acc[(2 * i) & 3] = add2(acc[(2 * i) & 3], a);
                acc[(2 * i + 1) & 3] = add2(acc[(2 * i + 1) & 3], b);
                u[i] = pack_e4m3x4(a.x, a.y, b.x, b.y);
              }
              tmem_st8(p_base + qq * 8, u);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t u[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const int c = q * 32 + h * 16 + 2 * i;
                  const float2 a = p_pair(c, masked_tile, C::poly_pair(i));
                  acc[i & 3] = add2(acc[i & 3], a);
                  u[i] = (ELEM == kBF16) ? pack_bf16x2(a.x, a.y) : pack_f16x2(a.x, a.y);
                }
                tmem_st8(p_base + qq * 16 + h * 8, u);
              }
            }
          }
        };
        // Masked tiles (causal diagonal, ragged end) zero the masked p one by
        // one, except in the 16-bit d = 128 and causal kernels' units of up to
        // 32 key tiles with a nonzero scale, where the masked tiles are a large
        // share (select-free form: causal mid +7%, causal N = 512 +16% at
        // d = 128 and +20% at d = 64, measured; the non-causal d = 64 / 256
        // and FP8 kernels, and long units, ran 1-2.5% slower with it).
        if (need_mask && (!C::MASK_NOSEL || cj == 0.0f || Jn > 32)) emit(true);
        else emit(false);
        {
          const float2 tt = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
          l_run += (ELEM == kE4M3) ? (tt.x + tt.y) * inv_pv : (tt.x + tt.y);
        }
        tmem_wait_st();
        tc_fence_before();
        if (VAR & kVarWholeP) mbar_arrive(&bars->p_full[buf][0]);
        mbar_arrive(&bars->p_full[buf][1]);
        if constexpr (ELEM == kE4M3) {
          if (j + 1 < Jn) {
            if (((j + 1) & 31) == 0) fp8_batch(j + 1);
            fp8_take(j + 1);
          }
        }
        }
      }

      // ---------------------------------------------------------- epilogue --
      if (ok) {
        bool oke = __all_sync(0xffffffffu, mbar_wait(&bars->o_full[t], (uint32_t)(oc & 1), abort_flag, prm.err));
        ++oc;
        if constexpr (C::CSPLIT == 2) {
          // the whole row's sum: exchange with the other column part
          if (oke) *xslot(xc & 1, part) = l_run;
          oke = bar_and(pair_bar, 64, oke);
          if (oke) l_run += *xslot(xc & 1, part ^ 1);
          ++xc;
        }
        ok = oke;
        if (ok) {
          tc_fence_after();
          const float inv_l = (l_run > 0.0f) ? (1.0f / l_run) : 0.0f;
          const float f = inv_l * v_mult;
          const uint32_t o_addr = tmem + lane_addr + C::O_COL0 + t * D + ocol0;
          const bool store = row < N;
          if (SPLIT && S > 1) {
            // split-KV partial: O normalised over this split's keys, fp32,
            // and the split's LSE (a row without visible keys: 0, -inf)
            const size_t pr = ((size_t)w.split * prm.BH + bh) * N + (size_t)(store ? row : 0);
            float* prow = prm.o_part + pr * D + ocol0;
#pragma unroll 1
            for (int c0 = 0; c0 < OCOLS; c0 += 32) {
              uint32_t u[32];
              tmem_ld32(o_addr + c0, u);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * f);
              if (store) {
#pragma unroll
                for (int i = 0; i < 4; ++i) st_global_v8(prow + c0 + 8 * i, u + 8 * i);
              }
            }
            if (store && part == 0) prm.lse_part[pr] = (m_run + lg2(l_run)) * 0.69314718055994530942f;
          } else if (C::EPI_TMA) {
            // this warp's 32 rows through its staging box, 64 columns at a
            // time: row `lane` of the box holds its 128 bytes with 16-byte
            // chunk c at position c ^ (lane % 8) (the map's 128-byte swizzle)
            uint8_t* stg = smem + C::OFF_EPI + (t * 4 + wq) * C::EPI_WARP_BYTES;
            const uint32_t my_row = smem_u32(stg) + (uint32_t)lane * 128u;
            const int row0 = q0 + wq * 32;
#pragma unroll 1
            for (int c0 = 0; c0 < OCOLS; c0 += C::EPI_BOX_COLS) {
              uint32_t u[32], u2[32];
              tmem_ld32(o_addr + c0, u);
              tmem_ld32(o_addr + c0 + 32, u2);
              tmem_wait_ld();
              uint32_t pk[32];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float a = __uint_as_float(u[2 * i]) * f, b = __uint_as_float(u[2 * i + 1]) * f;
                const float a2 = __uint_as_float(u2[2 * i]) * f, b2 = __uint_as_float(u2[2 * i + 1]) * f;
                pk[i] = (ELEM == kFP16) ? pack_f16x2(a, b) : pack_bf16x2(a, b);
                pk[16 + i] = (ELEM == kFP16) ? pack_f16x2(a2, b2) : pack_bf16x2(a2, b2);
              }
              // the previous box has been read out of the buffer
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
#pragma unroll
              for (int c = 0; c < 8; ++c)
                st_shared_v4(my_row + ((uint32_t)(c ^ (lane & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                             pk[4 * c + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              // rows at or past N are outside the map and not written
              if (lane == 0 && row0 < N) {
                tma_store_3d(&tm_o, stg, ocol0 + c0, row0, bh);
                bulk_commit_group();
              }
            }
            if (store && part == 0) prm.lse[(size_t)bh * N + row] = (m_run + lg2(l_run)) * 0.69314718055994530942f;
          } else {
          uint8_t* orow = reinterpret_cast<uint8_t*>(prm.o) + (((size_t)bh * N + (size_t)(store ? row : 0)) * D + ocol0) * 2;
#pragma unroll 1
          for (int c0 = 0; c0 < OCOLS; c0 += 32) {
            uint32_t u[32];
            tmem_ld32(o_addr + c0, u);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a = __uint_as_float(u[2 * i]) * f, b = __uint_as_float(u[2 * i + 1]) * f;
              pk[i] = (ELEM == kFP16) ? pack_f16x2(a, b) : pack_bf16x2(a, b);
            }
            if (store) {
              // each lane writes its own row: whole 32-byte sectors when the
              // output allows it (the C ABI only promises 16-byte alignment)
              if (prm.o_vec32) {
#pragma unroll
                for (int i = 0; i < 2; ++i) st_global_v8(orow + c0 * 2 + 32 * i, pk + 8 * i);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 2);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
              }
            }
          }
          if (store && part == 0) prm.lse[(size_t)bh * N + row] = (m_run + lg2(l_run)) * 0.69314718055994530942f;
          }
        }
      }
      g += Jn;
      } while (0);
    }
  }
  // the epilogue's bulk stores have completed (and stopped reading shared
  // memory) before the CTA ends
  if (C::EPI_TMA && warp < C::SOFTMAX_WARPS && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace fa

namespace fa {

// Everything one launch needs; filled by the C-ABI layer.
struct AttnLaunch {
  CUtensorMap q, k, v;
  CUtensorMap o;        // O [BH, N, D] 16-bit: box of 64 columns x 32 rows (the epilogue's bulk stores)
  AttnParams prm;
  int BH;
  long long max_ctas;   // 0: one CTA per SM
  cudaStream_t stream;
};

// Element-type code for FP8 inputs in internal_prepare_fwd (the C ABI's
// dtype codes cover bf16 and fp16).
constexpr int kDtypeE4M3 = 100;

// Checks the arguments of a forward call, encodes the tensor maps and fills
// the launch (defined in api.cu).  *empty: nothing to do (FA_OK).
fa_status internal_prepare_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                               int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d, int causal, float scale,
                               int dtype, const float* q_descale, const float* k_descale, const float* v_descale,
                               cudaStream_t stream, AttnLaunch* out, bool* empty);

template <int ELEM, int D, bool CAUSAL, bool SPLIT, int VAR = 0>
cudaError_t launch_attn(const AttnLaunch& L) {
  using C = AttnCfg<ELEM, D, CAUSAL, VAR>;
  auto kern = attn_fwd_kernel<ELEM, D, CAUSAL, SPLIT, VAR>;
  static bool attr_done[64] = {};  // the attribute is per function and device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  // persistent grid: one CTA per SM (shared memory admits no second one)
  static int sm_count[64] = {};
  if (dev >= 0 && dev < 64 && sm_count[dev] == 0) {
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const int sms = (dev >= 0 && dev < 64) ? sm_count[dev] : 148;
  const long long groups = (L.prm.N + C::NQT * kBM - 1) / (C::NQT * kBM);
  const long long n_groups_all = (long long)L.BH * groups * (SPLIT ? L.prm.splits : 1);
  // Non-causal two-tile groups: when the groups leave a last, partial wave
  // of at most half the SMs, run that wave's groups as single-tile units
  // (twice as many, each about 3/4 as long), so the last wave ends sooner.
  AttnParams prm = L.prm;
  prm.pair_units = (int)n_groups_all;
  if constexpr (!CAUSAL && !SPLIT && C::NQT == 2) {
    const long long rem = n_groups_all % sms;
    if (rem > 0 && 2 * rem <= sms) prm.pair_units = (int)(n_groups_all - rem);
  }
  const long long units = n_groups_all + (C::NQT - 1) * (n_groups_all - prm.pair_units);
  // Causal: chunks of heads whose K/V (read once from HBM, then re-read by
  // every Q tile of the head from L2) take up to about half of L2 at a time;
  // with all heads at once, long sequences re-read K/V from HBM many times.
  prm.head_chunk = prm.BH;
  if constexpr (CAUSAL && !SPLIT) {
    const long long kv_head_bytes = 2LL * L.prm.Nk * C::ROW_BYTES;
    const long long budget = 64LL << 20;
    const int qgroup = L.prm.Hq / L.prm.Hkv;
    long long chunk = (budget / (kv_head_bytes > 0 ? kv_head_bytes : 1)) * qgroup;
    if (chunk < qgroup) chunk = qgroup;
    if (chunk < prm.BH) prm.head_chunk = (int)chunk;
  }
  if constexpr (C::REALLOC) {
    // the register split must fit what the kernel is launched with, or the
    // growing warpgroups would wait for registers that never come
    static int regs_ok[64] = {};
    if (dev >= 0 && dev < 64 && regs_ok[dev] == 0) {
      cudaFuncAttributes fa_attr;
      e = cudaFuncGetAttributes(&fa_attr, kern);
      if (e != cudaSuccess) return e;
      regs_ok[dev] = (fa_attr.numRegs * C::THREADS >= 128 * C::CTRL_REGS + C::SOFTMAX_WARPS * 32 * C::SOFTMAX_REGS) ? 1 : -1;
    }
    if (dev < 0 || dev >= 64 || regs_ok[dev] != 1) return cudaErrorInvalidConfiguration;
  }
  // one CTA per unit, launched as 1x1x1 clusters so that running CTAs can
  // take over the units of CTAs that have not started (cluster launch control)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)units, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, L.q, L.k, L.v, L.o, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fa
