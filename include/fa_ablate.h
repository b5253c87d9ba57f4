/*
 * fa_ablate.h -- ablation entry point of libfa_ablate.so (a separate
 * library built beside libfa.so, which it links against; not part of the
 * product API).
 *
 * The attention forward of fa_fwd / fa_fwd_fp8 (B, H, N, d = 128, Hq = Hkv,
 * Nq = Nk) with one design choice of the kernel switched, so that what each
 * choice is worth can be timed from the committed tree.  The pages motivate
 * the comparison: "FlashAttention-3: async pipelines on Hopper", section
 * "second overlap" (two consumer groups alternating softmax and GEMMs, the
 * ping-pong measured at 570 -> 620-640 TFLOPS on H100) and section "third
 * overlap" (the next Q K^T during the softmax).  Variant codes (bits):
 *   0   the shipped kernel (fa_fwd / fa_fwd_fp8 of libfa.so)
 *   1   split softmax: two softmax warpgroups per Q tile, 64 key columns each
 *   2   eager rescale: O rescaled whenever a row maximum rises (no lazy threshold)
 *   4   whole P: P handed to the MMA warp in one piece, not in two halves
 *   8   one Q tile per CTA with S double-buffered (no two-tile alternation)
 *   16  no work stealing: each CTA runs only the unit it was launched with
 *   32  separate P: P gets its own tensor-memory columns, so the next Q K^T
 *       starts once the softmax has read S (d = 64 only: there S, P and O of
 *       two Q tiles fit the 512 columns)
 *   64  polynomial exponentials: 1 of every 8 pairs of P (d = 128 bf16) or
 *       3 of 8 (FP8, d = 64) computed on the FMA pipe by range reduction and
 *       a degree-3 minimax polynomial instead of the special-function unit
 *       (fa_debug_exp2 method 3 evaluates the same function)
 *   128 early partial Q K^T: the keys of the next tile whose S columns P
 *       (written over S from column 0) does not use are multiplied as soon as
 *       the first half of P arrives, the remaining keys after the second half
 *       (two narrower MMAs instead of one of N = 128)
 *   256 direct O stores: each thread writes its own row of O from registers
 *       (32-byte vector stores, 32 rows per warp instruction) instead of
 *       staging 64-column boxes in shared memory for bulk tensor stores; the
 *       ring keeps the slot the boxes take (d = 128 16-bit: 5 slots, not 4)
 * Built instances: d = 128 bf16 non-causal and FP8 non-causal with codes
 * 0, 1, 2, 4, 8, 16, 64, 128, 256; d = 128 bf16 causal with 0, 1, 8, 16,
 * 256; d = 64 bf16 non-causal with 0, 1, 32, 64, 128, 256 and causal with 0, 32.
 *   variant      one of the codes above
 *   fp8          0: q, k, v bf16 (descales ignored, may be NULL); 1: E4M3
 *                codes with [B, H, ceil(N/128)] fp32 descales as fa_fwd_fp8
 *   other arguments as fa_fwd / fa_fwd_fp8 (device pointers, [B, H, N, d]
 *   contiguous, o bf16, lse fp32 [B, H, N]); d is 64 or 128.
 * Errors: FA_ERR_UNSUPPORTED for a variant / type / head dimension / causal
 * combination that was not built; otherwise as fa_fwd.
 */
#ifndef FA_ABLATE_H
#define FA_ABLATE_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

fa_status fa_ablate_fwd(int variant, int fp8, const void* q, const void* k, const void* v, void* o, float* lse,
                        int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                        const float* q_descale, const float* k_descale, const float* v_descale,
                        cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_ABLATE_H */
