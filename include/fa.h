/*
 * fa.h -- C ABI of the fused exact attention forward library (libfa.so) for
 * NVIDIA GB300 (sm_103a).
 *
 * Operation.  Exact scaled-dot-product attention, forward pass:
 *     S = scale * Q K^T,   P = softmax(S) row-wise,   O = P V,
 *     LSE_i = ln sum_j exp(S_ij)
 * (definition: wmrh.cn FlashAttention V3 article, sec. 1.1 "self-attention
 * and the O(N^2) problem").  The kernels stream K/V tiles through shared
 * memory and run the online-softmax recurrence -- running row max m, running
 * row sum l, rescaled accumulator o, initially -inf, 0, 0, output o/l after
 * the last tile (same article, sec. 2.1; "FlashAttention-3: async pipelines
 * on Hopper" (charlestar.github.io), section "Online Softmax is still the
 * core of exact merging") -- so the N x N score matrix never reaches HBM.
 * Causal attention keeps the lower triangle, key j <= query i, and skips the
 * key tiles above the diagonal ("FlashAttention-3: async pipelines on
 * Hopper", section "why causal shapes are harder to schedule").  The LSE
 * output is not defined on the pages; here it is the natural log of the sum
 * of exponentials of the scaled, masked scores, in fp32.
 *
 * Conventions shared by every entry point
 *   - Tensors are contiguous row-major [B, H, N, d] (PyTorch SDPA order,
 *     wmrh.cn article sec. 6.4); LSE is [B, H, N] fp32.
 *   - Every tensor pointer is a DEVICE pointer on the current CUDA device,
 *     16-byte aligned, owned by the caller.  Inputs are only read; outputs are
 *     fully overwritten.  The library allocates no memory in these calls.
 *   - Work is enqueued on `stream` and the call returns without waiting.
 *     A launch error is reported as FA_ERR_CUDA; errors found by the kernels
 *     (a pipeline wait that ran out of time) are reported later by
 *     fa_check_device_error().
 *   - B*H*N == 0 is valid and does nothing.
 *   - Head dimension d must be 64, 128 or 256.  The library runs only on
 *     compute capability 10.3 (sm_103a); anything else is FA_ERR_UNSUPPORTED.
 *     There is no fallback path.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, negative size, non-finite scale, bad dtype */
    FA_ERR_UNSUPPORTED = 2,   /* head dimension or device not supported                            */
    FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call or kernel launch failed                 */
    FA_ERR_TIMEOUT = 4,       /* a kernel's pipeline wait ran out of time (see fa_check_device_error) */
    FA_ERR_SCRATCH_LIMIT = 5  /* problem larger than the library's static scratch (no-allocation entry point) */
} fa_status;

typedef enum {
    FA_DTYPE_BF16 = 0,
    FA_DTYPE_FP16 = 1
} fa_dtype;

/* Maximum number of rows per FP8 quantisation block (one scale per block). */
#define FA_FP8_BLOCK_ROWS 128

/*
 * fa_fwd -- BF16 / FP16 attention forward.
 *   q, k, v  [B, H, N, d] of `dtype` (device, read only)
 *   o        [B, H, N, d] of `dtype` (device, written), rounded to nearest even
 *   lse      [B, H, N] fp32 (device, written)
 *   causal   0: every key visible; 1: key j visible to query i iff j <= i
 *   scale    multiplies Q K^T before the softmax (usually 1/sqrt(d)); finite
 *   dtype    FA_DTYPE_BF16 or FA_DTYPE_FP16
 * Softmax statistics and accumulation are fp32; P is rounded to `dtype`
 * before the P V product ("FlashAttention-3: async pipelines on Hopper",
 * section "Online Softmax is still the core of exact merging": FP16/BF16
 * keep the rescaling and accumulation state in FP32).
 * Non-finite inputs are not checked.  A NaN in a query row makes that row's
 * O and LSE NaN; a NaN in key row j makes NaN every row that sees key j.  A
 * NaN or infinity in element (j, c) of V reaches column c of O in every row
 * that sees key j and also, with causal = 1, in the rows of j's 128-row tile
 * that precede j (P V multiplies their P = 0 by it); rows of earlier tiles,
 * the other columns and LSE are unaffected.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int64_t B, int64_t H, int64_t N, int64_t d,
                 int causal, float scale, int dtype, cudaStream_t stream);

/*
 * fa_fwd_fp8 -- FP8 E4M3 attention forward with per-block scales.
 *   q8, k8, v8  [B, H, N, d] E4M3 codes (device, read only), as written by
 *               fa_quant_fp8; real value = decode(code) * descale of its block
 *   q_descale, k_descale, v_descale
 *               [B, H, ceil(N/128)] fp32 (device): one scale per 128-row block
 *               ("FlashAttention-3: async pipelines on Hopper", section "why
 *               block quantization beats a per-tensor scale": the Q/K block
 *               scales are restored on each score tile, the V block scale is
 *               applied with the P V product)
 *   o           [B, H, N, d] bf16 (device, written);  lse [B, H, N] fp32
 *   causal, scale as in fa_fwd.
 * Q K^T and P V run on the FP8 tensor cores with fp32 accumulation; the
 * softmax state is fp32 ("FlashAttention-3: async pipelines on Hopper",
 * section "FP8 attention is still not FP8 end to end").  If Q and K were
 * rotated by the same orthogonal matrix (fa_quant_fp8 with signs), the
 * scores are unchanged and O needs no correction; V is never rotated.
 */
fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* v8, void* o, float* lse,
                     int64_t B, int64_t H, int64_t N, int64_t d,
                     int causal, float scale,
                     const float* q_descale, const float* k_descale, const float* v_descale,
                     cudaStream_t stream);

/*
 * fa_fwd_gqa -- fa_fwd for grouped-query / multi-query attention and for
 * different query and key lengths ("FlashAttention-3: async pipelines on
 * Hopper", section "how GQA/MQA changes the kernel's task count": several
 * query heads share one K/V head through the head index, K/V are never
 * copied in HBM).
 *   q    [B, Hq, Nq, d];  k, v [B, Hkv, Nk, d];  o [B, Hq, Nq, d];  lse [B, Hq, Nq]
 *   Hq must be a multiple of Hkv (>= 1); query head h reads K/V head
 *   h / (Hq / Hkv).  Nk >= 1 when Nq >= 1.
 *   causal: key j is visible to query i iff j <= i + (Nk - Nq) (the mask is
 *   aligned at the bottom right; for Nq == Nk this is j <= i).  A query row
 *   that sees no key (causal with Nq > Nk) gets O = 0 and LSE = -inf.
 * fa_fwd(q, k, v, o, lse, B, H, N, d, ...) equals
 * fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, N, d, ...).
 */
fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                     int causal, float scale, int dtype, cudaStream_t stream);

/*
 * fa_fwd_fp8_gqa -- fa_fwd_fp8 with the head and length conventions of
 * fa_fwd_gqa: q8 [B, Hq, Nq, d], q_descale [B, Hq, ceil(Nq/128)];
 * k8, v8 [B, Hkv, Nk, d], k_descale, v_descale [B, Hkv, ceil(Nk/128)].
 */
fa_status fa_fwd_fp8_gqa(const void* q8, const void* k8, const void* v8, void* o, float* lse,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                         int causal, float scale,
                         const float* q_descale, const float* k_descale, const float* v_descale,
                         cudaStream_t stream);

/*
 * fa_fwd_host -- fa_fwd_gqa on HOST buffers: the call copies q, k, v to the
 * device, runs the attention kernel and copies o and lse back, in chunks of
 * whole key/value heads (each with its query heads), so that the copies of
 * one chunk overlap the kernel of the previous one and the copies back of
 * the one before (4 chunks, or up to 16 when each still holds a wave of
 * work units; two host->device streams, two compute streams that
 * consecutive chunks alternate between, and a device->host stream, created
 * once per device and joined to `stream` with events; nothing is allocated
 * per call).
 *   q_host, o_host  [B, Hq, Nq, d]   bf16 or fp16 (dtype), HOST memory
 *   k_host, v_host  [B, Hkv, Nk, d]  same dtype, HOST memory
 *   lse_host        [B, Hq, Nq] fp32, HOST memory
 *                   Page-locked memory (cudaHostAlloc / cudaHostRegister)
 *                   lets the copies run asynchronously and overlap; with
 *                   pageable memory the results are the same but the copies
 *                   do not overlap.
 *   workspace       DEVICE pointer, 256-byte aligned, owned by the caller,
 *                   at least fa_fwd_host_workspace_bytes(...) bytes (device
 *                   copies of q, o, k, v, lse); overwritten
 * Asynchronous on `stream` like cudaMemcpyAsync: o_host and lse_host hold
 * the results once `stream` has synchronised; the host buffers must stay
 * valid until then.  Results are bit-identical to fa_fwd_gqa on device
 * copies of the same inputs.  Errors: as fa_fwd_gqa (host pointers need no
 * alignment), plus FA_ERR_INVALID_ARG for a missing, misaligned or too
 * small workspace.
 */
fa_status fa_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                      int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                      int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/*
 * fa_fwd_host_workspace_bytes -- device workspace fa_fwd_host needs:
 * 2*B*Hq*Nq*d*2 + 2*B*Hkv*Nk*d*2 + B*Hq*Nq*4 bytes, each part rounded up to
 * 256.  Writes *bytes (0 for an empty batch).  Same size checks as
 * fa_fwd_host.
 */
fa_status fa_fwd_host_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                                      size_t* bytes);

/*
 * fa_fwd_splitkv -- the forward pass of fa_fwd_gqa for decode-like shapes
 * (few query rows against a long key/value sequence), where batch x heads x
 * query tiles leave most SMs idle ("FlashAttention-3: async pipelines on
 * Hopper", sections "why GQA/MQA changes the kernel's task count" and
 * "prefill, decode and training gain differently": decode needs split-KV
 * and GQA packing to produce enough parallelism).
 *   Same inputs, outputs, layouts and masking as fa_fwd_gqa (q [B, Hq, Nq, d],
 *   k/v [B, Hkv, Nk, d], bf16 or fp16; causal masks bottom-right aligned).
 *   The Hq / Hkv query heads sharing a key/value head are processed as one
 *   head of (Hq / Hkv) * Nq rows, so every key/value byte is read once per
 *   group; each row's keys are split into num_splits runs processed in
 *   parallel, whose partial results (O normalised per run, fp32, and the
 *   run's LSE) go to `workspace` and are merged by LSE weights in a second
 *   kernel on the same stream.  The merge is exact in real arithmetic.
 *   num_splits   0: chosen for the current device (about eight work units
 *                per SM, at least 8 key tiles of 128 per run); else the
 *                requested count, capped at the number of 128-key tiles
 *                (runs are never empty).
 *   workspace    DEVICE pointer, 256-byte aligned, owned by the caller, at
 *                least the size fa_splitkv_workspace_bytes reports for the
 *                same shape and num_splits on the same device (NULL allowed
 *                when that size is 0: a single run writes O directly);
 *                overwritten; calls sharing it must not overlap on the GPU.
 * Errors: as fa_fwd_gqa, plus FA_ERR_INVALID_ARG for num_splits < 0 or a
 * missing, misaligned or too small workspace.
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                         int causal, float scale, int dtype, int num_splits,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_splitkv_workspace_bytes -- bytes of device workspace fa_fwd_splitkv
 * needs for this shape and num_splits on the current device (0 when the
 * keys are not split).  Writes *bytes; same argument checks as
 * fa_fwd_splitkv (no pointers besides bytes).
 */
fa_status fa_splitkv_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                                     int num_splits, size_t* bytes);

/*
 * fa_bwd -- gradients of the loss sum(dout * O) for O = fa_fwd_gqa(q, k, v):
 * dq, dk, dv (the pages list the backward pass dQ, dK, dV among the paths a
 * test must cover and compare its speed with FA2: "FlashAttention-3: async
 * pipelines on Hopper", sections "correctness validation must cover
 * asynchronous boundaries" and "how to read the paper's performance
 * numbers").  With P = softmax(scale q k^T) recomputed from the forward's
 * LSE, dP = dout v^T, D_i = dout_i . o_i and dS = P * (dP - D):
 *   dv = P^T dout,   dk = scale dS^T q,   dq = scale dS k,
 * dk and dv summed over the query heads of each key/value group.
 *   q, dout, o, dq  [B, Hq, Nq, d]   bf16 or fp16 (dtype), device
 *   k, v, dk, dv    [B, Hkv, Nk, d]  same dtype, device
 *   lse             [B, Hq, Nq] fp32, the natural-log LSE fa_fwd_gqa wrote
 *                   for the same q, k, v, causal and scale (-inf: a row that
 *                   sees no key; it gets dq = 0 and adds nothing)
 *   causal          0 / 1, masks aligned at the bottom right as in fa_fwd_gqa
 *   workspace       DEVICE pointer, 256-byte aligned, owned by the caller, at
 *                   least fa_bwd_workspace_bytes(B, Hq, Nq, d) bytes (an fp32
 *                   dQ accumulator and two floats per query row); overwritten;
 *                   calls sharing it must not overlap on the GPU
 * q, k, v, o, lse, dout are read only; dq, dk, dv are fully overwritten.
 * All pointers 16-byte aligned.  Asynchronous on `stream` (four kernels:
 * D and accumulator clear, the fused gradient kernel, dQ conversion), no
 * host synchronisation, no allocation.  dq is accumulated across key tiles
 * with fp32 reduce-adds, so its rounding may differ between runs.
 * Errors: FA_ERR_INVALID_ARG for bad pointers, alignment, sizes, dtype,
 * causal flag, scale or workspace; FA_ERR_UNSUPPORTED for d = 256 (the
 * backward kernel covers d = 64 and 128) or a device other than sm_103;
 * FA_ERR_CUDA for a launch failure; a pipeline timeout is reported by
 * fa_check_device_error.  B*Hq = 0 is a no-op; Nq = 0 writes dk = dv = 0.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv,
                 int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                 int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream);

/*
 * fa_bwd_workspace_bytes -- bytes of device workspace fa_bwd needs:
 * B*Hq*Nq*d*4 (fp32 dQ accumulator, rounded up to 256) + B*Hq*R*512 with R
 * the 64-row records per head: ceil(Nq/64) for d = 128, 2*ceil(Nq/128) for
 * d = 64 (the kernel's step is 128 query rows there); each record holds
 * its rows' log-sum-exp and D terms.  Writes *bytes.  FA_ERR_INVALID_ARG for negative sizes or a null
 * `bytes`, FA_ERR_UNSUPPORTED for d not in {64, 128, 256}.
 */
fa_status fa_bwd_workspace_bytes(int64_t B, int64_t Hq, int64_t Nq, int64_t d, size_t* bytes);

/*
 * fa_quant_fp8 -- quantise fp32 [B, H, N, d] to E4M3 with one scale per
 * 128-row block (per_tensor = 0) or one scale for the whole tensor
 * (per_tensor = 1, the baseline), optionally after the incoherent-processing
 * rotation x -> x diag(signs) H_d / sqrt(d) ("FlashAttention-3: async
 * pipelines on Hopper", section "how incoherent processing flattens
 * outliers": a random +-1 diagonal combined with a Hadamard matrix, applied
 * to both Q and K, never to V).
 *   x              [B, H, N, d] fp32 (device, read only)
 *   x8             [B, H, N, d] E4M3 codes (device, written)
 *   descale        [B, H, ceil(N/128)] fp32 (device, written): the value to
 *                  multiply a code by; scale = amax/448 of the (rotated) block
 *                  (wmrh.cn article sec. 3.3: 448 is the E4M3 maximum), 1 for
 *                  an all-zero block, times 1/sqrt(d) when rotating
 *   hadamard_signs HOST pointer to d int8 entries of +1/-1, or NULL for no
 *                  rotation; read during the call only
 *   per_tensor     0 or 1
 *   workspace      per_tensor = 1: DEVICE pointer to one float of scratch
 *                  (overwritten; calls sharing it must not overlap on the GPU);
 *                  per_tensor = 0: ignored, may be NULL
 * The rotated value y is fp32 (sign flip, then the Walsh-Hadamard butterfly
 * with strides 1, 2, 4, ...), scale = amax(y) / 448 rounded to fp32, and each
 * code is the E4M3 value nearest to the exact quotient y / scale (ties to
 * even, saturated at 448): a single rounding, decided exactly.
 * Errors: FA_ERR_INVALID_ARG for negative sizes, null or misaligned pointers
 * (x, x8 16-byte aligned), signs other than +-1, per_tensor not 0 / 1 or a
 * missing workspace; FA_ERR_UNSUPPORTED for d not in {64, 128, 256}, more
 * than 2^31 - 1 blocks, or a device other than sm_103; FA_ERR_CUDA for a
 * launch error.  B*H*N = 0 is a no-op.  A bounded wait inside the kernel that
 * runs out (about 2 s) sets the library's error word (fa_check_device_error
 * then returns FA_ERR_TIMEOUT) and marks the blocks it could not finish with
 * a NaN descale (per-tensor mode: an infinite scale) instead of leaving old
 * values.
 */
fa_status fa_quant_fp8(const float* x, void* x8, float* descale,
                       int64_t B, int64_t H, int64_t N, int64_t d,
                       const int8_t* hadamard_signs, int per_tensor, float* workspace,
                       cudaStream_t stream);

/*
 * fa_quant_fp8_qkv -- the FP8 inputs of one attention call in one call: Q and
 * K with block scales after the rotation (when hadamard_signs is not NULL),
 * V with block scales and no rotation (the pages rotate Q and K only, with
 * the same signs, so that Q K^T is unchanged).  Each result is exactly what
 * fa_quant_fp8(x, ..., per_tensor = 0) gives for that tensor.  The three
 * quantisations run on internal streams forked from `stream` and joined back
 * into it, so that each launch's CTAs start on the SMs the others' last CTAs
 * leave free (at B=4 H=16 N=4096 d=128: 95 us against 107 us for three
 * calls in a row); work enqueued on `stream` afterwards runs after all three.
 *   q, k, v        [B, Hq, Nq, d], [B, Hkv, Nk, d], [B, Hkv, Nk, d] fp32 (device, read only)
 *   q8, k8, v8     E4M3 codes of the same shapes (device, written)
 *   q_descale      [B, Hq, ceil(Nq/128)] fp32 (device, written); k_descale and
 *   v_descale      [B, Hkv, ceil(Nk/128)], as fa_quant_fp8's descale
 *   hadamard_signs as fa_quant_fp8 (applied to Q and K)
 * Errors: as fa_quant_fp8 for any of the three tensors, checked before
 * anything is launched; FA_ERR_CUDA if the internal streams cannot be
 * created.  A tensor with no element is skipped.  Calls on one device share
 * the internal streams (serialised by a lock; the launches of consecutive
 * calls still run in order on each of them).
 */
fa_status fa_quant_fp8_qkv(const float* q, const float* k, const float* v, void* q8, void* k8, void* v8,
                           float* q_descale, float* k_descale, float* v_descale,
                           int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                           const int8_t* hadamard_signs, cudaStream_t stream);

/*
 * fa_quant_fp8_rope -- fa_quant_fp8 with a rotary position embedding applied
 * to every row first, in the same pass ("FlashAttention-3: async pipelines on
 * Hopper", sections "why block quantization beats a per-tensor scale" and
 * "how incoherent processing flattens outliers": the block scales and the
 * Hadamard rotation can share one pass with a preceding RoPE).  The pages fix
 * no RoPE convention, so the angles come from the caller and both usual
 * channel pairings are offered:
 *   FA_ROPE_INTERLEAVED  pairs (2i, 2i+1), i < d/2
 *   FA_ROPE_HALF         pairs (i, i + d/2), i < d/2
 * Pair (a, b) of row n becomes (a*c - b*s, a*s + b*c) with c = rope_cos[n][i],
 * s = rope_sin[n][i], in fp32 with each product rounded before the sum; then
 * the optional rotation and the quantisation proceed as in fa_quant_fp8.
 *   rope_cos, rope_sin  [N, d/2] fp32 (device, read only, 16-byte aligned),
 *                       shared by every (b, h): row n is position n of each
 *                       sequence (offset positions by offsetting the tables)
 *   rope_layout         FA_ROPE_INTERLEAVED or FA_ROPE_HALF
 *   other arguments as for fa_quant_fp8.
 * Errors: FA_ERR_INVALID_ARG for a null or misaligned table or an unknown
 * layout, otherwise as fa_quant_fp8.
 */
#define FA_ROPE_INTERLEAVED 1
#define FA_ROPE_HALF 2
fa_status fa_quant_fp8_rope(const float* x, void* x8, float* descale,
                            int64_t B, int64_t H, int64_t N, int64_t d,
                            const float* rope_cos, const float* rope_sin, int rope_layout,
                            const int8_t* hadamard_signs, int per_tensor, float* workspace,
                            cudaStream_t stream);

/*
 * fa_quant_fp8_per_tensor_noalloc -- the per-tensor mode of fa_quant_fp8
 * (per_tensor = 1) for callers that cannot allocate device memory.  The
 * pages have no counterpart; it exists for the library's users.
 *
 * fa_quant_fp8 needs one float of device scratch from the caller in
 * per-tensor mode.  Callers that cannot allocate -- code running under a
 * framework that owns every device buffer, plug-ins whose host forbids
 * cudaMalloc (which may also synchronise the device), runtimes with a fixed
 * memory budget -- use this entry point instead: it takes the same inputs
 * and outputs but keeps its scratch in a device array compiled into the
 * library (about 256 KiB, held by every GPU that loads the library until
 * the process exits).  It calls no allocator.
 *   x, x8, descale, B, H, N, d, hadamard_signs: as for fa_quant_fp8; the
 *   output equals fa_quant_fp8 with per_tensor = 1 bit for bit.
 *   Limit: B * H * ceil(N / 128) <= FA_QUANT_NOALLOC_MAX_BLOCKS, else
 *   FA_ERR_SCRATCH_LIMIT and nothing is launched.
 *   The first call on each device looks up the scratch array's device
 *   address (with that device current); make that first call before any
 *   stream capture.
 *   All calls share the one scratch array and it keeps the last call's
 *   contents (each call writes every entry it reads, so nothing needs
 *   clearing; a block whose input load timed out writes +inf and sets the
 *   library's error word, see fa_check_device_error): calls that overlap on
 *   the GPU -- other streams, other host threads on the same device -- race
 *   and can produce wrong scales.
 *   Errors: as fa_quant_fp8 (per_tensor = 1), plus FA_ERR_SCRATCH_LIMIT.
 */
#define FA_QUANT_NOALLOC_MAX_BLOCKS 65536
fa_status fa_quant_fp8_per_tensor_noalloc(const float* x, void* x8, float* descale,
                                          int64_t B, int64_t H, int64_t N, int64_t d,
                                          const int8_t* hadamard_signs, cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* fa_status_string(fa_status status);

/*
 * fa_check_device_error -- synchronises `stream`, then reports and clears the
 * library's device error word on the current device: FA_ERR_TIMEOUT if a
 * kernel gave up on a pipeline wait since the last check, FA_ERR_CUDA if the
 * synchronisation itself failed, else FA_OK.
 */
fa_status fa_check_device_error(cudaStream_t stream);

/*
 * fa_debug_inject -- TEST HOOK for the failure path; not for production use.
 * flags bit 0: the next fa_fwd / fa_fwd_fp8 launch has its first CTA leave
 * one K/V ring slot unfilled (the next fa_bwd launch: one Q/dO stage of its
 * first CTA's second step), so the bounded waits on it run out (about 2 s):
 * the kernel then stops every role, frees its tensor memory and ends, and
 * fa_check_device_error() returns FA_ERR_TIMEOUT.  The output of that
 * launch is incomplete.  The flag is consumed by the next fa_fwd*,
 * fa_fwd_fp8* or fa_bwd call.
 * flags bit 1: the same for the next quantiser call (fa_quant_fp8,
 * fa_quant_fp8_rope or fa_quant_fp8_per_tensor_noalloc): the first CTA of its
 * first launch leaves one input slot unfilled; the blocks it cannot finish
 * get a NaN descale (per-tensor: an infinite maximum) and the error word is
 * set.
 * flags = 0 clears pending injections.  Values outside 0..3:
 * FA_ERR_INVALID_ARG.
 */
fa_status fa_debug_inject(int flags);

/*
 * fa_debug_exp2 -- TEST HOOK: evaluates, element by element, y[i] = 2^x[i]
 * the ways the forward kernels can compute the exponentials of P: method 0
 * with the special-function unit's ex2 as the shipped kernels do
 * (approximate, subnormal results flushed to zero), method 3 or 4 with the
 * FMA-pipe polynomial of that degree that the ablation variant 64 of
 * fa_ablate.h uses for a share of P (range
 * reduction x = n + f, |f| <= 1/2, minimax polynomial for 2^f; relative
 * error at most 7.5e-5 (degree 3) or 2.6e-6 (degree 4) for -125 <= x <= 127;
 * x below -126 gives a result of at most 2^-125.5; NaN gives NaN).  x, y:
 * device arrays of n fp32 values (y may equal x).  Asynchronous on `stream`.
 * FA_ERR_INVALID_ARG for n < 0, a null pointer with n > 0 or another method.
 */
fa_status fa_debug_exp2(const float* x, float* y, int64_t n, int method, cudaStream_t stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
