/*
 * Oracle for the exact attention forward pass -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  The product (the CUDA library under
 * exact_attention_forward_09_gb300/) never calls it and shares no code,
 * header, table or constant with it.
 *
 * What it computes, and the passages it follows:
 *
 *  oracle_attn_fwd   Scaled dot-product attention O = softmax(scale*Q K^T) V
 *                    [wmrh.cn FlashAttention V3 article, sec. 1.1 "self-attention
 *                    and the O(N^2) problem": scores QK^T, softmax, weighted sum
 *                    of V, with the 1/sqrt(d_k) factor].  The tiled online
 *                    softmax of FlashAttention reaches exactly this result
 *                    [same article, sec. 2.1 "V1 tiling"; "FlashAttention-3:
 *                    async pipelines on Hopper" (charlestar.github.io),
 *                    section "Online Softmax is still the core of exact
 *                    merging"], so the oracle is the plain definition: one row
 *                    of scores materialised, a two-pass softmax, fp64 all
 *                    through.  It also returns the row log-sum-exp
 *                    LSE_i = ln sum_j exp(s_ij), which the pages do not define;
 *                    it is the natural log of the scaled, masked scores.
 *                    Causal masking keeps the lower triangle ["FlashAttention-3:
 *                    async pipelines on Hopper", section "why causal shapes are
 *                    harder to schedule"]: key j is visible to query i iff
 *                    j <= i + (Nk - Nq) (the diagonal included).
 *
 *  oracle_quant_e4m3 Block quantisation to FP8 E4M3 with one scale per
 *                    128-row block, scale = amax / 448 ["FlashAttention-3:
 *                    async pipelines on Hopper", section "why block
 *                    quantization beats a per-tensor scale"; wmrh.cn article,
 *                    sec. 3.3: X_max = 448 for E4M3], optionally after the
 *                    incoherent-processing rotation x -> x diag(sigma) H_d / sqrt(d)
 *                    ["FlashAttention-3: async pipelines on Hopper", section
 *                    "how incoherent processing flattens outliers": random +-1
 *                    diagonal combined with a Hadamard matrix, O(d log d)].
 *                    The rotated value y is fp32 (the fast Walsh-Hadamard
 *                    butterfly with strides 1, 2, 4, ..., the textbook in-place
 *                    order, in fp32), the 1/sqrt(d) factor is carried in the
 *                    stored descale, s = amax / 448 rounded to fp32, and the
 *                    code is the E4M3 value nearest to the exact quotient y / s
 *                    (ties to even, saturated at 448): one rounding, from the
 *                    real number to E4M3, with no fp32 quotient in between.
 *                    The quotient is formed in fp64, which decides that
 *                    rounding exactly: an E4M3 midpoint has at most 5
 *                    significant bits, so y - m s (y and s of 24 bits) is
 *                    either 0 or at least about 2^-30 |y| away from it, far
 *                    beyond fp64's 2^-53 relative rounding of y / s.
 *
 *                    With a rotary position embedding requested, each row is
 *                    first turned pairwise by the caller's angles (the pages
 *                    let RoPE share the quantisation pass, same sections; they
 *                    give no RoPE formula, so it is the usual planar rotation
 *                    of channel pairs (2i, 2i+1) or (i, i + d/2):
 *                    a' = a cos - b sin, b' = a sin + b cos), in fp32 with each
 *                    product rounded before the sum, like the kernel.
 *
 *  oracle_attn_bwd   Gradients dQ, dK, dV of the loss sum(dO * O) for the
 *                    same attention (the pages list the backward pass among
 *                    the paths a test must cover and compare its speed with
 *                    FA2 ["FlashAttention-3: async pipelines on Hopper",
 *                    sections "correctness validation must cover asynchronous
 *                    boundaries" and "how to read the paper's performance
 *                    numbers"], but print no formula).  It is the derivative
 *                    of the definition above, written out per query row with
 *                    the row of probabilities materialised:
 *                      P_ij  = exp(s_ij - m_i) / l_i       (visible j only)
 *                      dP_ij = dO_i . v_j
 *                      D_i   = sum_j P_ij dP_ij
 *                      dS_ij = P_ij (dP_ij - D_i)
 *                      dQ_i  = scale sum_j dS_ij k_j
 *                      dK_j  = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i,
 *                    the last two summed over every query head of the
 *                    key/value head's group.
 *
 *  oracle_e4m3_encode / oracle_e4m3_decode
 *                    The E4M3 format from its definition: 1 sign bit, 4
 *                    exponent bits (bias 7), 3 mantissa bits, subnormals at
 *                    exponent field 0, largest finite value 448, code 0x7f/0xff
 *                    NaN, no infinities.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Attention, fp64.                                                          */
/* ------------------------------------------------------------------------ */

/*
 * q   [B, Hq,  Nq, d]   k, v [B, Hkv, Nk, d]   (row-major, contiguous)
 * rows: optional list of nrows query indices (NULL -> all Nq rows)
 * o   [B, Hq, R, d]     lse [B, Hq, R]          with R = rows ? nrows : Nq
 * Query head h reads key/value head h / (Hq / Hkv).
 * A query with no visible key gets o = 0 and lse = -inf.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attn_fwd(const double* q, const double* k, const double* v,
                    double* o, double* lse,
                    int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk,
                    int64_t d, int causal, double scale,
                    const int64_t* rows, int64_t nrows, int nthreads)
{
    if (B < 0 || Hq < 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int64_t R = rows ? nrows : Nq;
    const int64_t group = Hq / Hkv;
    const int64_t total = B * Hq * R;
    int bad = 0;
    if (nthreads <= 0) nthreads = 1;

#pragma omp parallel num_threads(nthreads)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s || !acc) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < total; ++t) {
            if (!s || !acc) continue;
            const int64_t bh = t / R;          /* (b, h) flattened           */
            const int64_t r = t % R;
            const int64_t b = bh / Hq, h = bh % Hq;
            const int64_t i = rows ? rows[r] : r;
            const double* qi = q + ((b * Hq + h) * Nq + i) * d;
            const double* kb = k + (b * Hkv + h / group) * Nk * d;
            const double* vb = v + (b * Hkv + h / group) * Nk * d;
            double* oi = o + (bh * R + r) * d;

            /* visible keys: j < jend */
            int64_t jend = Nk;
            if (causal) {
                int64_t lim = i + (Nk - Nq) + 1;
                if (lim < jend) jend = lim;
                if (jend < 0) jend = 0;
            }
            if (jend == 0) {
                for (int64_t c = 0; c < d; ++c) oi[c] = 0.0;
                lse[bh * R + r] = -INFINITY;
                continue;
            }
            /* pass 1: scores and their maximum */
            double m = -INFINITY;
            for (int64_t j = 0; j < jend; ++j) {
                const double* kj = kb + j * d;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += qi[c] * kj[c];
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            /* pass 2: exponentials, their sum, and the weighted sum of V */
            double l = 0.0;
            for (int64_t c = 0; c < d; ++c) acc[c] = 0.0;
            for (int64_t j = 0; j < jend; ++j) {
                const double p = exp(s[j] - m);
                const double* vj = vb + j * d;
                l += p;
                for (int64_t c = 0; c < d; ++c) acc[c] += p * vj[c];
            }
            for (int64_t c = 0; c < d; ++c) oi[c] = acc[c] / l;
            lse[bh * R + r] = m + log(l);
        }
        free(s);
        free(acc);
    }
    return bad ? -1 : 0;
}

/*
 * Backward pass.  q, dout, dq [B, Hq, Nq, d]; k, v, dk, dv [B, Hkv, Nk, d].
 * Work is split over (b, key/value head), so each thread owns the dK and dV
 * rows it accumulates into.  A query with no visible key gets dq = 0 and
 * contributes nothing.  Returns 0, or -1 on bad arguments / allocation
 * failure.
 */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv,
                    int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk,
                    int64_t d, int causal, double scale, int nthreads)
{
    if (B < 0 || Hq < 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int64_t group = Hq / Hkv;
    const int64_t total = B * Hkv;
    int bad = 0;
    if (nthreads <= 0) nthreads = 1;

#pragma omp parallel num_threads(nthreads)
    {
        const size_t nk1 = (size_t)(Nk > 0 ? Nk : 1);
        double* p = (double*)malloc(sizeof(double) * nk1);
        double* dp = (double*)malloc(sizeof(double) * nk1);
        if (!p || !dp) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < total; ++t) {
            if (!p || !dp) continue;
            const int64_t b = t / Hkv, hk = t % Hkv;
            const double* kb = k + (b * Hkv + hk) * Nk * d;
            const double* vbase = v + (b * Hkv + hk) * Nk * d;
            double* dkb = dk + (b * Hkv + hk) * Nk * d;
            double* dvb = dv + (b * Hkv + hk) * Nk * d;
            for (int64_t e = 0; e < Nk * d; ++e) {
                dkb[e] = 0.0;
                dvb[e] = 0.0;
            }
            for (int64_t h = hk * group; h < (hk + 1) * group; ++h) {
                for (int64_t i = 0; i < Nq; ++i) {
                    const int64_t row = (b * Hq + h) * Nq + i;
                    const double* qi = q + row * d;
                    const double* doi = dout + row * d;
                    double* dqi = dq + row * d;
                    for (int64_t c = 0; c < d; ++c) dqi[c] = 0.0;
                    int64_t jend = Nk;
                    if (causal) {
                        const int64_t visible = i + (Nk - Nq) + 1;
                        if (visible < jend) jend = visible;
                        if (jend < 0) jend = 0;
                    }
                    if (jend == 0) continue;
                    /* probabilities of the row */
                    double m = -INFINITY;
                    for (int64_t j = 0; j < jend; ++j) {
                        const double* kj = kb + j * d;
                        double qk = 0.0;
                        for (int64_t c = 0; c < d; ++c) qk += qi[c] * kj[c];
                        p[j] = scale * qk;
                        if (p[j] > m) m = p[j];
                    }
                    double l = 0.0;
                    for (int64_t j = 0; j < jend; ++j) {
                        p[j] = exp(p[j] - m);
                        l += p[j];
                    }
                    for (int64_t j = 0; j < jend; ++j) p[j] /= l;
                    /* dP = dO_i . v_j and D_i = sum_j P dP */
                    double Di = 0.0;
                    for (int64_t j = 0; j < jend; ++j) {
                        const double* vj = vbase + j * d;
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += doi[c] * vj[c];
                        dp[j] = dot;
                        Di += p[j] * dot;
                    }
                    for (int64_t j = 0; j < jend; ++j) {
                        const double ds = p[j] * (dp[j] - Di);
                        const double* kj = kb + j * d;
                        double* dkj = dkb + j * d;
                        double* dvj = dvb + j * d;
                        for (int64_t c = 0; c < d; ++c) {
                            dqi[c] += scale * ds * kj[c];
                            dkj[c] += scale * ds * qi[c];
                            dvj[c] += p[j] * doi[c];
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 codec.                                                           */
/* ------------------------------------------------------------------------ */

/* Nearest E4M3 value to x (ties to even), saturated at +-448. */
uint8_t oracle_e4m3_encode_f64(double x)
{
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    const double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);          /* saturate     */
    if (a < 0.015625) {                                      /* < 2^-6       */
        /* subnormal spacing 2^-9; a*512 is exact; nearbyint rounds half to
         * even in the default rounding mode.  q == 8 is the smallest normal
         * (exponent field 1, mantissa 0), whose code is also 8.             */
        const double qn = nearbyint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)qn);
    }
    int e2;
    (void)frexp(a, &e2);                                     /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    double qn = nearbyint(ldexp(a, 3 - E));                  /* 8 .. 16      */
    if (qn == 16.0) { qn = 8.0; E += 1; }
    const int field = E + 7;
    if (field > 15 || (field == 15 && (int)qn - 8 > 6)) return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (uint8_t)((field << 3) | ((int)qn - 8)));
}

uint8_t oracle_e4m3_encode(float x)
{
    return oracle_e4m3_encode_f64((double)x);
}

float oracle_e4m3_decode(uint8_t c)
{
    const int e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (c & 0x80) ? (float)-v : (float)v;
}

void oracle_e4m3_encode_array(const float* x, uint8_t* c, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) c[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t* c, float* x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) x[i] = oracle_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------------ */
/* Rotation and quantisation, fp32.                                          */
/* ------------------------------------------------------------------------ */

/* y <- H_d (sigma o x): sign flip, then the Walsh-Hadamard butterfly with
 * strides 1, 2, 4, ..., d/2 (Sylvester / natural order), fp32.  No 1/sqrt(d). */
void oracle_fwht_f32(const float* x, float* y, int64_t d, const int8_t* signs)
{
    for (int64_t c = 0; c < d; ++c) y[c] = (signs && signs[c] < 0) ? -x[c] : x[c];
    for (int64_t h = 1; h < d; h *= 2) {
        for (int64_t base = 0; base < d; base += 2 * h) {
            for (int64_t c = base; c < base + h; ++c) {
                const float a = y[c], b = y[c + h];
                y[c] = a + b;
                y[c + h] = a - b;
            }
        }
    }
}

/* Rotary embedding of one row: pairs (2i, 2i+1) (layout 1) or (i, i + d/2)
 * (layout 2) turned by angle i of the row: c[i] = cos, s[i] = sin, fp32. */
void oracle_rope_f32(const float* x, float* y, int64_t d, const float* c, const float* s, int layout)
{
    const int64_t half = d / 2;
    for (int64_t i = 0; i < half; ++i) {
        const int64_t ia = (layout == 1) ? 2 * i : i;
        const int64_t ib = (layout == 1) ? 2 * i + 1 : i + half;
        const float a = x[ia], b = x[ib];
        const float ac = a * c[i], bs = b * s[i], as = a * s[i], bc = b * c[i];
        y[ia] = ac - bs;
        y[ib] = as + bc;
    }
}

/*
 * x        [BH, N, d] fp32
 * codes    [BH, N, d] e4m3 codes
 * descale  [BH, ceil(N / block_rows)] fp32: dequantised value = code * descale
 * signs    d entries of +-1 (rotation on), or NULL (rotation off); d must then
 *          be a power of two.
 * per_tensor: one scale over the whole tensor instead of one per block.
 * rope_layout: 0 none, else 1 or 2 (see oracle_rope_f32), with rope_cos /
 *          rope_sin [N, d/2]: row n of every (b,h) uses row n of the tables.
 */
int oracle_quant_e4m3(const float* x, uint8_t* codes, float* descale,
                      int64_t BH, int64_t N, int64_t d, int64_t block_rows,
                      const int8_t* signs, int per_tensor,
                      const float* rope_cos, const float* rope_sin, int rope_layout)
{
    if (BH < 0 || N < 0 || d <= 0 || block_rows <= 0) return -1;
    if (signs && (d & (d - 1)) != 0) return -1;
    if (rope_layout && (rope_layout != 1 && rope_layout != 2)) return -1;
    if (rope_layout && (!rope_cos || !rope_sin || (d & 1))) return -1;
    const int64_t nblk = (N + block_rows - 1) / block_rows;
    const int64_t n = BH * N * d;
    float* y = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    if (!y) return -1;
    float* t = (float*)malloc(sizeof(float) * (size_t)d);
    if (!t) { free(y); return -1; }
    for (int64_t r = 0; r < BH * N; ++r) {
        const float* xr = x + r * d;
        if (rope_layout) {
            const int64_t n = r % N;
            oracle_rope_f32(xr, t, d, rope_cos + n * (d / 2), rope_sin + n * (d / 2), rope_layout);
            xr = t;
        }
        if (signs) oracle_fwht_f32(xr, y + r * d, d, signs);
        else memcpy(y + r * d, xr, sizeof(float) * (size_t)d);
    }
    free(t);
    const float rinv = signs ? (float)(1.0 / sqrt((double)d)) : 1.0f;

    float gmax = 0.0f;
    if (per_tensor)
        for (int64_t i = 0; i < n; ++i) { float a = fabsf(y[i]); if (a > gmax) gmax = a; }

    for (int64_t bh = 0; bh < BH; ++bh) {
        for (int64_t blk = 0; blk < nblk; ++blk) {
            const int64_t r0 = blk * block_rows;
            const int64_t r1 = (r0 + block_rows < N) ? r0 + block_rows : N;
            const float* yb = y + (bh * N + r0) * d;
            const int64_t cnt = (r1 - r0) * d;
            float amax = 0.0f;
            if (per_tensor) amax = gmax;
            else for (int64_t i = 0; i < cnt; ++i) { float a = fabsf(yb[i]); if (a > amax) amax = a; }
            const float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
            uint8_t* cb = codes + (bh * N + r0) * d;
            for (int64_t i = 0; i < cnt; ++i) cb[i] = oracle_e4m3_encode_f64((double)yb[i] / (double)s);
            descale[bh * nblk + blk] = s * rinv;
        }
    }
    free(y);
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
