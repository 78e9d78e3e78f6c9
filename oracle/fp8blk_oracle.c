/*
 * CPU oracle for the block-scaled FP8 linear-algebra path.
 *
 * TEST INFRASTRUCTURE ONLY. This file defines what the CUDA library must
 * compute. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load it; the library never does, and it shares no code, header, table
 * or constant with the library. It is written for clarity, not speed: plain
 * loops, one element at a time, fp64 where the pages leave the precision
 * free.
 *
 * Sources (the DeepSeek-V3 inference pages):
 *   [AQ] "Administrator & Developer Guide", 8.5.1 act_quant_kernel: per
 *        128-element block, absolute max, clamp to 1e-4, divide by 448 to get
 *        the scale; with scale_fmt "ue8m0" round the scale up to 2^ceil(log2 s);
 *        y = x / s cast to float8_e4m3fn; 448 is the largest e4m3fn magnitude.
 *   [WD] same guide, 8.5.2 weight_dequant_kernel: a 128x128 fp8 tile as fp32,
 *        times its single block scale, stored in the default dtype (bf16).
 *   [GM] same guide, 8.5.3 fp8_gemm_kernel: fp32 accumulator, per 128-wide K
 *        tile acc += dot(a, b) * a_s[:, None] * b_s[None, :]; a_s per row per
 *        K tile, b_s per 128x128 weight block.
 *   [SC] same guide, 6.3 The FP8 path, item 2: weight scale shape
 *        (ceil(out/128), ceil(in/128)), fp32.
 *   [PD] "Algolia docsearch" page (README), 3 "Dequantize FP8 weights using
 *        weight_scale_inv": (128x128 block) * weight_scale_inv; a block not
 *        aligned to 128 is zero-padded to 128 for the scale calculation.
 *   [UE] "User Guide", 7 FAQ "What is scale_fmt: ue8m0?": a pure power-of-two
 *        scale, rounded up.
 *   [MO] "Administrator & Developer Guide", 6.4 MoE expert routing and 8.4
 *        steps 2-5: per expert, the tokens routed to it, weighted by their
 *        gate weight, summed into y.
 *   [ML] same guide, 1.2 module map (MLP / Expert): w2(silu(w1 x) * w3 x).
 *   [MA] same guide, 8.3 MLA forward, steps 5 and 7 ("absorb"): q_nope is
 *        folded through wkv_b's no-positional rows, einsum("bshd,hdc->bshc"),
 *        and the attention output is projected to V through its last v rows,
 *        einsum("bshc,hdc->bshd"); wkv_b stored FP8 is used as its
 *        weight_dequant (8.5.2: fp32 code times block scale, stored bf16).
 *   [GT] same guide, 8.4 (the Gate: with n_groups > 1 the scores are viewed as
 *        groups, a group's score is its max without a bias and the sum of its
 *        top two with one, the top topk_groups groups are kept and the rest
 *        masked to -inf, then the top-k experts are picked) and 3.3 (score_func
 *        softmax or sigmoid, route_scale, expert groups and limited groups per
 *        config); "Repository overview" page, MoE data flow (scores, optional
 *        group masking, top-k indices, gather the original scores, normalize,
 *        route_scale); "User Guide", 7 FAQ (the gate bias of the dim-7168
 *        configs, used with sigmoid scores).
 *
 * Readings where the pages are silent:
 *   - "x / s" and "amax / 448" are IEEE fp32 divisions, correctly rounded.
 *   - e4m3 conversion rounds to nearest, ties to even, and saturates to
 *     +-448 (satfinite); zero and underflow keep their sign.
 *   - the ue8m0 scale is kept as an fp32 number holding a power of two.
 *   - bf16 output of a product or sum is round-to-nearest-even.
 *   - the synthetic master weights are quantised with the act_quant rule
 *     over each 128x128 block (edge blocks: only the real elements, which is
 *     the same amax as zero padding).
 *
 * Parity status of every function is pinned by tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define ORC_BLOCK 128
#define ORC_E4M3_MAX 448.0

/* ---- rounding to a binary floating-point format ------------------------ */

/* Round x to the nearest number with p significand bits whose exponent is at
 * least emin (numbers below 2^emin are subnormal in that format), ties to
 * even. No overflow handling: the callers bound the range. ldexp and ilogb
 * are exact; nearbyint rounds to nearest-even in the default mode. */
static double round_to_format(double x, int p, int emin)
{
    if (x == 0.0 || isnan(x) || isinf(x))
        return x;
    int e = ilogb(x);
    if (e < emin)
        e = emin;
    int q = e - (p - 1);          /* exponent of one unit in the last place */
    double y = ldexp(x, -q);      /* |y| < 2^p: exact */
    return ldexp(nearbyint(y), q);
}

/* ---- e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits ------ */

double orc_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int ex = (code >> 3) & 15;
    int man = code & 7;
    double v;
    if (ex == 15 && man == 7)
        return NAN;                               /* 0x7F, 0xFF: NaN */
    if (ex == 0)
        v = ldexp((double)man, -9);               /* subnormal: man * 2^-9 */
    else
        v = ldexp((double)(8 + man), ex - 10);    /* (1 + man/8) * 2^(ex-7) */
    return sign ? -v : v;
}

uint8_t orc_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    double r = round_to_format(a, 4, -6);  /* 4 significand bits, min normal 2^-6 */
    if (r > ORC_E4M3_MAX)
        r = ORC_E4M3_MAX;                  /* satfinite */
    if (r == 0.0)
        return sign;
    int e = ilogb(r);
    uint8_t code;
    if (e < -6) {
        code = (uint8_t)ldexp(r, 9);              /* subnormal field: r / 2^-9 */
    } else {
        int man = (int)(ldexp(r, -e) * 8.0) - 8;  /* r = (1 + man/8) 2^e */
        code = (uint8_t)(((e + 7) << 3) | man);
    }
    return (uint8_t)(sign | code);
}

/* ---- bf16 --------------------------------------------------------------- */

double orc_bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to bf16 (8 significand bits, fp32's exponent range) in one
 * step, ties to even, and return the bit pattern. */
uint16_t orc_bf16_encode(double x)
{
    if (isnan(x))
        return 0x7FC0;
    double r = round_to_format(x, 8, -126);
    float f = (float)r;   /* exact: r is representable in fp32 */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* ---- scale rule [AQ], [UE] ---------------------------------------------- */

/* Scale of one block from its absolute max: clamp to 1e-4, divide by 448
 * (fp32); with ue8m0 round up to the next power of two, 2^ceil(log2 s). */
float orc_block_scale(float amax, int ue8m0)
{
    float s = fmaxf(amax, 1e-4f) / 448.0f;
    if (ue8m0) {
        int e;
        double f = frexp((double)s, &e);   /* s = f * 2^e, f in [0.5, 1) */
        if (f != 0.5)
            s = (float)ldexp(1.0, e);      /* s in (2^(e-1), 2^e) -> 2^e */
    }
    return s;
}

/* ---- A1 act_quant [AQ] -------------------------------------------------- */

/* x: bf16 bits [M, K] row-major, K % 128 == 0.
 * q: e4m3 codes [M, K]; s: fp32 [M, K/128]. */
void orc_act_quant(const uint16_t *x, int64_t M, int64_t K, int ue8m0,
                   uint8_t *q, float *s)
{
    int64_t nb = K / ORC_BLOCK;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t *xb = x + m * K + b * ORC_BLOCK;
            float amax = 0.0f;
            for (int i = 0; i < ORC_BLOCK; ++i) {
                float v = (float)fabs(orc_bf16_decode(xb[i]));
                if (v > amax)
                    amax = v;
            }
            float sc = orc_block_scale(amax, ue8m0);
            s[m * nb + b] = sc;
            for (int i = 0; i < ORC_BLOCK; ++i) {
                float v = (float)orc_bf16_decode(xb[i]);
                q[m * K + b * ORC_BLOCK + i] = orc_e4m3_encode(v / sc);
            }
        }
    }
}

/* ---- weight quantisation (synthetic inputs) [PD], [SC] ------------------ */

/* w: fp32 [N, K]; any N, K >= 1. q: e4m3 [N, K]; s: [ceil(N/128), ceil(K/128)].
 * Each 128x128 block (edge blocks: the real elements, i.e. the block padded
 * with zeros, which changes no absolute max) gets the scale rule above. */
void orc_weight_quant(const float *w, int64_t N, int64_t K, int ue8m0,
                      uint8_t *q, float *s)
{
    int64_t nbn = (N + ORC_BLOCK - 1) / ORC_BLOCK;
    int64_t nbk = (K + ORC_BLOCK - 1) / ORC_BLOCK;
    for (int64_t bn = 0; bn < nbn; ++bn) {
        for (int64_t bk = 0; bk < nbk; ++bk) {
            float amax = 0.0f;
            for (int64_t n = bn * ORC_BLOCK; n < N && n < (bn + 1) * ORC_BLOCK; ++n)
                for (int64_t k = bk * ORC_BLOCK; k < K && k < (bk + 1) * ORC_BLOCK; ++k) {
                    float v = fabsf(w[n * K + k]);
                    if (v > amax)
                        amax = v;
                }
            float sc = orc_block_scale(amax, ue8m0);
            s[bn * nbk + bk] = sc;
            for (int64_t n = bn * ORC_BLOCK; n < N && n < (bn + 1) * ORC_BLOCK; ++n)
                for (int64_t k = bk * ORC_BLOCK; k < K && k < (bk + 1) * ORC_BLOCK; ++k)
                    q[n * K + k] = orc_e4m3_encode(w[n * K + k] / sc);
        }
    }
}

/* ---- A3 weight_dequant [WD], [PD] --------------------------------------- */

/* out[n, k] = bf16( fp32(decode(q[n, k])) * s[n/128, k/128] ), the product an
 * fp32 multiply. out is bf16 bits [N, K]. */
void orc_weight_dequant(const uint8_t *q, const float *s, int64_t N, int64_t K,
                        uint16_t *out)
{
    int64_t nbk = (K + ORC_BLOCK - 1) / ORC_BLOCK;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            float v = (float)orc_e4m3_decode(q[n * K + k]);
            float p = v * s[(n / ORC_BLOCK) * nbk + k / ORC_BLOCK];
            out[n * K + k] = orc_bf16_encode((double)p);
        }
}

/* ---- A2 fp8_gemm [GM] ---------------------------------------------------- */

/* One output element in fp64:
 *   sum over K blocks kb of a_s[m, kb] * w_s[n/128, kb] *
 *       sum over k in kb of decode(qa[m, k]) * decode(qw[n, k]).
 * The inner sums are exact in fp64 (128 products of at most 448^2). */
static double gemm_point(const uint8_t *qa, const float *as, const uint8_t *qw,
                         const float *ws, int64_t K, int64_t m, int64_t n)
{
    int64_t nbk = K / ORC_BLOCK;
    double total = 0.0;
    for (int64_t kb = 0; kb < nbk; ++kb) {
        double inner = 0.0;
        for (int64_t k = kb * ORC_BLOCK; k < (kb + 1) * ORC_BLOCK; ++k)
            inner += orc_e4m3_decode(qa[m * K + k]) * orc_e4m3_decode(qw[n * K + k]);
        total += (double)as[m * nbk + kb] * (double)ws[(n / ORC_BLOCK) * nbk + kb] * inner;
    }
    return total;
}

/* Full reference product, fp64 [M, N]. */
void orc_gemm(const uint8_t *qa, const float *as, const uint8_t *qw, const float *ws,
              int64_t M, int64_t N, int64_t K, double *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out[m * N + n] = gemm_point(qa, as, qw, ws, K, m, n);
}

/* Selected elements (ms[i], ns[i]) of the reference product. */
void orc_gemm_points(const uint8_t *qa, const float *as, const uint8_t *qw,
                     const float *ws, int64_t K, const int64_t *ms,
                     const int64_t *ns, int64_t npts, double *out)
{
    for (int64_t i = 0; i < npts; ++i)
        out[i] = gemm_point(qa, as, qw, ws, K, ms[i], ns[i]);
}

/* ---- A4 SwiGLU between the Linears [ML] --------------------------------- */

/* Each Linear returns bf16 (the default dtype), so h1 = bf16(w1 x) and
 * h3 = bf16(w3 x) arrive as bf16. g = bf16(silu(h1)) with
 * silu(v) = v / (1 + e^-v) evaluated in fp64; u = bf16(fp32(g) * fp32(h3)),
 * the product an fp32 multiply. All arrays are bf16 bits of length n. */
void orc_swiglu(const uint16_t *h1, const uint16_t *h3, int64_t n, uint16_t *u)
{
    for (int64_t i = 0; i < n; ++i) {
        double v = orc_bf16_decode(h1[i]);
        uint16_t g = orc_bf16_encode(v / (1.0 + exp(-v)));
        float p = (float)orc_bf16_decode(g) * (float)orc_bf16_decode(h3[i]);
        u[i] = orc_bf16_encode((double)p);
    }
}

/* ---- A5 MoE permutation [MO] -------------------------------------------- */

/* Groups the T*topk (token, slot) pairs by expert, keeping their original
 * order (t * topk + j) inside each expert. counts[e] = number of pairs routed
 * to e (a bincount); offsets[e] = exclusive prefix sum, offsets[E] = T*topk;
 * perm[offsets[e] + r] = t * topk + j of the r-th pair of expert e.
 * Returns 0, or -1 when an index lies outside [0, E). */
int orc_moe_permute(const int32_t *idx, int64_t T, int64_t topk, int64_t E,
                    int32_t *counts, int32_t *offsets, int32_t *perm)
{
    for (int64_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t i = 0; i < T * topk; ++i) {
        if (idx[i] < 0 || idx[i] >= E)
            return -1;
        counts[idx[i]] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    for (int64_t e = 0; e < E; ++e) {
        int32_t r = offsets[e];
        for (int64_t i = 0; i < T * topk; ++i)
            if (idx[i] == e)
                perm[r++] = (int32_t)i;
    }
    return 0;
}

/* ---- A4/A6/A7 one routed expert FFN and the weighted combine [MO], [ML] -- */

/* Expert FFN of one token whose activation is already quantised
 * (xq: e4m3 [dim], xs: fp32 [dim/128]), with block-quantised weights
 * w1, w3: [inter, dim] (scales [inter/128, dim/128]) and
 * w2: [dim, inter] (scales [dim/128, inter/128]). Writes the fp64 output of
 * the w2 Linear, o [dim]. Scratch: 3*inter uint16 + inter bytes +
 * inter/128 floats, allocated here. Steps: h1 = bf16(w1 x), h3 = bf16(w3 x),
 * u = swiglu(h1, h3), (uq, us) = act_quant(u), o = fp64 product uq w2^T. */
int orc_expert_ffn_u(const uint8_t *xq, const float *xs,
                     const uint8_t *w1, const float *w1s,
                     const uint8_t *w3, const float *w3s,
                     const uint8_t *w2, const float *w2s,
                     int64_t dim, int64_t inter, int ue8m0, double *o,
                     uint8_t *uq_out, float *us_out);

int orc_expert_ffn(const uint8_t *xq, const float *xs,
                   const uint8_t *w1, const float *w1s,
                   const uint8_t *w3, const float *w3s,
                   const uint8_t *w2, const float *w2s,
                   int64_t dim, int64_t inter, int ue8m0, double *o)
{
    return orc_expert_ffn_u(xq, xs, w1, w1s, w3, w3s, w2, w2s, dim, inter, ue8m0, o, NULL, NULL);
}

/* The same, also copying out the quantised intermediate u (uq_out: e4m3
 * [inter], us_out: fp32 [inter/128]) when those pointers are not NULL. */
int orc_expert_ffn_u(const uint8_t *xq, const float *xs,
                     const uint8_t *w1, const float *w1s,
                     const uint8_t *w3, const float *w3s,
                     const uint8_t *w2, const float *w2s,
                     int64_t dim, int64_t inter, int ue8m0, double *o,
                     uint8_t *uq_out, float *us_out)
{
    uint16_t *h1 = malloc(sizeof(uint16_t) * inter);
    uint16_t *h3 = malloc(sizeof(uint16_t) * inter);
    uint16_t *u = malloc(sizeof(uint16_t) * inter);
    uint8_t *uq = malloc((size_t)inter);
    float *us = malloc(sizeof(float) * (inter / ORC_BLOCK));
    if (!h1 || !h3 || !u || !uq || !us) {
        free(h1); free(h3); free(u); free(uq); free(us);
        return -1;
    }
    for (int64_t i = 0; i < inter; ++i) {
        h1[i] = orc_bf16_encode(gemm_point(xq, xs, w1, w1s, dim, 0, i));
        h3[i] = orc_bf16_encode(gemm_point(xq, xs, w3, w3s, dim, 0, i));
    }
    orc_swiglu(h1, h3, inter, u);
    orc_act_quant(u, 1, inter, ue8m0, uq, us);
    for (int64_t c = 0; c < dim; ++c)
        o[c] = gemm_point(uq, us, w2, w2s, inter, 0, c);
    if (uq_out)
        memcpy(uq_out, uq, (size_t)inter);
    if (us_out)
        memcpy(us_out, us, sizeof(float) * (inter / ORC_BLOCK));
    free(h1); free(h3); free(u); free(uq); free(us);
    return 0;
}

/* MoE output of one token t: y[t] = bf16( sum over slots j in order of
 * fp64(w[t, j]) * fp64(bf16(o_j)) ), o_j the expert FFN of expert idx[t, j].
 * With n_shared > 0 (Guide 8.4 steps 6 and 8: the shared MLP runs on every
 * token and the result is y + z), experts E .. E+n_shared-1 are shared:
 * z = bf16( sum of their bf16 outputs ) and the row is bf16(y + z).
 * Expert e's weights sit at row offset e*inter (w1, w3) and e*dim (w2) of the
 * stacked tensors; their scales at block-row offset e*inter/128 and
 * e*dim/128. y_row: bf16 bits [dim]. */
int orc_moe_token(const uint8_t *xq, const float *xs,
                  const int32_t *idx, const float *wts, int64_t t, int64_t topk,
                  const uint8_t *w1, const float *w1s,
                  const uint8_t *w3, const float *w3s,
                  const uint8_t *w2, const float *w2s,
                  int64_t dim, int64_t inter, int ue8m0, int64_t E, int64_t n_shared, uint16_t *y_row)
{
    int64_t kbd = dim / ORC_BLOCK, kbi = inter / ORC_BLOCK;
    double *acc = calloc((size_t)dim, sizeof(double));
    double *accs = calloc((size_t)dim, sizeof(double));
    double *o = malloc(sizeof(double) * dim);
    if (!acc || !accs || !o) {
        free(acc); free(accs); free(o);
        return -1;
    }
    /* routed slots, then (step 6 of 8.4) the shared experts E .. E+n_shared-1 */
    for (int64_t j = 0; j < topk + n_shared; ++j) {
        int64_t e = j < topk ? idx[t * topk + j] : E + (j - topk);
        int rc = orc_expert_ffn(xq + t * dim, xs + t * kbd,
                                w1 + e * inter * dim, w1s + e * (inter / ORC_BLOCK) * kbd,
                                w3 + e * inter * dim, w3s + e * (inter / ORC_BLOCK) * kbd,
                                w2 + e * dim * inter, w2s + e * (dim / ORC_BLOCK) * kbi,
                                dim, inter, ue8m0, o);
        if (rc) {
            free(acc); free(accs); free(o);
            return rc;
        }
        double wj = j < topk ? (double)wts[t * topk + j] : 1.0;
        double *dst = j < topk ? acc : accs;
        for (int64_t c = 0; c < dim; ++c)
            dst[c] += wj * orc_bf16_decode(orc_bf16_encode(o[c]));
    }
    /* y = routed sum (bf16); with shared experts the output is bf16(y + z),
     * z = bf16 of their summed (bf16) outputs: the guide's "Return (y + z)" */
    for (int64_t c = 0; c < dim; ++c) {
        if (n_shared == 0) {
            y_row[c] = orc_bf16_encode(acc[c]);
        } else {
            double y = orc_bf16_decode(orc_bf16_encode(acc[c]));
            double z = orc_bf16_decode(orc_bf16_encode(accs[c]));
            y_row[c] = orc_bf16_encode(y + z);
        }
    }
    free(acc); free(accs); free(o);
    return 0;
}

/* ---- MLA absorb projections [MA] ------------------------------------------ */

/* wkv_b: e4m3 [H*(dn+dv), C] with block scales [H*(dn+dv)/128, C/128]; head h
 * owns rows h*(dn+dv) .. +dn (no-positional part) and the next dv rows (v).
 * Weights are used as weight_dequant gives them: W = bf16(fp32(code) * s).
 * mode 0 (qk): in = q_nope bf16 [T, H, dn], out[t,h,c] = bf16( sum_d q[t,h,d] * W[h*(dn+dv)+d, c] ), out [T, H, C];
 * mode 1 (v):  in = x bf16 [T, H, C],      out[t,h,d] = bf16( sum_c x[t,h,c] * W[h*(dn+dv)+dn+d, c] ), out [T, H, dv].
 * Sums in fp64 (exact products of two bf16 numbers), one bf16 rounding. */
static double mla_w(const uint8_t *w, const float *ws, int64_t C, int64_t row, int64_t col)
{
    float f = (float)orc_e4m3_decode(w[row * C + col]) * ws[(row / ORC_BLOCK) * (C / ORC_BLOCK) + col / ORC_BLOCK];
    return orc_bf16_decode(orc_bf16_encode((double)f));
}

void orc_mla_absorb(const uint16_t *in, const uint8_t *w, const float *ws, int64_t T, int64_t H, int64_t dn,
                    int64_t dv, int64_t C, int mode, uint16_t *out)
{
    const int64_t hs = dn + dv;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            if (mode == 0) {
                const uint16_t *q = in + (t * H + h) * dn;
                for (int64_t c = 0; c < C; ++c) {
                    double acc = 0.0;
                    for (int64_t d = 0; d < dn; ++d)
                        acc += orc_bf16_decode(q[d]) * mla_w(w, ws, C, h * hs + d, c);
                    out[(t * H + h) * C + c] = orc_bf16_encode(acc);
                }
            } else {
                const uint16_t *x = in + (t * H + h) * C;
                for (int64_t d = 0; d < dv; ++d) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < C; ++c)
                        acc += orc_bf16_decode(x[c]) * mla_w(w, ws, C, h * hs + dn + d, c);
                    out[(t * H + h) * dv + d] = orc_bf16_encode(acc);
                }
            }
        }
}

/* ---- MoE gate: scores, group-limited top-k, weights [GT] ----------------- */

/* Per token t: scores s[e] from logits l[t, e] (sigmoid 1/(1+e^-l), or the
 * softmax over all E), computed in fp64 and rounded to fp32 once; selection
 * keys z[e] = s[e] + bias[e] in fp32 (z = s without a bias). With G > 1
 * groups of E/G consecutive experts: a group's score is its largest z (no
 * bias) or the fp32 sum of its two largest z (bias); the TG best groups stay,
 * the others' experts are masked out. The K best unmasked z give the experts,
 * in descending z order; every tie goes to the lower index. The weights are
 * the chosen experts' scores s (not z), divided by their sum when `normalize`
 * is set, times route_scale: fp64, rounded to fp32 once.
 * Returns 0, or -1 on a shape the rules cannot apply to. */
int orc_moe_gate(const float *logits, const float *bias, int64_t T, int64_t E, int64_t G, int64_t TG,
                 int64_t K, int sigmoid, float route_scale, int normalize, int32_t *idx, float *w)
{
    if (E < 1 || G < 1 || E % G || TG < 1 || TG > G || K < 1 || K > TG * (E / G))
        return -1;
    if (bias && G > 1 && E / G < 2)
        return -1;
    float *s = malloc(sizeof(float) * E), *z = malloc(sizeof(float) * E), *gs = malloc(sizeof(float) * G);
    int *allowed = malloc(sizeof(int) * E), *keep = malloc(sizeof(int) * G), *taken = malloc(sizeof(int) * E);
    if (!s || !z || !gs || !allowed || !keep || !taken) {
        free(s); free(z); free(gs); free(allowed); free(keep); free(taken);
        return -1;
    }
    const int64_t GS = E / G;
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        if (sigmoid) {
            for (int64_t e = 0; e < E; ++e)
                s[e] = (float)(1.0 / (1.0 + exp(-(double)l[e])));
        } else {
            double m = (double)l[0], sum = 0.0;
            for (int64_t e = 1; e < E; ++e)
                if ((double)l[e] > m)
                    m = (double)l[e];
            for (int64_t e = 0; e < E; ++e)
                sum += exp((double)l[e] - m);
            for (int64_t e = 0; e < E; ++e)
                s[e] = (float)(exp((double)l[e] - m) / sum);
        }
        for (int64_t e = 0; e < E; ++e) {
            z[e] = bias ? s[e] + bias[e] : s[e];
            allowed[e] = 1;
            taken[e] = 0;
        }
        if (G > 1) {
            for (int64_t g = 0; g < G; ++g) {
                /* the two largest z of the group, first index first on ties */
                int64_t a = g * GS, b = -1;
                for (int64_t e = g * GS + 1; e < (g + 1) * GS; ++e)
                    if (z[e] > z[a])
                        a = e;
                for (int64_t e = g * GS; e < (g + 1) * GS; ++e)
                    if (e != a && (b < 0 || z[e] > z[b]))
                        b = e;
                gs[g] = bias ? z[a] + z[b] : z[a];
                keep[g] = 0;
            }
            for (int64_t r = 0; r < TG; ++r) {
                int64_t best = -1;
                for (int64_t g = 0; g < G; ++g)
                    if (!keep[g] && (best < 0 || gs[g] > gs[best]))
                        best = g;
                keep[best] = 1;
            }
            for (int64_t e = 0; e < E; ++e)
                allowed[e] = keep[e / GS];
        }
        double sum = 0.0;
        for (int64_t j = 0; j < K; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e)
                if (allowed[e] && !taken[e] && (best < 0 || z[e] > z[best]))
                    best = e;
            taken[best] = 1;
            idx[t * K + j] = (int32_t)best;
            sum += (double)s[best];
        }
        for (int64_t j = 0; j < K; ++j) {
            double v = (double)s[idx[t * K + j]];
            if (normalize)
                v /= sum;
            w[t * K + j] = (float)(v * (double)route_scale);
        }
    }
    free(s); free(z); free(gs); free(allowed); free(keep); free(taken);
    return 0;
}

/* ---- array helpers for the pin tests ------------------------------------ */

void orc_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(v[i]);
}

void orc_bf16_encode_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_encode(v[i]);
}
