/*
 * fp8blk -- block-scaled FP8 linear algebra for one NVIDIA GB300 (sm_103a).
 *
 * The operations are those of the DeepSeek-V3 inference kernels as the
 * project's documentation pages describe them:
 *   - act_quant: "Administrator & Developer Guide", 8.5.1 act_quant_kernel;
 *   - weight_dequant: same guide, 8.5.2 weight_dequant_kernel, and the README
 *     ("Algolia docsearch" page) section 3, weight_scale_inv and zero padding;
 *   - fp8_gemm: same guide, 8.5.3 fp8_gemm_kernel, and 6.3 The FP8 path;
 *   - the routed-expert FFN: same guide, 6.4 MoE expert routing and 8.4.
 *
 * Conventions for every entry point:
 *   - Pointers are device pointers unless a name ends in _host. The caller
 *     owns all memory; the library never allocates or frees. Scratch memory
 *     is passed in as `workspace`.
 *   - Matrices are dense and row-major: the last dimension is contiguous
 *     (the pages' kernels assert contiguous 2-D tensors).
 *   - bf16 is IEEE bfloat16 (uint16 storage); e4m3 is float8_e4m3fn (one
 *     byte: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest
 *     magnitude 448, codes 0x7F/0xFF NaN).
 *   - Block size is 128: activation scales are one fp32 per (row, 128
 *     columns), weight scales one fp32 per 128x128 block.
 *   - scale_fmt is FP8BLK_SCALE_FP32 (0) or FP8BLK_SCALE_UE8M0 (1, scales
 *     rounded up to a power of two and still stored as fp32), optionally
 *     with FP8BLK_SCALE_PROMOTE (below).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; 0 = the legacy
 *     default stream). Arguments are checked on the host before any launch;
 *     a failed check launches nothing and returns a non-zero status.
 *   - Sizes of 0 are valid and launch nothing (except where noted).
 *   - Not thread-safe per workspace: calls that share a workspace must be
 *     ordered on one stream.
 *   - Overlap on a stream: the GEMM kernels, the MLA absorb kernels (and
 *     act_quant inside fp8blk_linear / fp8blk_ffn) let the next kernel of
 *     this library on the same stream start early (programmatic dependent
 *     launch). That kernel may begin loading its WEIGHT operands (w, w1, w3,
 *     w2; wkv_b and its scales for the MLA absorb) before the previous one
 *     has finished; it reads activations and activation scales, and writes
 *     anything, only after. Inside fp8blk_linear / fp8blk_ffn the GEMM's
 *     weight loads may even start while the library call before is still
 *     running. So a weight operand must not be the output of either of the
 *     two library calls issued just before it on the same stream. Kernels of
 *     other libraries are ordered as usual.
 */
#ifndef FP8BLK_H
#define FP8BLK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8BLK_API __attribute__((visibility("default")))
#else
#define FP8BLK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *fp8blk_stream_t; /* identical to cudaStream_t */

enum fp8blk_scale_fmt { FP8BLK_SCALE_FP32 = 0, FP8BLK_SCALE_UE8M0 = 1 };

/*
 * OR'ed into FP8BLK_SCALE_UE8M0 (scale_fmt = FP8BLK_SCALE_UE8M0 |
 * FP8BLK_SCALE_PROMOTE): the GEMMs of this call keep the per-128-K promotion
 * (each K block's tensor-core partial scaled by a_s * w_s and added in fp32
 * registers) instead of letting the tensor core apply the power-of-two scales.
 * Same arithmetic, another summation order. Per call, so callers in one
 * process may choose differently. The quantising entry points accept it and
 * quantise as FP8BLK_SCALE_UE8M0. Any other combination is FP8BLK_ERR_ARG.
 */
#define FP8BLK_SCALE_PROMOTE 0x10

enum fp8blk_status {
  FP8BLK_OK = 0,
  FP8BLK_ERR_NULL = 1,        /* a required pointer is NULL */
  FP8BLK_ERR_SHAPE = 2,       /* negative size, K % 128 != 0 where required, size limits */
  FP8BLK_ERR_ALIGN = 3,       /* a pointer is not aligned as documented */
  FP8BLK_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
  FP8BLK_ERR_ARCH = 5,        /* the current device is not sm_103 */
  FP8BLK_ERR_TIMEOUT = 6,     /* a kernel gave up waiting (see fp8blk_last_device_error) */
  FP8BLK_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
  FP8BLK_ERR_ARG = 8,         /* an enum argument is out of range */
  FP8BLK_ERR_TOO_LARGE = 9    /* needs more scratch than fp8blk_gemm_noalloc's built-in buffer */
};

/* Human-readable name of a status code (static string). */
FP8BLK_API const char *fp8blk_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
FP8BLK_API int fp8blk_version(void);

/*
 * act_quant ("Administrator & Developer Guide", 8.5.1): for each row m and
 * 128-column block b of x,
 *     amax = max |x[m, b*128 + i]|                        (fp32)
 *     s    = max(amax, 1e-4) / 448                        (fp32 division)
 *     s    = 2^ceil(log2 s)          if scale_fmt == UE8M0 (exact, rounded up)
 *     q[m, b*128 + i] = e4m3(x / s)  (fp32 division, round to nearest even,
 *                                     saturating at +-448, sign of zero kept)
 * x:  bf16 [M, K], 16-byte aligned.   q: e4m3 [M, K], 16-byte aligned.
 * s:  fp32 [M, K/128], 4-byte aligned.
 * K must be a multiple of 128 (FP8BLK_ERR_SHAPE otherwise, the pages' "Last
 * dimension size must be divisible by block_size").
 */
FP8BLK_API int fp8blk_act_quant(const void *x_bf16, int64_t M, int64_t K, void *q_e4m3, float *s, int scale_fmt,
                     fp8blk_stream_t stream);

/*
 * Block weight quantisation (README section 3: one fp32 scale per 128x128
 * block; a block not aligned to 128 is zero-padded to 128 for the scale
 * calculation and the padding is dropped after quantisation). Each block gets
 * the act_quant rule above over its real elements:
 *     s[bn, bk] = max(amax_block, 1e-4) / 448 (UE8M0: rounded up to 2^k),
 *     q[n, k]   = e4m3(w[n, k] / s[n/128, k/128]).
 * w: fp32 [N, K]; q: e4m3 [N, K]; s: fp32 [ceil(N/128), ceil(K/128)].
 * Any N, K >= 0. Pointers 4-byte aligned (w, s), q unaligned allowed.
 */
FP8BLK_API int fp8blk_weight_quant(const float *w_f32, int64_t N, int64_t K, void *q_e4m3, float *s, int scale_fmt,
                        fp8blk_stream_t stream);

/*
 * weight_dequant ("Administrator & Developer Guide", 8.5.2; README section 3):
 *     out[n, k] = bf16( fp32(q[n, k]) * s[n/128, k/128] )
 * one fp32 multiply, one round-to-nearest-even to bf16.
 * q: e4m3 [N, K]; s: fp32 [ceil(N/128), ceil(K/128)]; out: bf16 [N, K].
 * Any N, K >= 0; edge blocks are partial. No alignment beyond the element
 * size is required (16-byte aligned rows take the vector path).
 */
FP8BLK_API int fp8blk_weight_dequant(const void *q_e4m3, const float *s, int64_t N, int64_t K, void *out_bf16,
                          fp8blk_stream_t stream);

/*
 * fp8_gemm ("Administrator & Developer Guide", 8.5.3 and 6.3):
 *     C[m, n] = sum over 128-wide K blocks kb of
 *               a_s[m, kb] * w_s[n/128, kb] * sum_{k in kb} a[m, k] * w[n, k]
 * accumulated in fp32 (each K block's tensor-core partial is scaled and added
 * to the fp32 accumulator), stored as bf16 (round to nearest even).
 * a:   e4m3 [M, K] (activations, quantised by fp8blk_act_quant), 16-byte aligned.
 * a_s: fp32 [M, K/128].
 * w:   e4m3 [N, K] (weights), 16-byte aligned.
 * w_s: fp32 [ceil(N/128), K/128].
 * c:   bf16 [M, N]. 16-byte alignment and N % 8 == 0 take the vector store path.
 * K must be a multiple of 128; N need not be (the last weight block is
 * partial: rows past N contribute nothing). K == 0 writes zeros.
 * scale_fmt: FP8BLK_SCALE_FP32 or FP8BLK_SCALE_UE8M0 (same arithmetic).
 * Under UE8M0 every a_s and w_s must be a positive normal power of two (as
 * fp8blk_act_quant and fp8blk_weight_quant give them under UE8M0). GEMMs with
 * M > 128 on 128 x 256 tiles (the FFN, expert and large prefill GEMMs) then
 * let the tensor core apply the scales itself (block-scaled MMA,
 * one UE8M0 exponent per operand row and 32-wide K slice), and a scale that
 * is not such a power of two sets device error bit 0x80 (its outputs are
 * undefined). FP8BLK_SCALE_UE8M0 | FP8BLK_SCALE_PROMOTE keeps the per-block
 * promotion for UE8M0 as well.
 * workspace: device memory of at least fp8blk_gemm_workspace_bytes(M, N, K),
 * 256-byte aligned. Its first 64 KB hold the tile counters: ZERO-FILLED
 * before the first use, and every call leaves them at zero; the rest is
 * scratch whose contents do not matter. One workspace serves one stream at a
 * time, for GEMMs of any shape.
 */
FP8BLK_API size_t fp8blk_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
FP8BLK_API int fp8blk_gemm(const void *a_e4m3, const float *a_s, const void *w_e4m3, const float *w_s, void *c_bf16,
                int64_t M, int64_t N, int64_t K, int scale_fmt, void *workspace, size_t workspace_bytes,
                fp8blk_stream_t stream);

/*
 * FP8 linear layer ("Administrator & Developer Guide", 6.3, the gemm_impl
 * "fp8" branch of linear()): y = fp8_gemm(act_quant(x), w) with x bf16 [M, K],
 * w e4m3 [N, K] with scales w_s [ceil(N/128), K/128], y bf16 [M, N].
 * The quantised activation lives in the workspace:
 *     fp8blk_linear_workspace_bytes(M, N, K) bytes, 256-byte aligned, its first
 * 64 KB zero-filled before first use (as for fp8blk_gemm); one workspace
 * serves layers of any shape, one stream at a time.
 */
FP8BLK_API size_t fp8blk_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);
FP8BLK_API int fp8blk_linear(const void *x_bf16, const void *w_e4m3, const float *w_s, void *y_bf16, int64_t M, int64_t N,
                  int64_t K, int scale_fmt, void *workspace, size_t workspace_bytes, fp8blk_stream_t stream);

/*
 * How many kernels one fp8blk_linear call of shape (M, N, K) launches on the
 * current device, written to *kernels: 1 where act_quant runs inside the GEMM
 * kernel (M <= 2, the quantised x fits that kernel's shared memory, and the
 * slice-per-SM decode GEMM does not take the shape), 2 where act_quant and
 * fp8_gemm are kernels of their own, 0 for an empty problem (M, N or K zero).
 * Returns FP8BLK_ERR_NULL for a null kernels, FP8BLK_ERR_SHAPE for a shape
 * fp8blk_linear refuses, FP8BLK_ERR_ARCH / FP8BLK_ERR_CUDA as the device
 * check gives them.
 */
FP8BLK_API int fp8blk_linear_kernels(int64_t M, int64_t N, int64_t K, int *kernels);

/*
 * The same layer with the activation and the result in HOST memory
 * (x_host bf16 [M, K], y_host bf16 [M, N]), enqueued on `stream`; y_host is
 * valid once the stream has been synchronised. The weight stays on the device.
 * Page-locked buffers the device can address (cudaHostAlloc / pinned memory on
 * a unified-address system), 16-byte aligned, are read and written in place by
 * the layer's kernels (no staging copies). Any other buffer is copied to the
 * workspace and back (page-locked memory keeps those copies asynchronous).
 * Workspace: fp8blk_linear_host_workspace_bytes.
 */
FP8BLK_API size_t fp8blk_linear_host_workspace_bytes(int64_t M, int64_t N, int64_t K);
FP8BLK_API int fp8blk_linear_host(const void *x_host_bf16, const void *w_e4m3, const float *w_s, void *y_host_bf16,
                       int64_t M, int64_t N, int64_t K, int scale_fmt, void *workspace, size_t workspace_bytes,
                       fp8blk_stream_t stream);

/*
 * Fused w1/w3 GEMM of the SwiGLU FFN ("Administrator & Developer Guide", 1.2
 * module map: MLP / Expert compute w2(silu(w1 x) * w3 x); 6.3: every Linear
 * quantises its input). With h1 = bf16(x w1^T) and h3 = bf16(x w3^T) (each an
 * fp8_gemm as above):
 *     u = bf16( bf16(silu(h1)) * h3 ),  silu(v) = v / (1 + e^-v) in fp32,
 *     (u_q, u_s) = act_quant(u, scale_fmt)   -- the input of the w2 Linear.
 * x: e4m3 [M, dim] + x_s [M, dim/128]; w1, w3: e4m3 [inter, dim] + scales
 * [inter/128, dim/128]; u_q: e4m3 [M, inter] (16-byte aligned); u_s: fp32
 * [M, inter/128]. dim % 128 == 0, inter % 128 == 0. The act_quant of u happens
 * in the GEMM's epilogue (u never reaches memory in bf16).
 * Workspace: fp8blk_swiglu_workspace_bytes(M, inter, dim), laid out and kept
 * as fp8blk_gemm's (first 64 KB zero-filled before first use, left so).
 */
FP8BLK_API size_t fp8blk_swiglu_workspace_bytes(int64_t M, int64_t inter, int64_t dim);
FP8BLK_API int fp8blk_swiglu_gemm(const void *x_e4m3, const float *x_s, const void *w1_e4m3, const float *w1_s,
                                  const void *w3_e4m3, const float *w3_s, void *u_e4m3, float *u_s, int64_t M,
                                  int64_t inter, int64_t dim, int scale_fmt, void *workspace,
                                  size_t workspace_bytes, fp8blk_stream_t stream);

/*
 * Dense SwiGLU FFN (the guide's MLP with FP8 Linears): y = w2(u) with
 * u from fp8blk_swiglu_gemm on act_quant(x). x: bf16 [M, dim]; w2: e4m3
 * [dim, inter] + scales [dim/128, inter/128]; y: bf16 [M, dim].
 * Workspace: fp8blk_ffn_workspace_bytes(M, dim, inter), first 64 KB zero-filled
 * before first use (left so); one workspace serves FFNs of any shape.
 */
FP8BLK_API size_t fp8blk_ffn_workspace_bytes(int64_t M, int64_t dim, int64_t inter);
FP8BLK_API int fp8blk_ffn(const void *x_bf16, const void *w1_e4m3, const float *w1_s, const void *w3_e4m3,
                          const float *w3_s, const void *w2_e4m3, const float *w2_s, void *y_bf16, int64_t M,
                          int64_t dim, int64_t inter, int scale_fmt, void *workspace, size_t workspace_bytes,
                          fp8blk_stream_t stream);

/*
 * MoE routing permutation ("Administrator & Developer Guide", 6.4: the
 * per-expert bincount, then for each expert the (token, slot) pairs routed to
 * it). topk_idx: int32 [T, topk] expert ids. Outputs (device):
 *     counts[e]   = number of pairs routed to expert e, e < E,
 *     offsets[e]  = exclusive prefix sum of counts, offsets[E] = valid pairs,
 *     perm[offsets[e] + r] = t * topk + j of the r-th pair of expert e, in
 *                   increasing pair order (a stable sort by expert id).
 * Integer work, no host synchronisation. E <= 1024. Ids outside [0, E) join no
 * expert and set a bit read by fp8blk_last_device_error.
 * Workspace: device scratch of fp8blk_moe_permute_workspace_bytes(T, topk, E),
 * 256-byte aligned (ranks and per-chunk bases; any contents on entry).
 */
FP8BLK_API size_t fp8blk_moe_permute_workspace_bytes(int64_t T, int64_t topk, int64_t E);
FP8BLK_API int fp8blk_moe_permute(const int32_t *topk_idx, int64_t T, int64_t topk, int64_t E, int32_t *counts,
                                  int32_t *offsets, int32_t *perm, void *workspace, size_t workspace_bytes,
                                  fp8blk_stream_t stream);

/*
 * MLA "absorb" projections with the FP8 wkv_b ("Administrator & Developer
 * Guide", 8.3 steps 5 and 7, attn_impl "absorb"). wkv_b: e4m3 [H*(dn+dv), C]
 * with 128x128 block scales wkv_b_s fp32 [H*(dn+dv)/128, C/128]; head h owns
 * rows h*(dn+dv) .. +dn (no-positional part) and the dv rows after them (v).
 * W is wkv_b as weight_dequant gives it: bf16(fp32(code) * block scale).
 *   qk: q_nope bf16 [T, H, dn] -> out bf16 [T, H, C],
 *       out[t,h,c] = bf16( sum over d < dn of q_nope[t,h,d] * W[h*(dn+dv) + d, c] );
 *   v:  x bf16 [T, H, C] -> out bf16 [T, H, dv],
 *       out[t,h,d] = bf16( sum over c < C of x[t,h,c] * W[h*(dn+dv) + dn + d, c] ).
 * Products of bf16 numbers summed in fp32 (tensor cores, bf16 inputs). Shapes:
 * dn == dv == 128 (every config's qk_nope_head_dim and v_head_dim), C % 128 == 0
 * (kv_lora_rank), H >= 1, T >= 0; else FP8BLK_ERR_SHAPE. Activations, weights
 * and outputs 16-byte aligned, scales 4-byte aligned. No workspace.
 */
FP8BLK_API int fp8blk_mla_absorb_qk(const void *q_nope_bf16, const void *wkv_b_e4m3, const float *wkv_b_s,
                                    void *out_bf16, int64_t T, int64_t H, int64_t dn, int64_t dv, int64_t C,
                                    fp8blk_stream_t stream);
FP8BLK_API int fp8blk_mla_absorb_v(const void *x_bf16, const void *wkv_b_e4m3, const float *wkv_b_s, void *out_bf16,
                                   int64_t T, int64_t H, int64_t dn, int64_t dv, int64_t C, fp8blk_stream_t stream);

/*
 * MoE gate ("Administrator & Developer Guide", 8.4 the Gate and 3.3 per-config
 * fields; "Repository overview" page, MoE data flow: scores, optional group
 * masking, top-k indices, the original scores, normalize, route_scale).
 * Per token t, from the gate logits l[t, :] (fp32 [T, E]):
 *     s[e] = 1 / (1 + exp(-l[e]))   (FP8BLK_SCORE_SIGMOID), or
 *            softmax of l[t, :] over the E experts (FP8BLK_SCORE_SOFTMAX),
 *     z[e] = s[e] + bias[e]   (bias fp32 [E], optional: NULL means z = s),
 *     with n_groups > 1 groups of E / n_groups consecutive experts, a group
 *     scores its largest z (no bias) or the sum of its two largest z (bias);
 *     only the topk_groups best groups' experts stay eligible,
 *     topk_idx[t, j] = the eligible expert with the j-th largest z (ties go to
 *                      the lower index: j = 0 is the largest),
 *     topk_w[t, j]   = s[topk_idx[t, j]] / (normalize ? sum over j of those s : 1)
 *                      * route_scale.
 * Scores and sums are fp32 (the exponential is CUDA's expf, within 2 ulp).
 * Outputs: topk_idx int32 [T, topk], topk_w fp32 [T, topk] (device), ready for
 * fp8blk_moe_permute / fp8blk_moe_grouped_gemm. Shapes: E % 32 == 0 and
 * 32 <= E <= 256; n_groups divides 32 (so 1, 2, 4, 8, 16 or 32);
 * 1 <= topk_groups <= n_groups; 1 <= topk <= min(32, topk_groups * E / n_groups);
 * with a bias and n_groups > 1, groups of at least two experts. Otherwise
 * FP8BLK_ERR_SHAPE; a score_func other than the two, or a non-finite
 * route_scale, gives FP8BLK_ERR_ARG. Pointers 4-byte aligned. No workspace.
 */
#define FP8BLK_SCORE_SOFTMAX 0
#define FP8BLK_SCORE_SIGMOID 1
FP8BLK_API int fp8blk_moe_gate(const float *logits, const float *bias, int64_t T, int64_t E, int64_t n_groups,
                               int64_t topk_groups, int64_t topk, int score_func, float route_scale, int normalize,
                               int32_t *topk_idx, float *topk_w, fp8blk_stream_t stream);

/*
 * Gate and routing permutation together ("Administrator & Developer Guide",
 * 8.4: the Gate, then steps 2-5 group the (token, slot) pairs by expert):
 * topk_idx and topk_w exactly as fp8blk_moe_gate computes them, and counts,
 * offsets and perm exactly as fp8blk_moe_permute would compute them from
 * that topk_idx (counts[e] pairs per expert, offsets the exclusive prefix sum
 * with offsets[E] = T * topk, perm the pairs t * topk + j in increasing order
 * within each expert). Two launches: the gate kernel also ranks each pair
 * among its chunk's pairs of the same expert and writes the chunk's
 * histogram, its last CTA to finish turns the histograms into bases, counts
 * and offsets; one scatter pass writes perm. Same shape rules and errors as
 * fp8blk_moe_gate; counts int32 [E], offsets int32 [E + 1], perm int32
 * [T * topk], 4-byte aligned. T == 0 zeroes counts and offsets.
 * Workspace: fp8blk_moe_route_workspace_bytes(T, topk, E), 256-byte aligned;
 * its first 256 bytes hold an arrival counter: ZERO-FILLED before the first
 * use, and every call leaves it at zero. One workspace serves one stream at a
 * time.
 */
FP8BLK_API size_t fp8blk_moe_route_workspace_bytes(int64_t T, int64_t topk, int64_t E);
FP8BLK_API int fp8blk_moe_route(const float *logits, const float *bias, int64_t T, int64_t E, int64_t n_groups,
                                int64_t topk_groups, int64_t topk, int score_func, float route_scale, int normalize,
                                int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *offsets, int32_t *perm,
                                void *workspace, size_t workspace_bytes, fp8blk_stream_t stream);

/*
 * Routed-expert FFN ("Administrator & Developer Guide", 6.4 and 8.4 steps
 * 2-5): y[t] = bf16( sum over slots j (in order) of
 *                    topk_w[t, j] * bf16(FFN_{topk_idx[t, j]}(x[t])) ),
 * FFN_e(x) = w2_e(act_quant(bf16(silu(bf16(w1_e x))) * bf16(w3_e x))) with the
 * rounding of fp8blk_swiglu_gemm, accumulation of the sum in fp32.
 * Shared experts (8.4 steps 6 and 8: the shared MLP runs on every token and
 * the layer returns y + z): with n_shared > 0 the stacked weights hold the E
 * routed experts followed by n_shared shared experts of the same shape; every
 * token also goes through each of them with weight 1, and the row becomes
 *     bf16( y[t] + z[t] ),  z[t] = bf16( sum over shared s of bf16(FFN_{E+s}(x[t])) ),
 * in the same grouped launches as the routed rows. (A shared MLP of width
 * n * inter, as in the 16B and 236B configs, is the sum of n experts of width
 * inter up to the rounding of that sum.)
 * x: e4m3 [T, dim] + x_s [T, dim/128] (x quantised once per token: act_quant
 * is per row, so it commutes with routing). topk_idx int32 / topk_w fp32
 * [T, topk], routed ids in [0, E). Stacked expert weights (K = E + n_shared):
 * w1, w3 e4m3 [K*inter, dim] with scales [K*inter/128, dim/128]; w2 e4m3
 * [K*dim, inter] with scales [K*dim/128, inter/128]. y: bf16 [T, dim].
 * dim % 256 == 0, inter % 128 == 0, E + n_shared <= 1024.
 * Experts that receive no token read none of their weights.
 * Workspace: fp8blk_moe_workspace_bytes(T, topk, E, dim, inter, n_shared), 256-aligned.
 */
FP8BLK_API size_t fp8blk_moe_workspace_bytes(int64_t T, int64_t topk, int64_t E, int64_t dim, int64_t inter,
                                             int64_t n_shared);
FP8BLK_API int fp8blk_moe_grouped_gemm(const void *x_e4m3, const float *x_s, const int32_t *topk_idx,
                                       const float *topk_w, const void *w1_e4m3, const float *w1_s,
                                       const void *w3_e4m3, const float *w3_s, const void *w2_e4m3,
                                       const float *w2_s, void *y_bf16, int64_t T, int64_t topk, int64_t E,
                                       int64_t dim, int64_t inter, int64_t n_shared, int scale_fmt, void *workspace,
                                       size_t workspace_bytes, fp8blk_stream_t stream);

/*
 * fp8_gemm with no workspace argument and no device allocation: the same
 * computation, result and argument rules as fp8blk_gemm, but its scratch
 * (tile counters and stream-K partial sums) lives in a buffer of
 * FP8BLK_NOALLOC_SCRATCH_BYTES that the library itself holds in device memory,
 * on every GPU that loads the library, until the process exits.
 * The pages have no counterpart to this entry point: it exists for callers
 * that cannot allocate device memory themselves -- a plugin or custom layer
 * inside a serving engine that plans all device memory up front and forbids
 * allocation while it executes, a latency-critical loop that must never
 * reach cudaMalloc/cudaFree (cudaFree synchronises the device), or a caller
 * that is handed device pointers but has no allocator of its own.
 * - Arguments are checked first, exactly as fp8blk_gemm checks them (same
 *   statuses, same order); a call that fails them touches nothing.
 * - Size limit: then, problems whose scratch need (fp8blk_gemm_workspace_bytes)
 *   exceeds FP8BLK_NOALLOC_SCRATCH_BYTES return FP8BLK_ERR_TOO_LARGE and
 *   launch nothing. On a 152-SM GB300 every M <= 32 fits, for any N and K.
 * - The first call on a device looks up the buffer's device address; make that
 *   first call before any stream capture begins.
 * - Every call clears the tile counters in the buffer before its GEMM (a
 *   memset on `stream`) and allocates nothing.
 * - All calls on a device share the one buffer: calls that can overlap on the
 *   GPU (unordered streams) race and corrupt each other's results. Order them
 *   on one stream, or use fp8blk_gemm with a workspace per stream.
 */
#define FP8BLK_NOALLOC_SCRATCH_BYTES (8u << 20)
FP8BLK_API int fp8blk_gemm_noalloc(const void *a_e4m3, const float *a_s, const void *w_e4m3, const float *w_s,
                                   void *c_bf16, int64_t M, int64_t N, int64_t K, int scale_fmt,
                                   fp8blk_stream_t stream);

/*
 * Debug: synchronises `stream`, then returns and clears the device error
 * word of the current device (0 when no kernel reported a problem). Bits
 * 0x01-0x08: a GEMM role gave up waiting (producer, MMA, epilogue, drain);
 * 0x20: an expert id outside [0, E) (MoE); 0x40: an MLA kernel gave up
 * waiting; 0x80: a UE8M0-format scale that is not a positive normal power of
 * two. After a wait gave up, that kernel returned early: its outputs are
 * undefined and the workspace's first 64 KB must be zero-filled again before
 * reuse. The function returns FP8BLK_ERR_TIMEOUT when any bit is set.
 */
FP8BLK_API int fp8blk_last_device_error(fp8blk_stream_t stream, unsigned *device_error_bits);

#ifdef __cplusplus
}
#endif

#endif /* FP8BLK_H */
