// Division of a block's values by the block's scale, as the act_quant rule
// needs it: the IEEE fp32 quotient x / s, rounded to nearest, then encoded to
// e4m3.
//
// Every element of a 128-element block is divided by the same s, so the
// reciprocal r = RN(1/s) is formed once per block and each quotient costs a
// multiply and two FMAs: Markstein's correction (P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): q0 = RN(x r), e = x - q0 s (exact by FMA), q = RN(q0 + e r).
// The sign of q is taken from q0, so that -0 stays -0.
//
// Exactness: q equals RN(x / s) except where x is tiny enough for e to
// underflow or where the quotient is an fp32 denormal; in both cases the
// quotient is far below the smallest e4m3 code, so the e4m3 code is the same.
// An exhaustive GPU comparison of the e4m3 codes against the IEEE division
// over every finite bf16 x with |x| <= amax and every scale s the act_quant
// rule derives from a bf16 amax (fp32 and ue8m0 formats) finds no difference
// (tests/test_gpu_quotient.py). It therefore serves inputs that are bf16
// values quantised against their own block's amax: act_quant, the SwiGLU
// output u, the decode GEMM's in-kernel act_quant. Weight quantisation (fp32
// inputs) keeps the IEEE division.
#pragma once

namespace fp8blk {

// r: __frcp_rn(s) (the correctly rounded reciprocal, computed once per block).
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float q = __fmaf_rn(__fmaf_rn(-q0, s, x), r, q0);
  return __uint_as_float(__float_as_uint(q) | (__float_as_uint(q0) & 0x80000000u));
}

// The same for two values at once (packed f32x2 multiply and FMAs: per
// component the identical operations and roundings). sn2 = (-s, -s),
// r2 = (r, r).
__device__ __forceinline__ float2 div2_by_scale(float2 x, float2 sn2, float2 r2) {
  const float2 q0 = __fmul2_rn(x, r2);
  const float2 q = __ffma2_rn(__ffma2_rn(q0, sn2, x), r2, q0);
  return make_float2(__uint_as_float(__float_as_uint(q.x) | (__float_as_uint(q0.x) & 0x80000000u)),
                     __uint_as_float(__float_as_uint(q.y) | (__float_as_uint(q0.y) & 0x80000000u)));
}

}  // namespace fp8blk
