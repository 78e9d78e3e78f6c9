// Exhaustive check of the library's block quotient (fp8blk::div_by_scale,
// csrc/quotient.cuh) against CUDA's IEEE division: for every positive finite
// bf16 amax, the act_quant scale s (fp32: RN(max(amax, 1e-4) / 448); ue8m0:
// that rounded up to a power of two) and every finite bf16 x with |x| <= amax,
// the e4m3 codes of div_by_scale(x, s, RN(1/s)) and RN(x / s) must agree, and
// the packed div2_by_scale must give div_by_scale's bits in both lanes.
// Prints one line per format and exits non-zero on any difference.
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdio>

#include "quotient.cuh"

__device__ float act_scale(uint32_t amax_bits, bool ue8m0) {
  float s = __fdiv_rn(fmaxf(__uint_as_float(amax_bits << 16), 1e-4f), 448.0f);
  if (ue8m0) {
    uint32_t b = __float_as_uint(s);
    if (b & 0x007FFFFFu) b = (b & 0x7F800000u) + 0x00800000u;
    s = __uint_as_float(b);
  }
  return s;
}

__global__ void check(bool ue8m0, unsigned long long* counts) {
  const uint32_t amax_bits = blockIdx.x;  // 0x0000 .. 0x7F7F: +0 .. the largest finite bf16
  const float s = act_scale(amax_bits, ue8m0);
  const float r = __frcp_rn(s);
  unsigned long long n = 0, bad = 0;
  for (uint32_t xb = threadIdx.x; xb < 65536u; xb += blockDim.x) {
    if ((xb & 0x7FFFu) > amax_bits) continue;  // |x| <= amax (this also excludes inf and nan)
    const float x = __uint_as_float(xb << 16);
    const float q = fp8blk::div_by_scale(x, s, r);
    const float2 q2 = fp8blk::div2_by_scale(make_float2(x, -x), make_float2(-s, -s), make_float2(r, r));
    const auto got = __nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
    const auto want = __nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E4M3);
    const float qn = fp8blk::div_by_scale(-x, s, r);
    ++n;
    // the packed form must give the scalar form's bits in both lanes
    bad += (got != want) || (__float_as_uint(q2.x) != __float_as_uint(q)) ||
           (__float_as_uint(q2.y) != __float_as_uint(qn));
  }
  atomicAdd(counts, n);
  atomicAdd(counts + 1, bad);
}

int main() {
  unsigned long long* d;
  if (cudaMalloc(&d, 16) != cudaSuccess) return 2;
  int rc = 0;
  for (int f = 0; f < 2; ++f) {
    unsigned long long h[2] = {0, 0};
    cudaMemset(d, 0, 16);
    check<<<0x7F80, 256>>>(f == 1, d);
    if (cudaMemcpy(h, d, 16, cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
    std::printf("%s pairs %llu mismatches %llu\n", f ? "ue8m0" : "fp32", h[0], h[1]);
    if (h[1] != 0 || h[0] == 0) rc = 1;
  }
  return rc;
}
