// Elementwise kernels of the block-scaled FP8 path:
//   act_quant       -- "Administrator & Developer Guide", 8.5.1
//   weight_quant    -- README ("Algolia docsearch" page) section 3: 128x128
//                      block scales, non-aligned edges padded with zeros
//   weight_dequant  -- "Administrator & Developer Guide", 8.5.2
// All three are bound by HBM bandwidth: 128-bit loads and stores, grids sized
// in multiples of the SM count, no shared-memory staging needed (each thread
// owns whole 16-byte vectors and each 128-element block lives in 16 lanes).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8blk.h"
#include "host.cuh"
#include "ptx.cuh"
#include "quotient.cuh"

namespace fp8blk {
namespace {

// Scale of a 128-element (or 128x128) block: max(amax, 1e-4) / 448 as an IEEE
// fp32 division; with ue8m0, rounded up to a power of two on the bits
// (2^ceil(log2 s) exactly: unchanged when the mantissa is zero, otherwise the
// next power of two above).
__device__ __forceinline__ float block_scale(float amax, bool ue8m0) {
  float s = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
  if (ue8m0) {
    uint32_t b = __float_as_uint(s);
    if (b & 0x007FFFFFu) b = (b & 0x7F800000u) + 0x00800000u;
    s = __uint_as_float(b);
  }
  return s;
}

// Two fp32 values -> two e4m3 codes (round to nearest even, saturating), low
// byte = a.
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t w) {
  __nv_bfloat162 b;
  *reinterpret_cast<uint32_t*>(&b) = w;
  return b;
}
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---- act_quant -------------------------------------------------------------
// A 128-element block is 256 bytes of bf16: 16 lanes x 16 bytes, so a warp
// holds a pair of blocks (half-warp h takes block 2p + h of pair p). Blocks
// are contiguous in memory because K % 128 == 0: block b starts at element
// b * 128 whatever its row. Each warp takes kAqUnroll pairs per pass so that
// several 16-byte loads are in flight per thread. Loop bounds are uniform over
// the warp (the shuffles use the full mask); lanes past the end compute on
// zeros and store nothing.
constexpr int kAqThreads = 256;
#ifndef FP8BLK_AQ_UNROLL
#define FP8BLK_AQ_UNROLL 4
#endif
constexpr int kAqUnroll = FP8BLK_AQ_UNROLL;

__global__ void __launch_bounds__(kAqThreads) act_quant_kernel(const uint4* __restrict__ x, uint2* __restrict__ q,
                                                               float* __restrict__ s, int64_t nblocks,
                                                               bool ue8m0, bool trigger) {
  // Launched programmatically, this kernel may start before the previous one
  // on the stream ends: x is read only after that kernel has completed. The
  // next kernel (the GEMM that reads q and s only after its own dependency
  // wait, which follows this kernel's completion and so the previous one's)
  // may launch at once and start streaming its weights meanwhile.
  if (trigger) griddep_launch_dependents();
  griddep_wait();
  const int sub = threadIdx.x & 15;
  const int half = (threadIdx.x >> 4) & 1;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kAqThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kAqThreads) >> 5;
  const int64_t npairs = (nblocks + 1) >> 1;
  for (int64_t p0 = warp; p0 < npairs; p0 += nwarps * kAqUnroll) {
    uint4 v[kAqUnroll];
    int64_t blk[kAqUnroll];
#pragma unroll
    for (int u = 0; u < kAqUnroll; ++u) {
      const int64_t p = p0 + u * nwarps;
      blk[u] = (p < npairs) ? 2 * p + half : nblocks;
      v[u] = (blk[u] < nblocks) ? __ldcs(x + blk[u] * 16 + sub) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kAqUnroll; ++u) {
      // amax on the bf16 pairs (|.| by clearing the sign bits; bf16 max is
      // exact), then across the 16 lanes of the block.
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      __nv_bfloat162 m = __hmax2(__hmax2(as_bf162(w[0] & 0x7FFF7FFFu), as_bf162(w[1] & 0x7FFF7FFFu)),
                                 __hmax2(as_bf162(w[2] & 0x7FFF7FFFu), as_bf162(w[3] & 0x7FFF7FFFu)));
      float amax = fmaxf(__low2float(m), __high2float(m));
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off, 16));
      const float sc = block_scale(amax, ue8m0);
      const float rc = __frcp_rn(sc);  // the block's quotients: see quotient.cuh
      const float2 sn2 = make_float2(-sc, -sc), r2 = make_float2(rc, rc);
      uint32_t c[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 qk = div2_by_scale(make_float2(bf16_lo(w[k]), bf16_hi(w[k])), sn2, r2);
        c[k] = e4m3x2(qk.x, qk.y);
      }
      const uint32_t lo = c[0] | (c[1] << 16);
      const uint32_t hi = c[2] | (c[3] << 16);
      if (blk[u] < nblocks) {
        q[blk[u] * 16 + sub] = make_uint2(lo, hi);
        if (sub == 0) s[blk[u]] = sc;
      }
    }
  }
}

// ---- weight_quant ------------------------------------------------------------
// One CTA per 128x128 block. Thread t covers columns (t % 32) * 4 .. + 3 of
// rows t / 32 + 8 j, j < 16: 64 values held in registers between the amax
// reduction and the quantisation.
constexpr int kWqThreads = 256;

__global__ void __launch_bounds__(kWqThreads) weight_quant_kernel(const float* __restrict__ w, uint8_t* __restrict__ q,
                                                                  float* __restrict__ s, int64_t N, int64_t K,
                                                                  int64_t nbk, bool ue8m0) {
  __shared__ float warp_max[kWqThreads / 32];
  const int64_t bn = blockIdx.y, bk = blockIdx.x;
  const int t = threadIdx.x;
  const int64_t col0 = bk * kBlock + (t & 31) * 4;
  const int64_t row0 = bn * kBlock + (t >> 5);
  float v[16][4];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int64_t r = row0 + 8 * j;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t c = col0 + i;
      v[j][i] = (r < N && c < K) ? w[r * K + c] : 0.0f;
      amax = fmaxf(amax, fabsf(v[j][i]));
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  if ((t & 31) == 0) warp_max[t >> 5] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int i = 1; i < kWqThreads / 32; ++i) amax = fmaxf(amax, warp_max[i]);
  const float sc = block_scale(amax, ue8m0);
  if (t == 0) s[bn * nbk + bk] = sc;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int64_t r = row0 + 8 * j;
    if (r >= N) break;
    const uint16_t p01 = e4m3x2(__fdiv_rn(v[j][0], sc), __fdiv_rn(v[j][1], sc));
    const uint16_t p23 = e4m3x2(__fdiv_rn(v[j][2], sc), __fdiv_rn(v[j][3], sc));
    const uint8_t b[4] = {static_cast<uint8_t>(p01 & 0xFF), static_cast<uint8_t>(p01 >> 8),
                          static_cast<uint8_t>(p23 & 0xFF), static_cast<uint8_t>(p23 >> 8)};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (col0 + i < K) q[r * K + col0 + i] = b[i];
  }
}

// ---- weight_dequant ------------------------------------------------------------
// e4m3 -> f16 is exact (every e4m3 value is an f16 value) and f16 -> f32 is
// exact, so fp32(q) is obtained without rounding; then one fp32 multiply and
// one round-to-nearest-even to bf16.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ uint32_t dequant_pair(uint16_t two, float sc) {
  const float2 f = e4m3x2_to_float2(two);
  const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, sc), __fmul_rn(f.y, sc));
  return *reinterpret_cast<const uint32_t*>(&b);
}

constexpr int kDqThreads = 256;

// Vector path: K % 16 == 0 and both buffers 16-byte aligned. Thread i handles
// the 16 consecutive elements of vector i (one 128-block column, so one
// scale); each pass issues kDqUnroll vector loads before any arithmetic so that
// several are in flight per thread.
#ifndef FP8BLK_DQ_UNROLL
#define FP8BLK_DQ_UNROLL 1
#endif
constexpr int kDqUnroll = FP8BLK_DQ_UNROLL;

template <typename Index>
__global__ void __launch_bounds__(kDqThreads) weight_dequant_vec_kernel(const uint4* __restrict__ q,
                                                                        const float* __restrict__ s,
                                                                        uint4* __restrict__ out, Index nvec,
                                                                        Index kvec, Index nbk) {
  const Index stride = static_cast<Index>(gridDim.x) * kDqThreads;
  for (Index i0 = static_cast<Index>(blockIdx.x) * kDqThreads + threadIdx.x; i0 < nvec; i0 += stride * kDqUnroll) {
    uint4 v[kDqUnroll];
    float sc[kDqUnroll];
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
      const Index i = i0 + u * stride;
      if (i < nvec) {
        const Index n = i / kvec;
        const Index kv = i - n * kvec;
        sc[u] = __ldg(s + (n / kBlock) * nbk + (kv >> 3));  // 8 vectors per 128 columns
        v[u] = __ldcs(q + i);
      }
    }
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
      const Index i = i0 + u * stride;
      if (i >= nvec) break;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o[2 * j] = dequant_pair(static_cast<uint16_t>(w[j] & 0xFFFF), sc[u]);
        o[2 * j + 1] = dequant_pair(static_cast<uint16_t>(w[j] >> 16), sc[u]);
      }
      __stcs(out + 2 * i, make_uint4(o[0], o[1], o[2], o[3]));
      __stcs(out + 2 * i + 1, make_uint4(o[4], o[5], o[6], o[7]));
    }
  }
}

// Scalar path for any shape and alignment: one element per thread.
__global__ void __launch_bounds__(kDqThreads) weight_dequant_scalar_kernel(const uint8_t* __restrict__ q,
                                                                           const float* __restrict__ s,
                                                                           __nv_bfloat16* __restrict__ out,
                                                                           int64_t total, int64_t K, int64_t nbk) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kDqThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kDqThreads + threadIdx.x; i < total; i += stride) {
    const int64_t n = i / K, k = i - n * K;
    const float sc = s[(n / kBlock) * nbk + k / kBlock];
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(q[i]), __NV_E4M3);
    const float f = __half2float(*reinterpret_cast<const __half*>(&h));
    out[i] = __float2bfloat16_rn(__fmul_rn(f, sc));
  }
}

int grid_for(const DevInfo* d, int64_t work_items, int threads, int per_sm) {
  const int64_t need = (work_items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(d->sm_count) * per_sm;
  return static_cast<int>(need < cap ? (need < 1 ? 1 : need) : cap);
}

// One thread per work item, as many CTAs as that takes (the grid-stride loops
// cover anything past 2^30 CTAs). For the dequant stream this beats a grid
// capped at a few CTAs per SM: at any moment the resident CTAs work on one
// contiguous window of the matrix, and it measured 60 us against 79 us for a
// 18432 x 7168 weight (8 CTAs per SM, each striding over the whole matrix).
int grid_all(int64_t work_items, int threads) {
  const int64_t need = (work_items + threads - 1) / threads;
  const int64_t cap = int64_t{1} << 30;
  return static_cast<int>(need < 1 ? 1 : need < cap ? need : cap);
}

}  // namespace
}  // namespace fp8blk

using namespace fp8blk;

namespace fp8blk {

// act_quant launch; `trigger` lets the next kernel on the stream start early
// (used inside the linear / FFN entry points, whose next kernel is a GEMM that
// reads only its weights before it waits for this one).
int act_quant_launch(const void* x_bf16, int64_t M, int64_t K, void* q_e4m3, float* s, int scale_fmt,
                     cudaStream_t stream, bool trigger) {
  if (!scale_fmt_valid(scale_fmt)) return FP8BLK_ERR_ARG;
  if (M < 0 || K < 0 || K % kBlock != 0) return FP8BLK_ERR_SHAPE;
  if (M == 0 || K == 0) return FP8BLK_OK;
  if (!x_bf16 || !q_e4m3 || !s) return FP8BLK_ERR_NULL;
  if (!is_aligned(x_bf16, 16) || !is_aligned(q_e4m3, 16) || !is_aligned(s, 4)) return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  const int64_t nblocks = M * (K / kBlock);
  // A warp per pair of blocks, kAqUnroll pairs per pass, up to 8 CTAs per SM.
  const int grid = grid_for(d, (nblocks + 1) / 2 * 32 / kAqUnroll, kAqThreads, 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kAqThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, act_quant_kernel, static_cast<const uint4*>(x_bf16),
                                        static_cast<uint2*>(q_e4m3), s, nblocks, scale_fmt_ue8m0(scale_fmt),
                                        trigger));
}

}  // namespace fp8blk

extern "C" int fp8blk_act_quant(const void* x_bf16, int64_t M, int64_t K, void* q_e4m3, float* s, int scale_fmt,
                                fp8blk_stream_t stream) {
  return act_quant_launch(x_bf16, M, K, q_e4m3, s, scale_fmt, reinterpret_cast<cudaStream_t>(stream), false);
}

extern "C" int fp8blk_weight_quant(const float* w, int64_t N, int64_t K, void* q_e4m3, float* s, int scale_fmt,
                                   fp8blk_stream_t stream) {
  if (!scale_fmt_valid(scale_fmt)) return FP8BLK_ERR_ARG;
  if (N < 0 || K < 0) return FP8BLK_ERR_SHAPE;
  if (N == 0 || K == 0) return FP8BLK_OK;
  if (!w || !q_e4m3 || !s) return FP8BLK_ERR_NULL;
  if (!is_aligned(w, 4) || !is_aligned(s, 4)) return FP8BLK_ERR_ALIGN;
  const int64_t nbn = (N + kBlock - 1) / kBlock, nbk = (K + kBlock - 1) / kBlock;
  if (nbn > 65535 || nbk > 2147483647LL) return FP8BLK_ERR_SHAPE;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  dim3 grid(static_cast<unsigned>(nbk), static_cast<unsigned>(nbn));
  weight_quant_kernel<<<grid, kWqThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      w, static_cast<uint8_t*>(q_e4m3), s, N, K, nbk, scale_fmt_ue8m0(scale_fmt));
  return launch_status();
}

extern "C" int fp8blk_weight_dequant(const void* q_e4m3, const float* s, int64_t N, int64_t K, void* out_bf16,
                                     fp8blk_stream_t stream) {
  if (N < 0 || K < 0) return FP8BLK_ERR_SHAPE;
  if (N == 0 || K == 0) return FP8BLK_OK;
  if (!q_e4m3 || !s || !out_bf16) return FP8BLK_ERR_NULL;
  if (!is_aligned(s, 4) || !is_aligned(out_bf16, 2)) return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int64_t nbk = (K + kBlock - 1) / kBlock;
  if (K % 16 == 0 && is_aligned(q_e4m3, 16) && is_aligned(out_bf16, 16)) {
    const int64_t kvec = K / 16, nvec = N * kvec;
    const int grid = grid_all(nvec, kDqThreads);
    if (nvec < (int64_t{1} << 31)) {
      weight_dequant_vec_kernel<uint32_t><<<grid, kDqThreads, 0, cs>>>(
          static_cast<const uint4*>(q_e4m3), s, static_cast<uint4*>(out_bf16), static_cast<uint32_t>(nvec),
          static_cast<uint32_t>(kvec), static_cast<uint32_t>(nbk));
    } else {
      weight_dequant_vec_kernel<uint64_t><<<grid, kDqThreads, 0, cs>>>(
          static_cast<const uint4*>(q_e4m3), s, static_cast<uint4*>(out_bf16), static_cast<uint64_t>(nvec),
          static_cast<uint64_t>(kvec), static_cast<uint64_t>(nbk));
    }
  } else {
    const int64_t total = N * K;
    const int grid = grid_all(total, kDqThreads);
    weight_dequant_scalar_kernel<<<grid, kDqThreads, 0, cs>>>(static_cast<const uint8_t*>(q_e4m3), s,
                                                              static_cast<__nv_bfloat16*>(out_bf16), total, K, nbk);
  }
  return launch_status();
}
