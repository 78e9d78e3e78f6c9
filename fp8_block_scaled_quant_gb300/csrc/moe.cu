// Routed-expert FFN over block-scaled FP8 ("Administrator & Developer
// Guide", 6.4 MoE expert routing and 8.4 steps 2-5): for every expert e, the
// tokens routed to it go through w2(silu(w1 x) * w3 x) and the results are
// summed per token with the gate weights. The pages' loop (a host-side
// bincount + tolist(), then one Python iteration per expert) becomes:
//
//   moe_permute   one CTA: histogram of expert ids, exclusive scans (row
//                 offsets and 128-row tile counts per expert), and a stable
//                 scatter of the (token, slot) pairs into expert order;
//   moe_gather    the quantised token rows (and their scales) in that order;
//   grouped w1/w3 GEMM with the SwiGLU + act_quant epilogue (gemm.cu);
//   grouped w2 GEMM, each row written back to its (token, slot) position;
//   moe_combine   y[t] = bf16(sum_j w[t, j] * o[t, j]) in slot order.
//
// No host synchronisation: tile counts are read by the GEMMs on the device.
// The dense FFN (the "MLP" module of the guide's 1.2) is the same chain
// without routing: act_quant, the fused w1/w3 GEMM, and the w2 GEMM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8blk.h"
#include "host.cuh"
#include "ptx.cuh"

namespace fp8blk {

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
int act_quant_launch(const void* x_bf16, int64_t M, int64_t K, void* q_e4m3, float* s, int scale_fmt,
                     cudaStream_t stream, bool trigger);
int gemm_run(const void* a, const float* a_s, const void* w, const float* w_s, void* c, int64_t M, int64_t N,
             int64_t K, int scale_fmt, void* workspace, size_t workspace_bytes, cudaStream_t stream);
size_t swiglu_workspace_bytes(int64_t M, int64_t inter, int64_t K);
int swiglu_run(const void* xq, const float* xs, const void* w1, const float* w1s, const void* w3, const float* w3s,
               void* uq, float* us, int64_t M, int64_t inter, int64_t K, int scale_fmt, void* workspace,
               size_t workspace_bytes, cudaStream_t stream);
int grouped_swiglu_run(const void* xg, const float* xgs, const void* w1, const float* w1s, const void* w3,
                       const float* w3s, void* uq, float* us, int64_t rows, int64_t E, int64_t inter, int64_t K,
                       const int* grp_rows, const int* grp_mtiles, int scale_fmt, cudaStream_t stream);
int grouped_scatter_run(const void* uq, const float* us, const void* w2, const float* w2s, void* out,
                        const int* perm, int64_t rows, int64_t E, int64_t dim, int64_t inter, const int* grp_rows,
                        const int* grp_mtiles, cudaStream_t stream);

namespace {

constexpr int kMaxExperts = 1024;
constexpr int kPermThreads = 1024;
constexpr unsigned kDevErrBadExpert = 1u << 5;

// Exclusive scan of one value per thread over the 1024-thread block; returns
// the thread's prefix, *total gets the sum. `wsum` is 32 ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
      if (lane >= off) wi += o;
    }
    wsum[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) wsum[32] = wi;
  }
  __syncthreads();
  const int r = wsum[warp] + incl - v;
  *total = wsum[32];
  __syncthreads();
  return r;
}

// One CTA groups the n (token, slot) pairs by expert, keeping pair order
// (t * topk + j) inside each expert: counts, offsets[E + 1] (exclusive scan),
// mtiles[E + 1] (exclusive scan of ceil(count / 128)), and perm[offsets[e] + r]
// = the r-th pair of expert e. Pairs whose expert id is outside [0, E) join
// no expert and set an error bit.
__global__ void __launch_bounds__(kPermThreads) moe_permute_kernel(const int* __restrict__ idx, int n, int E,
                                                                   int* __restrict__ counts,
                                                                   int* __restrict__ offsets,
                                                                   int* __restrict__ mtiles,
                                                                   int* __restrict__ perm, unsigned* err) {
  extern __shared__ int sm[];
  int* cnt = sm;              // [E]
  int* base = cnt + E;        // [E] running output position per expert
  int* wsum = base + E;       // [40] scan scratch
  int* wtab = wsum + 40;      // [32][E] per-warp counts of the current chunk
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int e = tid; e < E; e += kPermThreads) cnt[e] = 0;
  __syncthreads();
  bool bad = false;
  for (int i = tid; i < n; i += kPermThreads) {
    const int e = __ldg(idx + i);
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else bad = true;
  }
  if (bad) atomicOr(err, kDevErrBadExpert);
  __syncthreads();

  const int c = tid < E ? cnt[tid] : 0;
  int total_rows, total_tiles;
  const int off = block_exclusive_scan(c, wsum, &total_rows);
  const int mt = block_exclusive_scan((c + 127) / 128, wsum, &total_tiles);
  if (tid < E) {
    if (counts) counts[tid] = c;
    offsets[tid] = off;
    if (mtiles) mtiles[tid] = mt;
    base[tid] = off;
  }
  if (tid == 0) {
    offsets[E] = total_rows;
    if (mtiles) mtiles[E] = total_tiles;
  }
  __syncthreads();

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < n; c0 += kPermThreads) {
    for (int k = tid; k < 32 * E; k += kPermThreads) wtab[k] = 0;
    __syncthreads();
    const int i = c0 + tid;
    int e = i < n ? __ldg(idx + i) : -1;
    if (e < 0 || e >= E) e = -1;
    const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
    const int wrank = __popc(m & lt_mask);
    if (e >= 0 && wrank == 0) wtab[warp * E + e] = __popc(m);
    __syncthreads();
    if (e >= 0) {
      int pre = 0;
      for (int w = 0; w < warp; ++w) pre += wtab[w * E + e];
      perm[base[e] + pre + wrank] = i;
    }
    __syncthreads();
    for (int x = tid; x < E; x += kPermThreads) {
      int s = 0;
      for (int w = 0; w < 32; ++w) s += wtab[w * E + x];
      base[x] += s;
    }
    __syncthreads();
  }
}

// xg[r] = xq[perm[r] / topk] and its scales, for r < offsets[E] (one warp per row).
__global__ void __launch_bounds__(256) moe_gather_kernel(const uint4* __restrict__ xq, const float* __restrict__ xs,
                                                         const int* __restrict__ perm,
                                                         const int* __restrict__ offsets, int E, int topk, int dim,
                                                         uint4* __restrict__ xg, float* __restrict__ xgs) {
  const int n = __ldg(offsets + E);
  const int dv = dim / 16, kb = dim / 128;
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; r < n; r += nwarps) {
    const long long t = __ldg(perm + r) / topk;
    const uint4* src = xq + t * dv;
    uint4* dst = xg + r * dv;
#pragma unroll 4
    for (int v = lane; v < dv; v += 32) dst[v] = __ldg(src + v);
    for (int k = lane; k < kb; k += 32) xgs[r * kb + k] = __ldg(xs + t * kb + k);
  }
}

// y[t, :] = bf16( sum over slots j in order of w[t, j] * o[t * topk + j, :] ),
// fp32 accumulation; slots routed to no valid expert contribute nothing.
// y[t] = bf16(sum over slots j in order of w[t, j] * o[t * topk + j]) in fp32.
// For topk <= kCombineMax all slots' ids, weights and output vectors are
// requested before the first FMA (the loads are independent; the FMAs keep the
// slot order); larger topk takes the plain loop.
constexpr int kCombineMax = 8;

__global__ void __launch_bounds__(256) moe_combine_kernel(const uint4* __restrict__ o, const int* __restrict__ idx,
                                                          const float* __restrict__ w, int T, int topk, int E,
                                                          int dim, uint4* __restrict__ y) {
  const int dv = dim / 8;
  const long long total = static_cast<long long>(T) * dv;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += stride) {
    const long long t = v / dv;
    const int c = static_cast<int>(v - t * dv);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    auto add = [&](float wj, const uint4& ov) {
      const uint32_t u[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] = fmaf(wj, __uint_as_float(u[q] << 16), acc[2 * q]);
        acc[2 * q + 1] = fmaf(wj, __uint_as_float(u[q] & 0xFFFF0000u), acc[2 * q + 1]);
      }
    };
    if (topk <= kCombineMax) {
      int e[kCombineMax];
      float wj[kCombineMax];
      uint4 ov[kCombineMax];
#pragma unroll
      for (int j = 0; j < kCombineMax; ++j) {
        e[j] = j < topk ? __ldg(idx + t * topk + j) : -1;
        wj[j] = j < topk ? __ldg(w + t * topk + j) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kCombineMax; ++j)
        if (e[j] >= 0 && e[j] < E) ov[j] = __ldg(o + (t * topk + j) * dv + c);
#pragma unroll
      for (int j = 0; j < kCombineMax; ++j)
        if (e[j] >= 0 && e[j] < E) add(wj[j], ov[j]);
    } else {
      for (int j = 0; j < topk; ++j) {
        const int ej = __ldg(idx + t * topk + j);
        if (ej < 0 || ej >= E) continue;
        add(__ldg(w + t * topk + j), __ldg(o + (t * topk + j) * dv + c));
      }
    }
    uint32_t r[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      r[q] = *reinterpret_cast<const uint32_t*>(&b);
    }
    y[v] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

size_t align256(size_t v) { return (v + 255) & ~size_t{255}; }

size_t permute_smem_bytes(int64_t E) { return static_cast<size_t>(2 * E + 40 + 32 * E) * sizeof(int); }

int launch_permute(const DevInfo* d, const int* idx, int64_t n, int64_t E, int* counts, int* offsets, int* mtiles,
                   int* perm, cudaStream_t stream) {
  static bool attr_done[64] = {};
  const size_t smem = permute_smem_bytes(kMaxExperts);
  if (d->device >= 64 || !attr_done[d->device]) {
    if (cudaFuncSetAttribute(moe_permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return FP8BLK_ERR_CUDA;
    if (d->device < 64) attr_done[d->device] = true;
  }
  moe_permute_kernel<<<1, kPermThreads, permute_smem_bytes(E), stream>>>(
      idx, static_cast<int>(n), static_cast<int>(E), counts, offsets, mtiles, perm, d->err_word);
  return launch_status();
}

}  // namespace
}  // namespace fp8blk

using namespace fp8blk;

extern "C" int fp8blk_moe_permute(const int32_t* topk_idx, int64_t T, int64_t topk, int64_t E, int32_t* counts,
                                  int32_t* offsets, int32_t* perm, fp8blk_stream_t stream) {
  if (T < 0 || topk < 0 || E <= 0 || E > kMaxExperts || T * topk > (int64_t{1} << 31) - 1) return FP8BLK_ERR_SHAPE;
  if (!counts || !offsets) return FP8BLK_ERR_NULL;
  if (T * topk > 0 && (!topk_idx || !perm)) return FP8BLK_ERR_NULL;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  return launch_permute(d, topk_idx, T * topk, E, counts, offsets, nullptr, perm,
                        reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t fp8blk_swiglu_workspace_bytes(int64_t M, int64_t inter, int64_t dim) {
  return swiglu_workspace_bytes(M, inter, dim);
}

extern "C" int fp8blk_swiglu_gemm(const void* x_e4m3, const float* x_s, const void* w1_e4m3, const float* w1_s,
                                  const void* w3_e4m3, const float* w3_s, void* u_e4m3, float* u_s, int64_t M,
                                  int64_t inter, int64_t dim, int scale_fmt, void* workspace, size_t workspace_bytes,
                                  fp8blk_stream_t stream) {
  return swiglu_run(x_e4m3, x_s, w1_e4m3, w1_s, w3_e4m3, w3_s, u_e4m3, u_s, M, inter, dim, scale_fmt, workspace,
                    workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

// FFN workspace: [x_q M*dim][x_s M*dim/128][u_q M*inter][u_s M*inter/128]
// [w1/w3 GEMM workspace][w2 GEMM workspace]. The two GEMM workspaces are
// separate: each keeps its tile counters at zero between calls, and neither
// may write partial sums where the other keeps its counters.
extern "C" size_t fp8blk_ffn_workspace_bytes(int64_t M, int64_t dim, int64_t inter) {
  if (M < 0 || dim < 0 || inter < 0) return 0;
  return align256(static_cast<size_t>(M) * dim) + align256(static_cast<size_t>(M) * (dim / kBlock) * 4) +
         align256(static_cast<size_t>(M) * inter) + align256(static_cast<size_t>(M) * (inter / kBlock) * 4) +
         align256(swiglu_workspace_bytes(M, inter, dim)) + gemm_workspace_bytes(M, dim, inter);
}

extern "C" int fp8blk_ffn(const void* x_bf16, const void* w1_e4m3, const float* w1_s, const void* w3_e4m3,
                          const float* w3_s, const void* w2_e4m3, const float* w2_s, void* y_bf16, int64_t M,
                          int64_t dim, int64_t inter, int scale_fmt, void* workspace, size_t workspace_bytes,
                          fp8blk_stream_t stream) {
  if (M < 0 || dim <= 0 || inter <= 0 || dim % kBlock || inter % kBlock) return FP8BLK_ERR_SHAPE;
  if (M == 0) return FP8BLK_OK;
  if (!workspace) return FP8BLK_ERR_WORKSPACE;
  if (!is_aligned(workspace, 256)) return FP8BLK_ERR_ALIGN;
  if (workspace_bytes < fp8blk_ffn_workspace_bytes(M, dim, inter)) return FP8BLK_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* p = static_cast<uint8_t*>(workspace);
  uint8_t* xq = p;
  p += align256(static_cast<size_t>(M) * dim);
  float* xs = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(M) * (dim / kBlock) * 4);
  uint8_t* uq = p;
  p += align256(static_cast<size_t>(M) * inter);
  float* us = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(M) * (inter / kBlock) * 4);
  const size_t g1 = align256(swiglu_workspace_bytes(M, inter, dim));
  uint8_t* g2p = p + g1;
  const size_t rest = workspace_bytes - (g2p - static_cast<uint8_t*>(workspace));
  if (int st = act_quant_launch(x_bf16, M, dim, xq, xs, scale_fmt, cs, true)) return st;
  if (int st = swiglu_run(xq, xs, w1_e4m3, w1_s, w3_e4m3, w3_s, uq, us, M, inter, dim, scale_fmt, p, g1, cs))
    return st;
  return gemm_run(uq, us, w2_e4m3, w2_s, y_bf16, M, dim, inter, scale_fmt, g2p, rest, cs);
}

namespace {

struct MoeLayout {
  size_t counts, offsets, mtiles, perm, xg, xgs, uq, us, o, total;
};

MoeLayout moe_layout(int64_t T, int64_t topk, int64_t E, int64_t dim, int64_t inter) {
  MoeLayout l{};
  const size_t n = static_cast<size_t>(T) * topk;
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  l.counts = take(E * 4);
  l.offsets = take((E + 1) * 4);
  l.mtiles = take((E + 1) * 4);
  l.perm = take(n * 4);
  l.xg = take(n * dim);
  l.xgs = take(n * (dim / kBlock) * 4);
  l.uq = take(n * inter);
  l.us = take(n * (inter / kBlock) * 4);
  l.o = take(n * dim * 2);
  l.total = off;
  return l;
}

}  // namespace

extern "C" size_t fp8blk_moe_workspace_bytes(int64_t T, int64_t topk, int64_t E, int64_t dim, int64_t inter) {
  if (T < 0 || topk < 0 || E <= 0 || dim < 0 || inter < 0) return 0;
  return moe_layout(T, topk, E, dim, inter).total;
}

extern "C" int fp8blk_moe_grouped_gemm(const void* x_e4m3, const float* x_s, const int32_t* topk_idx,
                                       const float* topk_w, const void* w1_e4m3, const float* w1_s,
                                       const void* w3_e4m3, const float* w3_s, const void* w2_e4m3,
                                       const float* w2_s, void* y_bf16, int64_t T, int64_t topk, int64_t E,
                                       int64_t dim, int64_t inter, int scale_fmt, void* workspace,
                                       size_t workspace_bytes, fp8blk_stream_t stream) {
  if (scale_fmt != FP8BLK_SCALE_FP32 && scale_fmt != FP8BLK_SCALE_UE8M0) return FP8BLK_ERR_ARG;
  if (T < 0 || topk < 0 || E <= 0 || E > kMaxExperts || dim <= 0 || inter <= 0 || dim % 256 || inter % kBlock)
    return FP8BLK_ERR_SHAPE;
  const int64_t n = T * topk;
  if (n > (int64_t{1} << 31) - 1 || E * inter > (int64_t{1} << 31) - 1 || E * dim > (int64_t{1} << 31) - 1)
    return FP8BLK_ERR_SHAPE;
  if (T == 0) return FP8BLK_OK;
  if (!y_bf16) return FP8BLK_ERR_NULL;
  if (topk == 0) return cuda_status(cudaMemsetAsync(y_bf16, 0, static_cast<size_t>(T) * dim * 2,
                                                    reinterpret_cast<cudaStream_t>(stream)));
  if (!x_e4m3 || !x_s || !topk_idx || !topk_w || !w1_e4m3 || !w1_s || !w3_e4m3 || !w3_s || !w2_e4m3 || !w2_s)
    return FP8BLK_ERR_NULL;
  if (!is_aligned(x_e4m3, 16) || !is_aligned(w1_e4m3, 16) || !is_aligned(w3_e4m3, 16) ||
      !is_aligned(w2_e4m3, 16) || !is_aligned(y_bf16, 16) || !is_aligned(x_s, 4) || !is_aligned(w1_s, 4) ||
      !is_aligned(w3_s, 4) || !is_aligned(w2_s, 4) || !is_aligned(topk_idx, 4) || !is_aligned(topk_w, 4))
    return FP8BLK_ERR_ALIGN;
  const MoeLayout l = moe_layout(T, topk, E, dim, inter);
  if (!workspace || workspace_bytes < l.total) return FP8BLK_ERR_WORKSPACE;
  if (!is_aligned(workspace, 256)) return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* counts = reinterpret_cast<int*>(ws + l.counts);
  int* offsets = reinterpret_cast<int*>(ws + l.offsets);
  int* mtiles = reinterpret_cast<int*>(ws + l.mtiles);
  int* perm = reinterpret_cast<int*>(ws + l.perm);
  uint8_t* xg = ws + l.xg;
  float* xgs = reinterpret_cast<float*>(ws + l.xgs);
  uint8_t* uq = ws + l.uq;
  float* us = reinterpret_cast<float*>(ws + l.us);
  void* o = ws + l.o;

  if (int st = launch_permute(d, topk_idx, n, E, counts, offsets, mtiles, perm, cs)) return st;
  // One warp per routed row (at most T * topk of them), as many CTAs as that
  // takes: the resident CTAs then copy one contiguous window of rows at a time.
  const long long gather_grid = (static_cast<long long>(n) + 7) / 8;
  moe_gather_kernel<<<static_cast<unsigned>(gather_grid < (1LL << 30) ? gather_grid : (1LL << 30)), 256, 0, cs>>>(static_cast<const uint4*>(x_e4m3), x_s, perm, offsets,
                                                 static_cast<int>(E), static_cast<int>(topk), static_cast<int>(dim),
                                                 reinterpret_cast<uint4*>(xg), xgs);
  if (int st = launch_status()) return st;
  if (int st = grouped_swiglu_run(xg, xgs, w1_e4m3, w1_s, w3_e4m3, w3_s, uq, us, n, E, inter, dim, offsets, mtiles,
                                  scale_fmt, cs))
    return st;
  if (int st = grouped_scatter_run(uq, us, w2_e4m3, w2_s, o, perm, n, E, dim, inter, offsets, mtiles, cs))
    return st;
  // One thread per 8-element output vector (grid-stride past 2^30 CTAs).
  const long long vecs = T * (dim / 8);
  const int grid = static_cast<int>((vecs + 255) / 256 < (1LL << 30) ? (vecs + 255) / 256 : (1LL << 30));
  moe_combine_kernel<<<grid, 256, 0, cs>>>(static_cast<const uint4*>(o), topk_idx, topk_w, static_cast<int>(T),
                                           static_cast<int>(topk), static_cast<int>(E), static_cast<int>(dim),
                                           static_cast<uint4*>(y_bf16));
  return launch_status();
}
