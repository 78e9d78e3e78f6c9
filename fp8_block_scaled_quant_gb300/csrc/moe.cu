// Routed-expert FFN over block-scaled FP8 ("Administrator & Developer
// Guide", 6.4 MoE expert routing and 8.4 steps 2-5): for every expert e, the
// tokens routed to it go through w2(silu(w1 x) * w3 x) and the results are
// summed per token with the gate weights. The pages' loop (a host-side
// bincount + tolist(), then one Python iteration per expert) becomes:
//
//   moe_permute   three passes: per chunk of 1024 pairs, each pair's rank
//                 among the chunk's earlier pairs of its expert and the
//                 chunk's histogram; one CTA turns the histograms into
//                 per-(chunk, expert) bases, row offsets and 128-row tile
//                 counts; a scatter puts every pair at base + rank (a stable
//                 sort of the (token, slot) pairs by expert id);
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
                        const int* grp_mtiles, int scale_fmt, cudaStream_t stream);

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

// The permutation groups the n (token, slot) pairs by expert, keeping pair
// order (t * topk + j) inside each expert: counts, offsets[E + 1] (exclusive
// scan), mtiles[E + 1] (exclusive scan of ceil(count / 128)), and
// perm[offsets[e] + r] = the r-th pair of expert e. Pairs whose expert id is
// outside [0, E) join no expert and set an error bit.
//
// Rank pass: CTA c takes pairs [1024 c, 1024 c + 1024). A pair's rank among
// the chunk's earlier pairs of its expert is its rank inside its warp
// (__match_any_sync) plus the counts of that expert in the chunk's earlier
// warps; hist[c][e] is the chunk's count of expert e.
constexpr int kPermChunk = kPermThreads;

__global__ void __launch_bounds__(kPermThreads) moe_rank_kernel(const int* __restrict__ idx, int n, int E,
                                                                int* __restrict__ rank, int* __restrict__ hist,
                                                                unsigned* err) {
  extern __shared__ int wtab[];  // [32][E]: per-warp counts, then their prefix over warps
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int k = tid; k < 32 * E; k += kPermThreads) wtab[k] = 0;
  __syncthreads();
  const int i = static_cast<int>(blockIdx.x) * kPermChunk + tid;
  int e = i < n ? __ldg(idx + i) : -1;
  if (i < n && (e < 0 || e >= E)) atomicOr(err, kDevErrBadExpert);
  if (e < 0 || e >= E) e = -1;
  const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
  const int wrank = __popc(m & ((1u << lane) - 1u));
  if (e >= 0 && wrank == 0) wtab[warp * E + e] = __popc(m);
  __syncthreads();
  for (int x = tid; x < E; x += kPermThreads) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = wtab[w * E + x];
      wtab[w * E + x] = run;
      run += c;
    }
    hist[static_cast<size_t>(blockIdx.x) * E + x] = run;
  }
  __syncthreads();
  if (e >= 0) rank[i] = wtab[warp * E + e] + wrank;
}

// Offsets pass (one CTA, thread x for expert x): the histograms become
// per-chunk bases (offsets[x] + the expert's pairs in earlier chunks), and
// counts, offsets and tile counts are written.
__global__ void __launch_bounds__(kPermThreads) moe_offsets_kernel(int* __restrict__ hist_base, int nchunks, int E,
                                                                   int* __restrict__ counts,
                                                                   int* __restrict__ offsets,
                                                                   int* __restrict__ mtiles) {
  __shared__ int wsum[40];
  const int tid = threadIdx.x;
  int total = 0;
  if (tid < E) {
    for (int c = 0; c < nchunks; ++c) {
      const int h = hist_base[static_cast<size_t>(c) * E + tid];
      hist_base[static_cast<size_t>(c) * E + tid] = total;
      total += h;
    }
  }
  int rows, tiles;
  const int off = block_exclusive_scan(total, wsum, &rows);
  const int mt = block_exclusive_scan((total + 127) / 128, wsum, &tiles);
  if (tid < E) {
    if (counts) counts[tid] = total;
    offsets[tid] = off;
    if (mtiles) mtiles[tid] = mt;
    for (int c = 0; c < nchunks; ++c) hist_base[static_cast<size_t>(c) * E + tid] += off;
  }
  if (tid == 0) {
    offsets[E] = rows;
    if (mtiles) mtiles[E] = tiles;
  }
}

// Scatter pass: perm[base[chunk][e] + rank] = pair, for every valid pair
// (chunks of `chunk` consecutive pairs).
__global__ void __launch_bounds__(256) moe_scatter_kernel(const int* __restrict__ idx, const int* __restrict__ rank,
                                                          const int* __restrict__ base, int n, int E, int chunk,
                                                          int* __restrict__ perm) {
  const int i = static_cast<int>(blockIdx.x) * 256 + static_cast<int>(threadIdx.x);
  if (i >= n) return;
  const int e = __ldg(idx + i);
  if (e < 0 || e >= E) return;
  perm[__ldg(base + static_cast<size_t>(i / chunk) * E + e) + __ldg(rank + i)] = i;
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

// y[t] = bf16(sum over routed slots j < n_routed, in order, of w[t, j] * o[t * topk + j]),
// fp32 accumulation; slots routed to no valid expert contribute nothing. Slots
// n_routed .. topk-1 are shared experts (weight 1): their fp32 sum z is
// rounded to bf16 and the row is bf16(bf16(routed sum) + z), the guide's y + z.
// For n_routed <= kCombineMax all routed slots' ids, weights and output vectors
// are requested before the first FMA (the loads are independent; the FMAs keep
// the slot order); more slots take the plain loop.
constexpr int kCombineMax = 8;

__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__global__ void __launch_bounds__(256) moe_combine_kernel(const uint4* __restrict__ o, const int* __restrict__ idx,
                                                          const float* __restrict__ w, int T, int topk,
                                                          int n_routed, int E, int dim, uint4* __restrict__ y) {
  const int dv = dim / 8;
  const long long total = static_cast<long long>(T) * dv;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += stride) {
    const long long t = v / dv;
    const int c = static_cast<int>(v - t * dv);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    auto add = [](float* a, float wj, const uint4& ov) {
      const uint32_t u[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[2 * q] = fmaf(wj, __uint_as_float(u[q] << 16), a[2 * q]);
        a[2 * q + 1] = fmaf(wj, __uint_as_float(u[q] & 0xFFFF0000u), a[2 * q + 1]);
      }
    };
    if (n_routed <= kCombineMax) {
      int e[kCombineMax];
      float wj[kCombineMax];
      uint4 ov[kCombineMax];
#pragma unroll
      for (int j = 0; j < kCombineMax; ++j) {
        e[j] = j < n_routed ? __ldg(idx + t * topk + j) : -1;
        wj[j] = j < n_routed ? __ldg(w + t * topk + j) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kCombineMax; ++j)
        if (e[j] >= 0 && e[j] < E) ov[j] = __ldg(o + (t * topk + j) * dv + c);
#pragma unroll
      for (int j = 0; j < kCombineMax; ++j)
        if (e[j] >= 0 && e[j] < E) add(acc, wj[j], ov[j]);
    } else {
      for (int j = 0; j < n_routed; ++j) {
        const int ej = __ldg(idx + t * topk + j);
        if (ej < 0 || ej >= E) continue;
        add(acc, __ldg(w + t * topk + j), __ldg(o + (t * topk + j) * dv + c));
      }
    }
    uint32_t r[4];
    if (n_routed < topk) {
      float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int j = n_routed; j < topk; ++j) add(z, __ldg(w + t * topk + j), __ldg(o + (t * topk + j) * dv + c));
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(round_bf16(acc[q]), round_bf16(z[q]));
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      r[q] = *reinterpret_cast<const uint32_t*>(&b);
    }
    y[v] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

// Routing with shared experts: slot j < k of token t copies the routed id
// (ids outside [0, E) become -1, join no expert, and set the error bit) and
// its weight; slots k .. k+ns-1 name the shared experts E .. E+ns-1, weight 1.
__global__ void __launch_bounds__(256) moe_augment_kernel(const int* __restrict__ idx, const float* __restrict__ w,
                                                          long long T, int k, int E, int ns,
                                                          int* __restrict__ aidx, float* __restrict__ aw,
                                                          unsigned* err) {
  const int kk = k + ns;
  const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= T * kk) return;
  const long long t = i / kk;
  const int j = static_cast<int>(i - t * kk);
  if (j < k) {
    int e = __ldg(idx + t * k + j);
    if (e < 0 || e >= E) {
      e = -1;
      atomicOr(err, kDevErrBadExpert);
    }
    aidx[i] = e;
    aw[i] = __ldg(w + t * k + j);
  } else {
    aidx[i] = E + (j - k);
    aw[i] = 1.0f;
  }
}

size_t align256(size_t v) { return (v + 255) & ~size_t{255}; }


// Scratch of the permutation: ranks [n], then per-(chunk, expert) bases.
size_t permute_scratch_bytes(int64_t n, int64_t E) {
  const int64_t nchunks = (n + kPermChunk - 1) / kPermChunk;
  return align256(static_cast<size_t>(n) * 4) + align256(static_cast<size_t>(nchunks) * E * 4);
}

int launch_permute(const DevInfo* d, const int* idx, int64_t n, int64_t E, int* counts, int* offsets, int* mtiles,
                   int* perm, void* scratch, cudaStream_t stream) {
  static bool attr_done[64] = {};
  if (d->device >= 64 || !attr_done[d->device]) {
    if (cudaFuncSetAttribute(moe_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             32 * kMaxExperts * 4) != cudaSuccess)
      return FP8BLK_ERR_CUDA;
    if (d->device < 64) attr_done[d->device] = true;
  }
  const int nchunks = static_cast<int>((n + kPermChunk - 1) / kPermChunk);
  int* rank = static_cast<int*>(scratch);
  int* base = reinterpret_cast<int*>(static_cast<uint8_t*>(scratch) + align256(static_cast<size_t>(n) * 4));
  if (nchunks > 0) {
    moe_rank_kernel<<<nchunks, kPermThreads, static_cast<size_t>(32) * E * 4, stream>>>(
        idx, static_cast<int>(n), static_cast<int>(E), rank, base, d->err_word);
    if (int st = launch_status()) return st;
  }
  moe_offsets_kernel<<<1, kPermThreads, 0, stream>>>(base, nchunks, static_cast<int>(E), counts, offsets, mtiles);
  if (int st = launch_status()) return st;
  if (n > 0) {
    moe_scatter_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(idx, rank, base, static_cast<int>(n),
                                                                                   static_cast<int>(E), kPermChunk,
                                                                                   perm);
  }
  return launch_status();
}

// ---- MoE gate ------------------------------------------------------------------
// Per token ("Administrator & Developer Guide", 8.4 and 3.3; "Repository
// overview" MoE data flow): scores s from the logits (sigmoid, or softmax over
// the E experts), selection keys z = s + bias (z = s without a bias); with G > 1
// groups of E/G consecutive experts a group scores its largest z (no bias) or
// the sum of its two largest (bias), and only the TG best groups' experts stay
// eligible; the K best eligible z give the experts in descending order (ties:
// lower index); the weights are their s, divided by the sum of the K when
// `normalize`, times route_scale.
//
// One warp per token. Lane l holds experts [l V, l V + V) (E = 32 V), so a
// group is a run of 32 / G whole lanes: group maxima and top-two pairs merge
// with shuffles inside that run. Each top-k round is a warp argmax over 64-bit
// keys (order-preserving bits of z, then the complement of the index).
constexpr int kGateWarps = 8;

__device__ __forceinline__ uint64_t gate_key(float z, int e) {
  const uint32_t u = __float_as_uint(z);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// The gate of token t, computed by one warp: lane j < K ends with the expert
// of slot j in *out_idx and its weight (normalised, times route_scale) in
// *out_w.
template <int V>
__device__ __forceinline__ void gate_token(const float* __restrict__ logits, const float* __restrict__ bias, int t,
                                           int G, int TG, int K, int sigmoid, float route_scale, int normalize,
                                           int lane, int* out_idx, float* out_w) {
  constexpr int E = 32 * V;
  const float* l = logits + static_cast<size_t>(t) * E + lane * V;
  float s[V], z[V];
  if (sigmoid) {
#pragma unroll
    for (int i = 0; i < V; ++i) s[i] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-__ldg(l + i))));
  } else {
    float x[V], m = -INFINITY;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      x[i] = __ldg(l + i);
      m = fmaxf(m, x[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      x[i] = expf(__fsub_rn(x[i], m));
      sum = __fadd_rn(sum, x[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, o));
#pragma unroll
    for (int i = 0; i < V; ++i) s[i] = __fdiv_rn(x[i], sum);
  }
#pragma unroll
  for (int i = 0; i < V; ++i) z[i] = bias ? __fadd_rn(s[i], __ldg(bias + lane * V + i)) : s[i];

  // Group selection: a lane is eligible while its group is kept.
  bool eligible = true;
  if (G > 1) {
    const int lpg = 32 / G;  // lanes per group
    float a = -INFINITY, b = -INFINITY;  // this lane's two largest z
#pragma unroll
    for (int i = 0; i < V; ++i) {
      if (z[i] > a) {
        b = a;
        a = z[i];
      } else if (z[i] > b) {
        b = z[i];
      }
    }
    for (int o = lpg >> 1; o > 0; o >>= 1) {  // merge the pairs of the group's lanes
      const float a2 = __shfl_xor_sync(0xFFFFFFFFu, a, o);
      const float b2 = __shfl_xor_sync(0xFFFFFFFFu, b, o);
      const float hi = fmaxf(a, a2);
      b = fmaxf(fminf(a, a2), fmaxf(b, b2));
      a = hi;
    }
    const float gscore = bias ? __fadd_rn(a, b) : a;
    const int g = lane / lpg;
    bool kept = false;
    for (int r = 0; r < TG; ++r) {
      const uint64_t best = warp_max_u64(kept ? 0ull : gate_key(gscore, g));
      if (static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best)) == g) kept = true;
    }
    eligible = kept;
  }

  // Top-k experts among the eligible lanes' z.
  uint32_t taken = 0;
  int my_idx = 0;
  float my_s = 0.0f, sum = 0.0f;
  for (int j = 0; j < K; ++j) {
    uint64_t key = 0;
    if (eligible) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const uint64_t k = (taken >> i) & 1u ? 0ull : gate_key(z[i], lane * V + i);
        key = k > key ? k : key;
      }
    }
    key = warp_max_u64(key);
    const int e = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key));
    const int owner = e / V;
    float se = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (lane == owner && e - lane * V == i) {
        se = s[i];
        taken |= 1u << i;
      }
    se = __shfl_sync(0xFFFFFFFFu, se, owner);
    sum = __fadd_rn(sum, se);
    if (lane == j) {
      my_idx = e;
      my_s = se;
    }
  }
  *out_idx = my_idx;
  *out_w = __fmul_rn(normalize ? __fdiv_rn(my_s, sum) : my_s, route_scale);
}

template <int V>
__global__ void __launch_bounds__(kGateWarps * 32) moe_gate_kernel(const float* __restrict__ logits,
                                                                   const float* __restrict__ bias, int T, int G,
                                                                   int TG, int K, int sigmoid, float route_scale,
                                                                   int normalize, int32_t* __restrict__ idx,
                                                                   float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = static_cast<int>(blockIdx.x) * kGateWarps + static_cast<int>(threadIdx.x >> 5);
  if (t >= T) return;  // whole warps leave together
  int e;
  float v;
  gate_token<V>(logits, bias, t, G, TG, K, sigmoid, route_scale, normalize, lane, &e, &v);
  if (lane < K) {
    idx[static_cast<size_t>(t) * K + lane] = e;
    w[static_cast<size_t>(t) * K + lane] = v;
  }
}

// Gate and permutation in one launch. CTA c takes tokens [32 c, 32 c + 32)
// (one warp each) and so the pairs [32 K c, 32 K (c + 1)) of the permutation:
// after the gate it ranks each pair among the chunk's earlier pairs of its
// expert and writes the chunk's per-expert histogram, as the rank pass does.
// The last CTA to arrive on the workspace counter (no CTA waits for another)
// turns the histograms into per-(chunk, expert) bases and writes counts and
// offsets, then resets the counter; one scatter pass finishes the sort.
constexpr int kRouteTokens = 32;

template <int V>
__global__ void __launch_bounds__(1024) moe_route_kernel(const float* __restrict__ logits,
                                                         const float* __restrict__ bias, int T, int G, int TG, int K,
                                                         int sigmoid, float route_scale, int normalize,
                                                         int32_t* __restrict__ idx, float* __restrict__ w,
                                                         int* __restrict__ rank, int* __restrict__ hist,
                                                         int* __restrict__ arrivals, int nchunks,
                                                         int* __restrict__ counts, int* __restrict__ offsets) {
  constexpr int E = 32 * V;
  __shared__ int ids[kRouteTokens * 32];
  __shared__ int wtab[32 * E];  // per-warp counts of each expert, then their prefix over warps
  __shared__ int wsum[40];
  __shared__ int last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = static_cast<int>(blockIdx.x) * kRouteTokens + warp;
  for (int k = tid; k < 32 * E; k += 1024) wtab[k] = 0;
  if (t < T) {
    int e;
    float v;
    gate_token<V>(logits, bias, t, G, TG, K, sigmoid, route_scale, normalize, lane, &e, &v);
    if (lane < K) {
      idx[static_cast<size_t>(t) * K + lane] = e;
      w[static_cast<size_t>(t) * K + lane] = v;
      ids[warp * K + lane] = e;
    }
  } else if (lane < K) {
    ids[warp * K + lane] = -1;
  }
  __syncthreads();
  // Ranks: thread p holds pair p of the chunk (global pair 32 K c + p).
  const int npairs = kRouteTokens * K;
  const int e = tid < npairs ? ids[tid] : -1;
  const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
  const int wrank = __popc(m & ((1u << lane) - 1u));
  if (e >= 0 && wrank == 0) wtab[warp * E + e] = __popc(m);
  __syncthreads();
  for (int x = tid; x < E; x += 1024) {
    int run = 0;
    for (int q = 0; q < 32; ++q) {
      const int c = wtab[q * E + x];
      wtab[q * E + x] = run;
      run += c;
    }
    hist[static_cast<size_t>(blockIdx.x) * E + x] = run;
  }
  __syncthreads();
  if (e >= 0) rank[static_cast<size_t>(blockIdx.x) * npairs + tid] = wtab[warp * E + e] + wrank;
  // Arrive; the last CTA computes the bases.
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(arrivals, 1) == nchunks - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // Bases of every (chunk, expert): thread (s, e) takes expert e and the s-th
  // of kSlices ranges of chunks; the ranges' sums are scanned per expert (in
  // shared memory, reusing wtab), the totals over experts.
  constexpr int kSlices = 1024 / E;
  const int e_t = tid % E, s_t = tid / E;  // threads past kSlices * E take no chunks
  const int c0 = s_t < kSlices ? static_cast<int>(static_cast<long long>(s_t) * nchunks / kSlices) : 0;
  const int c1 = s_t < kSlices ? static_cast<int>(static_cast<long long>(s_t + 1) * nchunks / kSlices) : 0;
  int part = 0;
  for (int c = c0; c < c1; ++c) part += __ldcg(hist + static_cast<size_t>(c) * E + e_t);
  __syncthreads();
  if (s_t < kSlices) wtab[s_t * E + e_t] = part;
  __syncthreads();
  int before = 0, total = 0;
  for (int q = 0; q < kSlices; ++q) {
    const int v = wtab[q * E + e_t];
    before += q < s_t ? v : 0;
    total += v;
  }
  int rows;
  const int off = block_exclusive_scan(tid < E ? total : 0, wsum, &rows);
  if (tid < E) {
    counts[tid] = total;
    offsets[tid] = off;
  }
  __syncthreads();
  if (tid < E) wtab[tid] = off;  // expert offsets, for every slice's threads
  __syncthreads();
  int run = wtab[e_t] + before;
  for (int c = c0; c < c1; ++c) {
    int* h = hist + static_cast<size_t>(c) * E + e_t;
    const int v = __ldcg(h);
    *h = run;
    run += v;
  }
  if (tid == 0) {
    offsets[E] = rows;
    *arrivals = 0;
  }
}

int launch_gate(const float* logits, const float* bias, int64_t T, int64_t E, int64_t G, int64_t TG, int64_t K,
                int sigmoid, float route_scale, int normalize, int32_t* idx, float* w, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((T + kGateWarps - 1) / kGateWarps);
  const int t = static_cast<int>(T), g = static_cast<int>(G), tg = static_cast<int>(TG), k = static_cast<int>(K);
#define FP8BLK_GATE_CASE(v)                                                                                   \
  case v:                                                                                                     \
    moe_gate_kernel<v><<<grid, kGateWarps * 32, 0, stream>>>(logits, bias, t, g, tg, k, sigmoid, route_scale, \
                                                              normalize, idx, w);                             \
    break;
  switch (E / 32) {
    FP8BLK_GATE_CASE(1)
    FP8BLK_GATE_CASE(2)
    FP8BLK_GATE_CASE(3)
    FP8BLK_GATE_CASE(4)
    FP8BLK_GATE_CASE(5)
    FP8BLK_GATE_CASE(6)
    FP8BLK_GATE_CASE(7)
    FP8BLK_GATE_CASE(8)
    default: return FP8BLK_ERR_SHAPE;
  }
#undef FP8BLK_GATE_CASE
  return launch_status();
}

// Workspace of the fused route: [arrival counter, 256 B][ranks: T*K ints][bases: chunks x E ints].
size_t route_workspace_bytes(int64_t T, int64_t K, int64_t E) {
  const int64_t nchunks = (T + kRouteTokens - 1) / kRouteTokens;
  return 256 + align256(static_cast<size_t>(T) * K * 4) + align256(static_cast<size_t>(nchunks) * E * 4);
}

int launch_route(const float* logits, const float* bias, int64_t T, int64_t E, int64_t G, int64_t TG, int64_t K,
                 int sigmoid, float route_scale, int normalize, int32_t* idx, float* w, int* counts, int* offsets,
                 int* perm, void* workspace, cudaStream_t stream) {
  const int nchunks = static_cast<int>((T + kRouteTokens - 1) / kRouteTokens);
  int* arrivals = static_cast<int*>(workspace);
  int* rank = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + 256);
  int* base = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + 256 + align256(static_cast<size_t>(T) * K * 4));
  const int t = static_cast<int>(T), g = static_cast<int>(G), tg = static_cast<int>(TG), k = static_cast<int>(K);
#define FP8BLK_ROUTE_CASE(v)                                                                                      \
  case v:                                                                                                         \
    moe_route_kernel<v><<<nchunks, 1024, 0, stream>>>(logits, bias, t, g, tg, k, sigmoid, route_scale, normalize, \
                                                      idx, w, rank, base, arrivals, nchunks, counts, offsets);    \
    break;
  switch (E / 32) {
    FP8BLK_ROUTE_CASE(1)
    FP8BLK_ROUTE_CASE(2)
    FP8BLK_ROUTE_CASE(3)
    FP8BLK_ROUTE_CASE(4)
    FP8BLK_ROUTE_CASE(5)
    FP8BLK_ROUTE_CASE(6)
    FP8BLK_ROUTE_CASE(7)
    FP8BLK_ROUTE_CASE(8)
    default: return FP8BLK_ERR_SHAPE;
  }
#undef FP8BLK_ROUTE_CASE
  if (int st = launch_status()) return st;
  const int64_t n = T * K;
  moe_scatter_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
      idx, rank, base, static_cast<int>(n), static_cast<int>(E), kRouteTokens * k, perm);
  return launch_status();
}

}  // namespace
}  // namespace fp8blk

using namespace fp8blk;

extern "C" size_t fp8blk_moe_permute_workspace_bytes(int64_t T, int64_t topk, int64_t E) {
  if (T < 0 || topk < 0 || E <= 0) return 0;
  const size_t b = permute_scratch_bytes(T * topk, E);
  return b > 256 ? b : 256;
}

extern "C" int fp8blk_moe_permute(const int32_t* topk_idx, int64_t T, int64_t topk, int64_t E, int32_t* counts,
                                  int32_t* offsets, int32_t* perm, void* workspace, size_t workspace_bytes,
                                  fp8blk_stream_t stream) {
  if (T < 0 || topk < 0 || E <= 0 || E > kMaxExperts || T * topk > (int64_t{1} << 31) - 1) return FP8BLK_ERR_SHAPE;
  if (!counts || !offsets) return FP8BLK_ERR_NULL;
  if (T * topk > 0 && (!topk_idx || !perm)) return FP8BLK_ERR_NULL;
  if (!workspace || workspace_bytes < fp8blk_moe_permute_workspace_bytes(T, topk, E)) return FP8BLK_ERR_WORKSPACE;
  if (!is_aligned(workspace, 256)) return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  return launch_permute(d, topk_idx, T * topk, E, counts, offsets, nullptr, perm, workspace,
                        reinterpret_cast<cudaStream_t>(stream));
}

namespace {

int gate_shape_status(const float* bias, int64_t T, int64_t E, int64_t n_groups, int64_t topk_groups, int64_t topk,
                      int score_func, float route_scale) {
  if (score_func != FP8BLK_SCORE_SOFTMAX && score_func != FP8BLK_SCORE_SIGMOID) return FP8BLK_ERR_ARG;
  if (!(route_scale == route_scale) || route_scale == INFINITY || route_scale == -INFINITY) return FP8BLK_ERR_ARG;
  if (T < 0 || T > (int64_t{1} << 31) - 1 || E < 32 || E > 256 || E % 32 || n_groups < 1 || 32 % n_groups ||
      topk_groups < 1 || topk_groups > n_groups || topk < 1 || topk > 32 || topk > topk_groups * (E / n_groups) ||
      (bias && n_groups > 1 && E / n_groups < 2))
    return FP8BLK_ERR_SHAPE;
  return FP8BLK_OK;
}

}  // namespace

extern "C" size_t fp8blk_moe_route_workspace_bytes(int64_t T, int64_t topk, int64_t E) {
  if (T < 0 || topk < 0 || E <= 0) return 0;
  return route_workspace_bytes(T, topk, E);
}

extern "C" int fp8blk_moe_route(const float* logits, const float* bias, int64_t T, int64_t E, int64_t n_groups,
                                int64_t topk_groups, int64_t topk, int score_func, float route_scale, int normalize,
                                int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets, int32_t* perm,
                                void* workspace, size_t workspace_bytes, fp8blk_stream_t stream) {
  if (int st = gate_shape_status(bias, T, E, n_groups, topk_groups, topk, score_func, route_scale)) return st;
  if (T * topk > (int64_t{1} << 31) - 1) return FP8BLK_ERR_SHAPE;
  if (!counts || !offsets) return FP8BLK_ERR_NULL;
  if (T > 0 && (!logits || !topk_idx || !topk_w || !perm)) return FP8BLK_ERR_NULL;
  if (!is_aligned(logits, 4) || !is_aligned(topk_idx, 4) || !is_aligned(topk_w, 4) || !is_aligned(counts, 4) ||
      !is_aligned(offsets, 4) || !is_aligned(perm, 4) || (bias && !is_aligned(bias, 4)))
    return FP8BLK_ERR_ALIGN;
  if (!workspace || workspace_bytes < route_workspace_bytes(T, topk, E)) return FP8BLK_ERR_WORKSPACE;
  if (!is_aligned(workspace, 256)) return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {  // no pairs: every count and offset is zero
    if (cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, cs) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, cs) != cudaSuccess)
      return FP8BLK_ERR_CUDA;
    return FP8BLK_OK;
  }
  return launch_route(logits, bias, T, E, n_groups, topk_groups, topk, score_func == FP8BLK_SCORE_SIGMOID,
                      route_scale, normalize != 0, topk_idx, topk_w, counts, offsets, perm, workspace, cs);
}

extern "C" int fp8blk_moe_gate(const float* logits, const float* bias, int64_t T, int64_t E, int64_t n_groups,
                               int64_t topk_groups, int64_t topk, int score_func, float route_scale, int normalize,
                               int32_t* topk_idx, float* topk_w, fp8blk_stream_t stream) {
  if (int st = gate_shape_status(bias, T, E, n_groups, topk_groups, topk, score_func, route_scale)) return st;
  if (T == 0) return FP8BLK_OK;
  if (!logits || !topk_idx || !topk_w) return FP8BLK_ERR_NULL;
  if (!is_aligned(logits, 4) || !is_aligned(topk_idx, 4) || !is_aligned(topk_w, 4) || (bias && !is_aligned(bias, 4)))
    return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  return launch_gate(logits, bias, T, E, n_groups, topk_groups, topk, score_func == FP8BLK_SCORE_SIGMOID,
                     route_scale, normalize != 0, topk_idx, topk_w, reinterpret_cast<cudaStream_t>(stream));
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

// FFN workspace: [GEMM workspace][x_q M*dim][x_s M*dim/128][u_q M*inter]
// [u_s M*inter/128]. The w1/w3 GEMM and the w2 GEMM share the GEMM workspace,
// which comes first so that its tile counters sit at the same offset whatever
// the shape. Sharing is safe: each GEMM touches the workspace only after its
// dependency wait, so the w2 GEMM starts on it once the w1/w3 GEMM has
// completed and left its counters at zero.
static size_t ffn_gemm_bytes(int64_t M, int64_t dim, int64_t inter) {
  const size_t a = swiglu_workspace_bytes(M, inter, dim), b = gemm_workspace_bytes(M, dim, inter);
  return align256(a > b ? a : b);
}

extern "C" size_t fp8blk_ffn_workspace_bytes(int64_t M, int64_t dim, int64_t inter) {
  if (M < 0 || dim < 0 || inter < 0) return 0;
  return ffn_gemm_bytes(M, dim, inter) + align256(static_cast<size_t>(M) * dim) +
         align256(static_cast<size_t>(M) * (dim / kBlock) * 4) + align256(static_cast<size_t>(M) * inter) +
         align256(static_cast<size_t>(M) * (inter / kBlock) * 4);
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
  uint8_t* gws = static_cast<uint8_t*>(workspace);
  const size_t gbytes = ffn_gemm_bytes(M, dim, inter);
  uint8_t* p = gws + gbytes;
  uint8_t* xq = p;
  p += align256(static_cast<size_t>(M) * dim);
  float* xs = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(M) * (dim / kBlock) * 4);
  uint8_t* uq = p;
  p += align256(static_cast<size_t>(M) * inter);
  float* us = reinterpret_cast<float*>(p);
  if (int st = act_quant_launch(x_bf16, M, dim, xq, xs, scale_fmt, cs, true)) return st;
  if (int st = swiglu_run(xq, xs, w1_e4m3, w1_s, w3_e4m3, w3_s, uq, us, M, inter, dim, scale_fmt, gws, gbytes, cs))
    return st;
  return gemm_run(uq, us, w2_e4m3, w2_s, y_bf16, M, dim, inter, scale_fmt, gws, gbytes, cs);
}

namespace {

struct MoeLayout {
  size_t counts, offsets, mtiles, perm, pscratch, aidx, aw, xg, xgs, uq, us, o, total;
};

// topk counts every slot of a token, shared experts included; E every expert.
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
  l.pscratch = take(permute_scratch_bytes(static_cast<int64_t>(n), E));
  l.aidx = take(n * 4);
  l.aw = take(n * 4);
  l.xg = take(n * dim);
  l.xgs = take(n * (dim / kBlock) * 4);
  l.uq = take(n * inter);
  l.us = take(n * (inter / kBlock) * 4);
  l.o = take(n * dim * 2);
  l.total = off;
  return l;
}

}  // namespace

extern "C" size_t fp8blk_moe_workspace_bytes(int64_t T, int64_t topk, int64_t E, int64_t dim, int64_t inter,
                                             int64_t n_shared) {
  if (T < 0 || topk < 0 || E <= 0 || dim < 0 || inter < 0 || n_shared < 0) return 0;
  return moe_layout(T, topk + n_shared, E + n_shared, dim, inter).total;
}

extern "C" int fp8blk_moe_grouped_gemm(const void* x_e4m3, const float* x_s, const int32_t* topk_idx,
                                       const float* topk_w, const void* w1_e4m3, const float* w1_s,
                                       const void* w3_e4m3, const float* w3_s, const void* w2_e4m3,
                                       const float* w2_s, void* y_bf16, int64_t T, int64_t topk, int64_t E,
                                       int64_t dim, int64_t inter, int64_t n_shared, int scale_fmt, void* workspace,
                                       size_t workspace_bytes, fp8blk_stream_t stream) {
  if (!scale_fmt_valid(scale_fmt)) return FP8BLK_ERR_ARG;
  if (T < 0 || topk < 0 || n_shared < 0 || E <= 0 || E + n_shared > kMaxExperts || dim <= 0 || inter <= 0 ||
      dim % 256 || inter % kBlock)
    return FP8BLK_ERR_SHAPE;
  const int64_t slots = topk + n_shared, experts = E + n_shared;  // per token; in the stacked weights
  const int64_t n = T * slots;
  if (n > (int64_t{1} << 31) - 1 || experts * inter > (int64_t{1} << 31) - 1 ||
      experts * dim > (int64_t{1} << 31) - 1)
    return FP8BLK_ERR_SHAPE;
  if (T == 0) return FP8BLK_OK;
  if (!y_bf16) return FP8BLK_ERR_NULL;
  if (slots == 0) return cuda_status(cudaMemsetAsync(y_bf16, 0, static_cast<size_t>(T) * dim * 2,
                                                     reinterpret_cast<cudaStream_t>(stream)));
  if (!x_e4m3 || !x_s || (topk > 0 && (!topk_idx || !topk_w)) || !w1_e4m3 || !w1_s || !w3_e4m3 || !w3_s ||
      !w2_e4m3 || !w2_s)
    return FP8BLK_ERR_NULL;
  if (!is_aligned(x_e4m3, 16) || !is_aligned(w1_e4m3, 16) || !is_aligned(w3_e4m3, 16) ||
      !is_aligned(w2_e4m3, 16) || !is_aligned(y_bf16, 16) || !is_aligned(x_s, 4) || !is_aligned(w1_s, 4) ||
      !is_aligned(w3_s, 4) || !is_aligned(w2_s, 4) || !is_aligned(topk_idx, 4) || !is_aligned(topk_w, 4))
    return FP8BLK_ERR_ALIGN;
  const MoeLayout l = moe_layout(T, slots, experts, dim, inter);
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

  // Shared experts (Guide 8.4 step 6: the shared MLP runs on every token)
  // become extra slots naming experts E .. E+n_shared-1, so one permutation,
  // one pair of grouped GEMMs and one combine serve routed and shared rows.
  const int32_t* ridx = topk_idx;
  const float* rw = topk_w;
  if (n_shared > 0) {
    int* aidx = reinterpret_cast<int*>(ws + l.aidx);
    float* aw = reinterpret_cast<float*>(ws + l.aw);
    moe_augment_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, cs>>>(
        topk_idx, topk_w, T, static_cast<int>(topk), static_cast<int>(E), static_cast<int>(n_shared), aidx, aw,
        d->err_word);
    if (int st = launch_status()) return st;
    ridx = aidx;
    rw = aw;
  }
  if (int st = launch_permute(d, ridx, n, experts, counts, offsets, mtiles, perm, ws + l.pscratch, cs)) return st;
  // One warp per routed row (at most T * slots of them), as many CTAs as that
  // takes: the resident CTAs then copy one contiguous window of rows at a time.
  const long long gather_grid = (static_cast<long long>(n) + 7) / 8;
  moe_gather_kernel<<<static_cast<unsigned>(gather_grid < (1LL << 30) ? gather_grid : (1LL << 30)), 256, 0, cs>>>(
      static_cast<const uint4*>(x_e4m3), x_s, perm, offsets, static_cast<int>(experts), static_cast<int>(slots),
      static_cast<int>(dim), reinterpret_cast<uint4*>(xg), xgs);
  if (int st = launch_status()) return st;
  if (int st = grouped_swiglu_run(xg, xgs, w1_e4m3, w1_s, w3_e4m3, w3_s, uq, us, n, experts, inter, dim, offsets,
                                  mtiles, scale_fmt, cs))
    return st;
  if (int st = grouped_scatter_run(uq, us, w2_e4m3, w2_s, o, perm, n, experts, dim, inter, offsets, mtiles,
                                   scale_fmt, cs))
    return st;
  // One thread per 8-element output vector (grid-stride past 2^30 CTAs).
  const long long vecs = T * (dim / 8);
  const int grid = static_cast<int>((vecs + 255) / 256 < (1LL << 30) ? (vecs + 255) / 256 : (1LL << 30));
  moe_combine_kernel<<<grid, 256, 0, cs>>>(static_cast<const uint4*>(o), ridx, rw, static_cast<int>(T),
                                           static_cast<int>(slots), static_cast<int>(topk),
                                           static_cast<int>(experts), static_cast<int>(dim),
                                           static_cast<uint4*>(y_bf16));
  return launch_status();
}
