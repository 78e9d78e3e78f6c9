// Decode-sized block-scaled FP8 GEMM (M <= 16 tokens) for sm_103a
// ("Administrator & Developer Guide", 8.5.3 fp8_gemm_kernel; 6.3 The FP8 path):
//
//   C[m, n] = sum_kb a_s[m, kb] * w_s[n/128, kb] * sum_{k in kb} a[m, k] w[n, k]
//
// At decode sizes the layer is one pass over the weight; what a launch does
// after its dependency wait (the previous kernel wrote a and a_s) decides its
// time. So:
//   - One CTA per slice of R weight rows (R = ceil(N / SMs) rounded up to 8,
//     one CTA per SM). Before the wait, one thread requests the whole slice,
//     R rows x K, in a few large TMA boxes (a 3-D map: 128 bytes of a K block
//     x R rows x K blocks, 128-byte swizzle), so the weight stream runs while
//     the previous kernel finishes.
//   - Warps = K slices x row-group parts (at most five 16-row groups per warp
//     with one token fragment, three with two; at most 16 warps). Right after
//     the wait every warp loads its tokens' operand
//     fragments and a_s for its K blocks straight from global memory into
//     registers (the next K block's while it multiplies the current one), so
//     no CTA-wide staging stands between the wait and the first product.
//   - Per K block and row group a warp runs four mma.sync m16n8k32 (e4m3 x
//     e4m3, fp32 accumulate; weight rows as M, tokens as N) into a fresh
//     register accumulator and promotes it, acc += D * (a_s[m, kb] *
//     w_s[n / 128, kb]), as soon as that block's box has landed: the boxes
//     that land first are multiplied while the rest stream in. One token
//     fragment serves all of the warp's row groups.
//   - The K slices' fp32 sums are added in slice order in shared memory and
//     stored as bf16.
//
// Operand fragments. Lane (g = lane / 4, t = lane % 4) of a warp loads bytes
// [32 t, 32 t + 32) of the K block for weight rows g and g + 8 of a group and
// for token g (and g + 8 with two token fragments). MMA j (0..3) of the
// block takes bytes [8 j, 8 j + 8) of those 32: the first four fill the
// fragment slots of k = 4 t .. 4 t + 3, the last four those of
// k = 4 t + 16 .. 4 t + 19. Each K position of the block thus goes to exactly
// one (MMA, slot) pair, the same for both operands, so the four MMAs form
// every product a[m, k] w[n, k] of the block once.
//
// Every mbarrier wait is bounded (2 s): on expiry the CTA records an error
// bit, skips its remaining work, waits (bounded) for its copies and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fp8blk.h"
#include "host.cuh"
#include "ptx.cuh"

namespace fp8blk {

namespace {

constexpr int kDecodeMaxWarps = 16;
// Warps a CTA aims for: K slices x row-group parts.
constexpr int kDecodeWarps = 16;
// Most 16-row groups one warp multiplies: its accumulators stay in registers
// (five with one token fragment, three with two).
__host__ __device__ constexpr int decode_groups_per_warp(int nt) { return nt == 1 ? 5 : 3; }
#ifndef FP8BLK_DECODE_BOXES
#define FP8BLK_DECODE_BOXES 4
#endif
constexpr int kDecodeSmemLimit = 232448;

struct DecodeParams {
  const uint8_t* a;   // e4m3 [M, K]
  const float* a_s;   // [M, Kb]
  const float* w_s;   // [ceil(N / 128), Kb]
  __nv_bfloat16* c;   // bf16 [M, N]
  unsigned* err;      // device error word
  int M, N, K, Kb;
  int R;              // weight rows per CTA (a multiple of 8)
  int groups;         // 16-row groups per CTA, ceil(R / 16)
  int kslices;        // K slices (warps = kslices * gparts)
  int gparts;         // row-group parts per K slice, at most decode_groups_per_warp groups each
  int nbox, kbb;      // weight boxes per CTA and K blocks per box
  int wblk;           // weight-scale rows (128-row blocks) staged per CTA
  uint32_t off_ws, off_bar;  // shared-memory offsets from the 1024-byte aligned base
};

// 3-D tiled load of the box at (x, y, z) into shared memory; the transaction
// bytes complete on `bar`. Out-of-range elements are zero-filled.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// d += A (16 x 32, rows) * B (32 x 8, columns), e4m3 operands, fp32 accumulators.
__device__ __forceinline__ void mma_e4m3_16x8x32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT>
__global__ void __launch_bounds__(kDecodeMaxWarps * 32, 1)
    fp8_gemm_decode_kernel(const __grid_constant__ CUtensorMap wmap, const DecodeParams p) {
  constexpr int kTok = NT * 8;  // token columns (tokens past M are zero)
  constexpr int kGpw = decode_groups_per_warp(NT);
  extern __shared__ uint8_t dsmem[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t{1023});
  float* wss = reinterpret_cast<float*>(sm + p.off_ws);  // [wblk][Kb]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.off_bar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + p.nbox);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nthr = blockDim.x;
  const int r0 = blockIdx.x * p.R;
  const uint32_t box_bytes = static_cast<uint32_t>(p.kbb) * p.R * 128;

  if (tid == 0) {
    *abort_flag = 0;
    for (int b = 0; b < p.nbox; ++b) mbar_init(&bars[b], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    tma_prefetch_desc(&wmap);
    for (int b = 0; b < p.nbox; ++b) {
      mbar_arrive_expect_tx(&bars[b], box_bytes);
      tma_load_3d(sm + static_cast<size_t>(b) * box_bytes, &wmap, &bars[b], 0, r0, b * p.kbb);
    }
  }
  // The weight scales of the slice's 128-row blocks (a weight operand: read
  // before the wait), by the last warp (warp 0's lane 0 issues the copies).
  const int blk0 = r0 / 128;
  const int nwb = (p.N + 127) / 128;
  for (int i = tid - (nthr - 32 > 0 ? nthr - 32 : 0); i >= 0 && i < p.wblk * p.Kb; i += 32) {
    const int b = blk0 + i / p.Kb;
    wss[i] = b < nwb ? p.w_s[static_cast<size_t>(b) * p.Kb + i % p.Kb] : 0.f;
  }
  griddep_launch_dependents();
  griddep_wait();

  const int ks = warp / p.gparts, gp = warp % p.gparts;
  const int g = lane >> 2, t = lane & 3;
  const int kb0 = ks * p.Kb / p.kslices, kb1 = (ks + 1) * p.Kb / p.kslices;
  const int gfirst = gp * p.groups / p.gparts, ng = (gp + 1) * p.groups / p.gparts - gfirst;

  // This lane's token fragments and activation scales for K block kb.
  auto load_tokens = [&](int kb, uint4 (&bx)[NT][2], float (&sa)[NT][2]) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int m = n * 8 + g, m2 = n * 8 + 2 * t;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        bx[n][h] = m < p.M ? *reinterpret_cast<const uint4*>(p.a + static_cast<size_t>(m) * p.K + kb * 128 + t * 32 +
                                                               h * 16)
                           : make_uint4(0u, 0u, 0u, 0u);
      sa[n][0] = m2 < p.M ? p.a_s[static_cast<size_t>(m2) * p.Kb + kb] : 0.f;
      sa[n][1] = m2 + 1 < p.M ? p.a_s[static_cast<size_t>(m2 + 1) * p.Kb + kb] : 0.f;
    }
  };
  uint4 bx[NT][2], bn[NT][2];
  float sa[NT][2], sn[NT][2];
  load_tokens(kb0, bx, sa);
  __syncthreads();  // the weight scales are in shared memory

  float acc[kGpw][NT][4];
#pragma unroll
  for (int gi = 0; gi < kGpw; ++gi)
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[gi][n][0] = acc[gi][n][1] = acc[gi][n][2] = acc[gi][n][3] = 0.f;

  int waited = -1;
  for (int kb = kb0; kb < kb1; ++kb) {
    if (kb + 1 < kb1) load_tokens(kb + 1, bn, sn);
    const int box = kb / p.kbb;
    if (box != waited) {
      // mma.sync needs the whole warp: leave together if any lane gave up.
      const bool landed = mbar_wait(&bars[box], 0, abort_flag, p.err, kDevErrTimeoutProducer);
      if (!__all_sync(0xFFFFFFFFu, landed)) break;
      waited = box;
    }
    const uint8_t* wk = sm + static_cast<size_t>(kb) * p.R * 128;
#pragma unroll
    for (int gi = 0; gi < kGpw; ++gi) {
      if (gi < ng) {
        // Weight rows rl and rh of K block kb: chunks 2t and 2t + 1 of each
        // 128-byte row, at chunk ^ (row % 8) (the 128-byte swizzle; rows of
        // a box start on 1024-byte boundaries every 8 rows since R % 8 == 0).
        const int rl = (gfirst + gi) * 16 + g, rh = rl + 8;
        const bool hi_ok = rh < p.R;
        uint4 alo[2], ahi[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          alo[h] = *reinterpret_cast<const uint4*>(wk + rl * 128 + (((2 * t + h) ^ (rl & 7)) << 4));
          ahi[h] = hi_ok ? *reinterpret_cast<const uint4*>(wk + rh * 128 + (((2 * t + h) ^ (rh & 7)) << 4))
                         : make_uint4(0u, 0u, 0u, 0u);
        }
        const float wsl = wss[(min(r0 + rl, p.N - 1) / 128 - blk0) * p.Kb + kb];
        const float wsh = wss[(min(r0 + rh, p.N - 1) / 128 - blk0) * p.Kb + kb];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_e4m3_16x8x32(d, alo[0].x, ahi[0].x, alo[0].y, ahi[0].y, bx[n][0].x, bx[n][0].y);
          mma_e4m3_16x8x32(d, alo[0].z, ahi[0].z, alo[0].w, ahi[0].w, bx[n][0].z, bx[n][0].w);
          mma_e4m3_16x8x32(d, alo[1].x, ahi[1].x, alo[1].y, ahi[1].y, bx[n][1].x, bx[n][1].y);
          mma_e4m3_16x8x32(d, alo[1].z, ahi[1].z, alo[1].w, ahi[1].w, bx[n][1].z, bx[n][1].w);
          // D[i]: row rl (i < 2) or rh, token n * 8 + 2t + (i & 1).
          acc[gi][n][0] = fmaf(d[0], sa[n][0] * wsl, acc[gi][n][0]);
          acc[gi][n][1] = fmaf(d[1], sa[n][1] * wsl, acc[gi][n][1]);
          acc[gi][n][2] = fmaf(d[2], sa[n][0] * wsh, acc[gi][n][2]);
          acc[gi][n][3] = fmaf(d[3], sa[n][1] * wsh, acc[gi][n][3]);
        }
      }
    }
    if (kb + 1 < kb1) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        bx[n][0] = bn[n][0];
        bx[n][1] = bn[n][1];
        sa[n][0] = sn[n][0];
        sa[n][1] = sn[n][1];
      }
    }
  }
  __syncthreads();  // every warp is done with the weight boxes
  if (*abort_flag) {
    // A box never landed: wait (bounded) for the copies, then leave.
    if (tid == 0)
      for (int b = 0; b < p.nbox; ++b) mbar_wait(&bars[b], 0, nullptr, p.err, kDevErrTimeoutDrain);
    return;
  }

  // K-slice partials into the weight area: part[ks][token][row of the slice],
  // rows of `rp` floats (rp % 32 == 4: the 32 lanes of one store hit 32 banks).
  float* part = reinterpret_cast<float*>(sm);
  const int rp = p.groups * 16 + 4;
#pragma unroll
  for (int gi = 0; gi < kGpw; ++gi) {
    if (gi < ng) {
      const int rl = (gfirst + gi) * 16 + g, rh = rl + 8;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        float* q = part + static_cast<size_t>(ks * kTok + n * 8 + 2 * t) * rp;
        q[rl] = acc[gi][n][0];
        q[rp + rl] = acc[gi][n][1];
        q[rh] = acc[gi][n][2];
        q[rp + rh] = acc[gi][n][3];
      }
    }
  }
  __syncthreads();
  // Each output: its K slices' partials added in slice order (with one token
  // fragment loaded eight at a time; with two, whose accumulators leave fewer
  // registers, one at a time).
  for (int i = tid; i < p.M * p.R; i += nthr) {
    const int m = i / p.R, r = i - m * p.R;
    if (r0 + r >= p.N) continue;
    const float* col = part + static_cast<size_t>(m) * rp + r;
    float s = col[0];
    if constexpr (NT == 1) {
#pragma unroll
      for (int q0 = 0; q0 < kDecodeMaxWarps; q0 += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = q0 + u > 0 && q0 + u < p.kslices ? col[static_cast<size_t>(q0 + u) * kTok * rp] : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (q0 + u > 0 && q0 + u < p.kslices) s += v[u];
      }
    } else {
      for (int q = 1; q < p.kslices; ++q) s += col[static_cast<size_t>(q) * kTok * rp];
    }
    p.c[static_cast<size_t>(m) * p.N + r0 + r] = __float2bfloat16_rn(s);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn slice_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// The e4m3 weight [N, K] as a 3-D tensor (128 bytes of a K block, row, K
// block; strides K and 128 bytes) read in boxes of 128 x R rows x kbb blocks,
// 128-byte swizzled; rows past N and blocks past Kb read as zeros.
bool make_slice_map(CUtensorMap* map, const void* w, uint64_t N, uint64_t K, uint32_t R, uint32_t kbb) {
  EncodeTiledFn enc = slice_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {128, N, K / 128};
  const cuuint64_t strides[2] = {K, 128};
  const cuuint32_t box[3] = {128, R, kbb};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(w), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DecodePlan {
  bool ok;
  int nt, ctas, warps;
  size_t smem;
  DecodeParams p;
};

uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

DecodePlan decode_plan(int64_t M, int64_t N, int64_t K, int sm_count) {
  DecodePlan d{};
  if (M < 1 || M > 16 || N < 1 || K < kBlock || K % kBlock != 0 || sm_count < 1) return d;
  if (N > (int64_t{1} << 31) - 1 || K > (int64_t{1} << 20)) return d;
  const int64_t Kb = K / kBlock;
  int64_t R = (N + sm_count - 1) / sm_count;
  R = (R + 7) / 8 * 8;
  if (R > 256) return d;  // a TMA box has at most 256 rows
  int nbox = static_cast<int>(Kb < FP8BLK_DECODE_BOXES ? Kb : FP8BLK_DECODE_BOXES);
  const int64_t kbb = (Kb + nbox - 1) / nbox;
  if (kbb > 256) return d;
  nbox = static_cast<int>((Kb + kbb - 1) / kbb);  // every box holds at least one K block
  const int groups = static_cast<int>((R + 15) / 16);
  d.nt = M <= 8 ? 1 : 2;
  const int gpw = decode_groups_per_warp(d.nt);
  int gparts = (groups + gpw - 1) / gpw;
  int kslices = kDecodeWarps / gparts;
  if (kslices < 1) kslices = 1;
  if (kslices > Kb) kslices = static_cast<int>(Kb);
  // Few K blocks: spread the row groups over more warps instead.
  const int more = kDecodeWarps / kslices;
  if (more > gparts) gparts = more < groups ? more : groups;
  const int tok = d.nt * 8;
  const uint64_t wbytes = static_cast<uint64_t>(nbox) * kbb * R * 128;
  const uint64_t pbytes = static_cast<uint64_t>(kslices) * tok * (groups * 16 + 4) * 4;
  const uint64_t area = round_up(static_cast<uint32_t>(wbytes > pbytes ? wbytes : pbytes), 16);
  const int wblk = static_cast<int>((R + 127) / 128 + 1);
  DecodeParams& p = d.p;
  p.off_ws = static_cast<uint32_t>(area);
  p.off_bar = round_up(p.off_ws + static_cast<uint32_t>(wblk * Kb * 4), 8);
  d.smem = 1024 + p.off_bar + static_cast<size_t>(nbox) * 8 + 8;
  if (area > (uint64_t{1} << 30) || d.smem > kDecodeSmemLimit) return d;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.Kb = static_cast<int>(Kb);
  p.R = static_cast<int>(R);
  p.groups = groups;
  p.kslices = kslices;
  p.gparts = gparts;
  p.nbox = nbox;
  p.kbb = static_cast<int>(kbb);
  p.wblk = wblk;
  d.ctas = static_cast<int>((N + R - 1) / R);
  d.warps = kslices * gparts;
  d.ok = d.warps <= kDecodeMaxWarps;
  return d;
}

template <int NT>
int decode_launch(const DevInfo* dev, const CUtensorMap& map, const DecodePlan& d, cudaStream_t stream) {
  static bool attr_done[64] = {};
  auto kern = fp8_gemm_decode_kernel<NT>;
  if (dev->device >= 64 || !attr_done[dev->device]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecodeSmemLimit) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
      return FP8BLK_ERR_CUDA;
    if (dev->device < 64) attr_done[dev->device] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(d.ctas));
  cfg.blockDim = dim3(static_cast<unsigned>(d.warps * 32));
  cfg.dynamicSmemBytes = d.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, map, d.p));
}

}  // namespace

bool decode_gemm_fits(int64_t M, int64_t N, int64_t K, int sm_count) {
  return decode_plan(M, N, K, sm_count).ok;
}

// Runs C = A W^T with the decode kernel when the shape fits it (*used = true);
// otherwise launches nothing. The arguments have passed fp8_gemm's checks
// (non-empty shape, K > 0, pointers present and aligned).
int decode_gemm_run(const DevInfo* dev, const void* a, const float* a_s, const void* w, const float* w_s, void* c,
                    int64_t M, int64_t N, int64_t K, cudaStream_t stream, bool* used) {
  *used = false;
  DecodePlan d = decode_plan(M, N, K, dev->sm_count);
  if (!d.ok) return FP8BLK_OK;
  CUtensorMap map;
  if (!make_slice_map(&map, w, static_cast<uint64_t>(N), static_cast<uint64_t>(K), static_cast<uint32_t>(d.p.R),
                      static_cast<uint32_t>(d.p.kbb)))
    return FP8BLK_ERR_CUDA;
  d.p.a = static_cast<const uint8_t*>(a);
  d.p.a_s = a_s;
  d.p.w_s = w_s;
  d.p.c = static_cast<__nv_bfloat16*>(c);
  d.p.err = dev->err_word;
  *used = true;
  return d.nt == 1 ? decode_launch<1>(dev, map, d, stream) : decode_launch<2>(dev, map, d, stream);
}

}  // namespace fp8blk
