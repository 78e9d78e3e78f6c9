// Decode-sized block-scaled FP8 GEMM on weight slices ("Administrator &
// Developer Guide", 8.5.3 fp8_gemm_kernel and 6.3 The FP8 path):
//
//   C[m, n] = sum_kb a_s[m, kb] * w_s[n/128, kb] * sum_{k in kb} a[m, k] w[n, k]
//
// for M <= 64 tokens, where the layer is bound by streaming the weight. One
// CTA per SM takes an equal slice of R weight rows (R a multiple of 8, at most
// 128) over all of K, so no SM idles and no partial sums leave the CTA.
//
// What bounds a chain of dependent decode launches is the part of each launch
// that runs after its dependency wait. So the weight slice moves in as few
// TMA boxes as possible -- 3-D boxes whose third dimension is the K block, G
// K blocks (up to all of K) per box -- and those boxes are requested before
// the wait (weights never depend on the previous kernel). After the wait come
// only the activation boxes (same G K blocks of the M tokens), the MMAs and the
// promotion. Measured on the decode layer (N = 10944, K = 2048): 16 boxes of
// one K block per CTA run a dependent chain at ~6.3 us per launch, one or two
// large boxes at ~3.8 us (a TMA-only stream).
//
// Roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: a ring of `stages` stages, each one weight box
//               [G K blocks][R rows][128 B] and one activation box
//               [G][BN tokens][128 B] (rows past M zero-filled), 128-byte
//               swizzled like 2-D tiles; the weight boxes of the first
//               `stages` stages before griddepcontrol.wait.
//   warp 1      MMA issuer: per K block four tcgen05.mma kind::f8f6f4
//               (M = 128: the R slice rows, lanes past R compute values nobody
//               reads; N = BN tokens; K = 32 each) into a fresh TMEM partial
//               (a ring of P partials of BN fp32 columns).
//   warps 2-5   promotion and epilogue: thread = TMEM lane = slice row;
//               acc[j] += partial[j] * (a_s[j, kb] * w_s[row block, kb]) in
//               fp32 per K block (the pages' acc += dot(a, b) * a_s * b_s),
//               scales staged once in shared memory; bf16 stores.
//
// Every mbarrier wait is bounded; on expiry the CTA records an error bit,
// drains its own copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8blk.h"
#include "host.cuh"
#include "ptx.cuh"

namespace fp8blk {

namespace {

constexpr int kDecThreads = 192;
constexpr int kDecEpiWarp0 = 2;
constexpr int kDecMaxStages = 4;
// Bytes past the ring that the 128-row MMA read of the last stage's last
// weight tile may reach (lanes past the slice), beyond that stage's
// activation tiles.
__host__ __device__ constexpr int dec_pad(int rows, int BN, int G) {
  return (128 - rows) * 128 > BN * 128 * G ? (128 - rows) * 128 - BN * 128 * G : 0;
}

// Stage split limits (tuning): at most FP8BLK_DECODE_MAX_G K blocks per box,
// and at least FP8BLK_DECODE_MIN_STAGES stages when K allows.
#ifndef FP8BLK_DECODE_MAX_G
#define FP8BLK_DECODE_MAX_G 256
#endif
#ifndef FP8BLK_DECODE_MIN_STAGES
#define FP8BLK_DECODE_MIN_STAGES 1
#endif
// Shared memory the decode kernel may use per CTA (bytes; 0: all the device offers).
#ifndef FP8BLK_DECODE_SMEM
#define FP8BLK_DECODE_SMEM 0
#endif

// Optional phase trace (compile with -DFP8BLK_TRACE): %globaltimer stamps per
// CTA, read back with fp8trace_decode_read(). Default builds contain none.
#ifdef FP8BLK_TRACE
__device__ unsigned long long g_dec_trace[8 * 1024 * 16];
#define DEC_STAMP(slot)                                                                                 \
  do {                                                                                                  \
    if (blockIdx.x < 1024) g_dec_trace[((p.trace_id & 7) * 1024 + blockIdx.x) * 16 + (slot)] = global_timer_ns(); \
  } while (0)
#else
#define DEC_STAMP(slot) do { } while (0)
#endif

struct DecodeParams {
  const float* a_s;    // [M, Kb]
  const float* w_s;    // [ceil(N / 128), Kb]
  __nv_bfloat16* c;    // [M, N]
  unsigned* err;       // device error word
  int M, N, Kb, n_wblocks;
  int rows;            // weight rows per slice (multiple of 8, <= 128)
  int G;               // K blocks per stage
  int stages;          // stages in the ring (<= kDecMaxStages)
  int stage_bytes;     // (rows + BN) * 128 * G, a multiple of 1024
  int trace_id;        // phase-trace builds only
};

// Each 32-wide K slice of a K block goes to its own TMEM accumulator (S
// slices per partial): the four MMAs of a K block then do not wait on one
// another's result, and the epilogue adds the four in fp32 before scaling
// (the same sum in another order).
#ifndef FP8BLK_DECODE_SPLIT
#define FP8BLK_DECODE_SPLIT 1
#endif
template <int BN>
struct DecCfg {
  static constexpr int S = FP8BLK_DECODE_SPLIT ? 4 : 1;  // accumulators per K block
  static constexpr int P = 512 / (S * BN) < 8 ? 512 / (S * BN) : 8;  // TMEM partials (K blocks in flight)
  static constexpr int kCols = S * BN;                                // TMEM columns per partial
  static constexpr int kTmemCols = P * kCols < 32 ? 32 : P * kCols;
  static_assert(P >= 2 && P * kCols <= 512, "TMEM has 512 columns");
};

__host__ __device__ constexpr size_t dec_scale_bytes(int Kb, int BN) {
  return ((static_cast<size_t>(Kb) * BN + 2 * static_cast<size_t>(Kb)) * 4 + 15) & ~size_t{15};
}

__host__ __device__ constexpr size_t dec_bar_bytes(int P) { return (2 * kDecMaxStages + 2 * P + 1) * 8 + 16; }

template <int BN>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                       const DecodeParams p) {
  using C = DecCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  float* as_sm = reinterpret_cast<float*>(ring + static_cast<size_t>(p.stages) * p.stage_bytes +
                                          ((dec_pad(p.rows, BN, p.G) + 15) & ~15));  // [Kb][BN]
  float* ws_sm = as_sm + static_cast<size_t>(p.Kb) * BN;  // [2][Kb]: the slice's (at most two) weight blocks
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(as_sm) + dec_scale_bytes(p.Kb, BN));
  uint64_t* empty = full + kDecMaxStages;
  uint64_t* tfull = empty + kDecMaxStages;
  uint64_t* tempty = tfull + C::P;
  uint64_t* drain = tempty + C::P;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The next kernel on the stream may start its prologue (and its weight
  // loads); it touches nothing this one writes before its own wait.
  griddep_launch_dependents();
  if (threadIdx.x == 0) DEC_STAMP(0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int q = 0; q < C::P; ++q) {
      mbar_init(&tfull[q], 1);
      mbar_init(&tempty[q], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_a);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const int r0 = static_cast<int>(blockIdx.x) * p.rows;
  const int nst = (p.Kb + p.G - 1) / p.G;  // stages' worth of K blocks in the slice
  const uint32_t w_bytes = static_cast<uint32_t>(p.rows) * 128u * p.G;
  const uint32_t a_bytes = static_cast<uint32_t>(BN) * 128u * p.G;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const int npre = nst < p.stages ? nst : p.stages;
      for (int s = 0; s < npre; ++s) {  // weights first: they do not depend on the previous kernel
        mbar_arrive_expect_tx(&full[s], w_bytes + a_bytes);
        tma_load_3d(ring + static_cast<size_t>(s) * p.stage_bytes, &tmap_w, &full[s], 0, r0, s * p.G);
      }
      DEC_STAMP(1);
      griddep_wait();
      DEC_STAMP(2);
      for (int s = 0; s < npre; ++s)
        tma_load_3d(ring + static_cast<size_t>(s) * p.stage_bytes + w_bytes, &tmap_a, &full[s], 0, 0, s * p.G);
      int issued = npre;
      bool ok = true;
      for (; issued < nst; ++issued) {
        const int slot = issued % p.stages;
        const uint32_t ph = static_cast<uint32_t>((issued / p.stages - 1) & 1);
        if (!mbar_wait(&empty[slot], ph, abort_flag, p.err, kDevErrTimeoutProducer)) {
          ok = false;
          break;
        }
        uint8_t* st = ring + static_cast<size_t>(slot) * p.stage_bytes;
        mbar_arrive_expect_tx(&full[slot], w_bytes + a_bytes);
        tma_load_3d(st, &tmap_w, &full[slot], 0, r0, issued * p.G);
        tma_load_3d(st + w_bytes, &tmap_a, &full[slot], 0, 0, issued * p.G);
      }
      if (!ok) {  // let the copies already issued land before the CTA exits
        const int first = issued - p.stages < 0 ? 0 : issued - p.stages;
        for (int i = first; i < issued; ++i)
          mbar_wait(&full[i % p.stages], static_cast<uint32_t>((i / p.stages) & 1), nullptr, p.err,
                    kDevErrTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    const bool leader = elect_one_sync();
    constexpr uint32_t kIdesc = idesc_e4m3_f32(128, BN);
    int pb = 0;
    uint32_t pph = 0;
    bool ok = true;
    for (int i = 0; ok && i < nst; ++i) {
      const int slot = i % p.stages;
      if (!__all_sync(0xFFFFFFFFu,
                      mbar_wait(&full[slot], static_cast<uint32_t>((i / p.stages) & 1), abort_flag, p.err,
                                kDevErrTimeoutMma))) {
        ok = false;
        break;
      }
      if (leader && i == 0) DEC_STAMP(3);
      if (leader && i == nst - 1) DEC_STAMP(4);
      const uint32_t st = smem_u32(ring + static_cast<size_t>(slot) * p.stage_bytes);
      for (int g = 0; g < p.G && i * p.G + g < p.Kb; ++g) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tempty[pb], pph ^ 1u, abort_flag, p.err, kDevErrTimeoutMma))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint64_t ad = sdesc_kmajor_sw128(st + static_cast<uint32_t>(g * p.rows * 128));
        const uint64_t bd = sdesc_kmajor_sw128(st + w_bytes + static_cast<uint32_t>(g * BN * 128));
        const uint32_t d = tmem_base + static_cast<uint32_t>(pb * C::kCols);
        if (leader) {
#pragma unroll
          for (int k = 0; k < 4; ++k)  // 32-byte K slices: the start address advances by 32 B
            if constexpr (C::S == 4) mma_e4m3(d + static_cast<uint32_t>(k * BN), ad + 2 * k, bd + 2 * k, kIdesc, 0u);
            else mma_e4m3(d, ad + 2 * k, bd + 2 * k, kIdesc, k > 0 ? 1u : 0u);
          mma_commit(&tfull[pb]);
        }
        __syncwarp();
        if (++pb == C::P) {
          pb = 0;
          pph ^= 1u;
        }
      }
      if (leader) mma_commit(&empty[slot]);  // the stage's MMAs done: its smem may be refilled
      __syncwarp();
    }
    if (leader) {  // every MMA issued has completed before TMEM is released
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, p.err, kDevErrTimeoutDrain);
    }
    __syncwarp();
  } else {
    // ---------------- promotion + epilogue ----------------
    const int et = static_cast<int>(threadIdx.x) - kDecEpiWarp0 * 32;  // 0 .. 127
    const int quarter = warp & 3;                                     // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const int blk0 = r0 >> 7;
    griddep_wait();  // activation scales and the output belong to the previous kernel until now
    // Scales of the whole slice: activation scales [Kb][BN] (zero past M),
    // the slice's weight-block scales [2][Kb] (zero past the last block).
    for (int i = et; i < p.Kb * BN; i += 128) {
      const int j = i / p.Kb, kb = i - j * p.Kb;
      as_sm[kb * BN + j] = j < p.M ? __ldg(p.a_s + static_cast<size_t>(j) * p.Kb + kb) : 0.0f;
    }
    for (int i = et; i < 2 * p.Kb; i += 128) {
      const int b = i / p.Kb, kb = i - b * p.Kb;
      ws_sm[i] = blk0 + b < p.n_wblocks ? __ldg(p.w_s + static_cast<size_t>(blk0 + b) * p.Kb + kb) : 0.0f;
    }
    named_barrier_sync(1, 128);
    if (et == 0) DEC_STAMP(5);
    const int n = r0 + row;
    const bool valid = row < p.rows && n < p.N;
    const float* wsr = ws_sm + (valid ? ((n >> 7) - blk0) : 0) * p.Kb;
    float acc[BN];
#pragma unroll
    for (int j = 0; j < BN; ++j) acc[j] = 0.0f;
    int pb = 0;
    uint32_t pph = 0;
    bool ok = true;
    for (int kb = 0; kb < p.Kb; ++kb) {
      const float w = wsr[kb];
      const float* as_kb = as_sm + kb * BN;
      if (!mbar_wait(&tfull[pb], pph, abort_flag, p.err, kDevErrTimeoutEpilogue)) {
        ok = false;
        break;
      }
      if (et == 0 && kb == 0) DEC_STAMP(6);
      tc_fence_after_sync();
      const uint32_t ta = t_lane + static_cast<uint32_t>(pb * C::kCols);
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float sum[16];
        if constexpr (C::S == 4 && BN == 16) {
          // the four K-slice accumulators (columns k * 16 + j), one load, added in fp32
          uint32_t v[64];
          tmem_ld_32x32b_x64(ta, v);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            sum[j] = (__uint_as_float(v[j]) + __uint_as_float(v[16 + j])) +
                     (__uint_as_float(v[32 + j]) + __uint_as_float(v[48 + j]));
        } else if constexpr (C::S == 4) {
          // the four K-slice accumulators of these 16 columns, added in fp32
          uint32_t v0[16], v1[16], v2[16], v3[16];
          tmem_ld_32x32b_x16(ta + static_cast<uint32_t>(c0), v0);
          tmem_ld_32x32b_x16(ta + static_cast<uint32_t>(BN + c0), v1);
          tmem_ld_32x32b_x16(ta + static_cast<uint32_t>(2 * BN + c0), v2);
          tmem_ld_32x32b_x16(ta + static_cast<uint32_t>(3 * BN + c0), v3);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            sum[j] = (__uint_as_float(v0[j]) + __uint_as_float(v1[j])) + (__uint_as_float(v2[j]) + __uint_as_float(v3[j]));
        } else {
          uint32_t v[16];
          tmem_ld_32x32b_x16(ta + static_cast<uint32_t>(c0), v);
#pragma unroll
          for (int j = 0; j < 16; ++j) sum[j] = __uint_as_float(v[j]);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[c0 + j] = fmaf(sum[j], as_kb[c0 + j] * w, acc[c0 + j]);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[pb]);
      if (++pb == C::P) {
        pb = 0;
        pph ^= 1u;
      }
    }
    if (et == 0) DEC_STAMP(7);
    if (ok && valid) {
#pragma unroll
      for (int j = 0; j < BN; ++j)
        if (j < p.M) p.c[static_cast<size_t>(j) * p.N + n] = __float2bfloat16_rn(acc[j]);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
  if (threadIdx.x == 0) DEC_STAMP(8);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 3-D view of a K-major e4m3 matrix [rows, K]: (128-byte K slice, row, K
// block), boxes of 128 B x box_rows x G, 128-byte swizzled; rows and K blocks
// past the matrix read as zeros.
bool make_kblock_map(EncodeTiledFn enc, CUtensorMap* map, const void* base, uint64_t rows, uint64_t K,
                     uint32_t box_rows, uint32_t G) {
  const cuuint64_t dims[3] = {128, rows, K / 128};
  const cuuint64_t strides[2] = {K, 128};
  const cuuint32_t box[3] = {128, box_rows, G};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
int decode_launch(const DevInfo* d, const CUtensorMap& mw, const CUtensorMap& ma, const DecodeParams& prm,
                  size_t smem, int grid, cudaStream_t stream) {
  auto kern = decode_gemm_kernel<BN>;
  static bool attr_done[64] = {};
  if (d->device >= 64 || !attr_done[d->device]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, d->smem_optin) != cudaSuccess)
      return FP8BLK_ERR_CUDA;
    if (d->device < 64) attr_done[d->device] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, mw, ma, prm));
}

}  // namespace

namespace {

// K blocks per stage and stages for slices of `rows` rows and BN tokens
// within `budget` bytes of stages: the fewest boxes -- all of K in one stage
// if it fits, else the largest G that leaves two or more stages.
bool decode_stages(int rows, int BN, int Kb, size_t budget, int* G, int* stages, int* stage_bytes) {
  const int gmax = Kb < FP8BLK_DECODE_MAX_G ? Kb : FP8BLK_DECODE_MAX_G;
  for (int g = gmax < 256 ? gmax : 256; g >= 1; g = g > 8 ? 8 : g / 2) {
    const size_t sb = static_cast<size_t>(rows + BN) * 128 * g;
    const int nst = (Kb + g - 1) / g;
    if (nst < FP8BLK_DECODE_MIN_STAGES && g > 1) continue;
    int fit = static_cast<int>(budget / sb);
    if (fit > kDecMaxStages) fit = kDecMaxStages;
    if (fit > nst) fit = nst;
    if (fit >= 2 || (fit >= 1 && nst == 1)) {
      *G = g;
      *stages = fit;
      *stage_bytes = static_cast<int>(sb);
      return true;
    }
    if (g == 1) break;
  }
  return false;
}

struct DecodeLayout {
  int rows, BN, G, stages, stage_bytes;
  size_t smem;
};

// The slice layout of a decode GEMM, or false when slices do not apply: M
// above 64, slices (N / SMs rounded up to whole 8-row swizzle atoms) beyond
// one MMA's 128 rows or below 48 rows (128-row tiles split over K serve
// better), or stages that do not fit `smem_optin` bytes.
bool decode_layout(int64_t M, int64_t N, int64_t K, int sm_count, int smem_optin, DecodeLayout* L) {
  if (M < 1 || M > 64 || N < 1 || K < kBlock || K % kBlock || sm_count < 1) return false;
  const int64_t rows = ((N + sm_count - 1) / sm_count + 7) / 8 * 8;
  if (rows < 48 || rows > 128) return false;
  const int Kb = static_cast<int>(K / kBlock);
  L->rows = static_cast<int>(rows);
  L->BN = M <= 16 ? 16 : M <= 32 ? 32 : 64;
  if (FP8BLK_DECODE_SMEM > 0 && FP8BLK_DECODE_SMEM < smem_optin) smem_optin = FP8BLK_DECODE_SMEM;
  // The pad is at most 15 KB (rows >= 48); budget for it, then size it for the chosen split.
  const int P = L->BN == 16 ? DecCfg<16>::P : L->BN == 32 ? DecCfg<32>::P : DecCfg<64>::P;
  const size_t fixed = 1024 + dec_scale_bytes(Kb, L->BN) + dec_bar_bytes(P);
  const size_t pad_max = static_cast<size_t>(dec_pad(L->rows, 0, 1) + 15) & ~size_t{15};
  if (static_cast<size_t>(smem_optin) <= fixed + pad_max) return false;
  if (!decode_stages(L->rows, L->BN, Kb, smem_optin - fixed - pad_max, &L->G, &L->stages, &L->stage_bytes))
    return false;
  L->smem = fixed + ((static_cast<size_t>(dec_pad(L->rows, L->BN, L->G)) + 15) & ~size_t{15}) +
            static_cast<size_t>(L->stages) * L->stage_bytes;
  return true;
}

}  // namespace

// Weight rows per slice for a decode GEMM on `sm_count` SMs (0: no slices).
int decode_slice_rows(int64_t M, int64_t N, int64_t K, int sm_count, int smem_optin) {
  DecodeLayout L;
  return decode_layout(M, N, K, sm_count, smem_optin, &L) ? L.rows : 0;
}

// Decode GEMM on weight slices (rows from decode_slice_rows on this device).
// Arguments are checked by the caller (gemm_run). Sets *used = false,
// launching nothing, when the shape takes no slices here.
int decode_gemm_run(const void* a, const float* a_s, const void* w, const float* w_s, void* c, int64_t M, int64_t N,
                    int64_t K, int rows, cudaStream_t stream, bool* used) {
  *used = false;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  DecodeLayout L;
  if (!decode_layout(M, N, K, d->sm_count, d->smem_optin, &L) || L.rows != rows) return FP8BLK_OK;
  const int BN = L.BN, G = L.G, stages = L.stages, stage_bytes = L.stage_bytes;
  const int Kb = static_cast<int>(K / kBlock);
  static EncodeTiledFn enc = nullptr;
  if (!enc) {
    void* fp = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return FP8BLK_ERR_CUDA;
    enc = reinterpret_cast<EncodeTiledFn>(fp);
  }
  CUtensorMap mw, ma;
  if (!make_kblock_map(enc, &mw, w, static_cast<uint64_t>(N), static_cast<uint64_t>(K), static_cast<uint32_t>(rows),
                       static_cast<uint32_t>(G)) ||
      !make_kblock_map(enc, &ma, a, static_cast<uint64_t>(M), static_cast<uint64_t>(K), static_cast<uint32_t>(BN),
                       static_cast<uint32_t>(G)))
    return FP8BLK_ERR_CUDA;
  DecodeParams prm{};
  prm.a_s = a_s;
  prm.w_s = w_s;
  prm.c = static_cast<__nv_bfloat16*>(c);
  prm.err = d->err_word;
  prm.M = static_cast<int>(M);
  prm.N = static_cast<int>(N);
  prm.Kb = Kb;
  prm.n_wblocks = static_cast<int>((N + 127) / 128);
  prm.rows = rows;
  prm.G = G;
  prm.stages = stages;
  prm.stage_bytes = stage_bytes;
#ifdef FP8BLK_TRACE
  static int trace_counter = 0;
  prm.trace_id = trace_counter++ & 7;
#endif
  const size_t smem = L.smem;
  const int grid = static_cast<int>((N + rows - 1) / rows);
  *used = true;
  switch (BN) {
    case 16: return decode_launch<16>(d, mw, ma, prm, smem, grid, stream);
    case 32: return decode_launch<32>(d, mw, ma, prm, smem, grid, stream);
    default: return decode_launch<64>(d, mw, ma, prm, smem, grid, stream);
  }
}

}  // namespace fp8blk

#ifdef FP8BLK_TRACE
extern "C" __attribute__((visibility("default"))) int fp8trace_decode_read(unsigned long long* host, int n) {
  return cudaMemcpyFromSymbol(host, fp8blk::g_dec_trace, sizeof(unsigned long long) * n) == cudaSuccess ? 0 : 1;
}
extern "C" __attribute__((visibility("default"))) int fp8trace_decode_clear(void) {
  static unsigned long long zeros[8 * 1024 * 16];
  return cudaMemcpyToSymbol(fp8blk::g_dec_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : 1;
}
#endif
