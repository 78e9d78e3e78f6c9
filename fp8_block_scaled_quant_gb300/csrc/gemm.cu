// Block-scaled FP8 GEMM for sm_103a ("Administrator & Developer Guide", 8.5.3
// fp8_gemm_kernel, and 6.3 The FP8 path):
//
//   C[m, n] = sum_kb a_s[m, kb] * w_s[n/128, kb] * sum_{k in kb} a[m, k] w[n, k]
//
// Design (one CTA per SM, warp-specialised, persistent):
//   warp 0      TMA producer: per 128-wide K block, one 128x128 tile of the
//               "lane" operand and one BN x 128 tile of the "column" operand
//               into a STAGES-deep shared-memory ring (mbarrier full/empty).
//   warp 1      MMA issuer: four tcgen05.mma kind::f8f6f4 (K = 32 each) per K
//               block into a fresh TMEM partial (a ring of P partials of BN
//               fp32 columns), then tcgen05.commit to free the smem stage and
//               to publish the partial.
//   warps 2..   promotion / epilogue: tcgen05.ld each partial, multiply by
//               the block's a_s * w_s and add into fp32 registers (the pages'
//               acc += dot(a, b) * a_s * b_s), then bf16 stores.
//
// Operand roles. For M > 128 the activation rows are the MMA's M (TMEM lanes)
// and weight rows its N (columns), BN = 128 or 256. For decode-sized M <= 128
// the roles swap: 128 weight rows fill the MMA's M, so the weight scale is one
// number per CTA tile, and the M tokens (padded to BN = 16..128 by the TMA
// zero fill) are the columns, each with its own activation scale.
//
// Schedule. Tiles are numbered lane-tile fastest. The first dp_waves * grid
// tiles go round-robin to whole CTAs (data-parallel waves: concurrent tiles
// share column-operand tiles in L2); the rest are split stream-K: the K-block
// iterations of those tiles are divided evenly over all CTAs, and a tile cut
// between CTAs is finished by whichever of them arrives last on its counter,
// which sums the fp32 partials in part order (deterministic) and stores bf16.
//
// Every mbarrier wait is bounded (2 s): on expiry the CTA records an error bit,
// stops issuing work, waits (bounded) for its own copies and MMAs in flight,
// frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fp8blk.h"
#include "host.cuh"
#include "ptx.cuh"

namespace fp8blk {

struct GemmParams {
  const float* a_s;    // [M, Kb]
  const float* w_s;    // [n_wblocks, Kb]
  __nv_bfloat16* c;    // [M, N]
  float* slots;        // stream-K partial slots, 2 per CTA, BN * 128 floats each ([col][lane])
  int* counters;       // one arrival counter per tile (zero between calls)
  unsigned* err;       // device error word
  int M, N, Kb, n_wblocks;
  int tiles_lane, tiles_col;
  int grid;            // CTAs
  int dp_waves;        // tiles [0, dp_waves * grid) run whole, round-robin
  int sk_tiles;        // the remaining tiles run stream-K
  long long sk_iters;  // sk_tiles * Kb
  int vec_store;       // C rows 16-byte aligned and N % 8 == 0
};

namespace {

struct Unit {
  int tile, kb0, kb1, part, nparts;
};

// The sequence of work units of one CTA. Producer, MMA issuer and epilogue
// each walk it with their own copy and so agree on every unit.
struct Sched {
  const GemmParams& p;
  int c, j;
  long long it, it_end;

  __device__ Sched(const GemmParams& prm, int cta) : p(prm), c(cta), j(0) {
    it = static_cast<long long>(c) * p.sk_iters / p.grid;
    it_end = static_cast<long long>(c + 1) * p.sk_iters / p.grid;
  }
  // CTA whose stream-K range [c*S/G, (c+1)*S/G) holds iteration i. Every CTA
  // has a non-empty range because S >= G.
  __device__ long long cta_of(long long i) const { return ((i + 1) * p.grid - 1) / p.sk_iters; }

  __device__ bool next(Unit& u) {
    if (j < p.dp_waves) {
      u.tile = c + j * p.grid;
      u.kb0 = 0;
      u.kb1 = p.Kb;
      u.part = 0;
      u.nparts = 1;
      ++j;
      return true;
    }
    if (it >= it_end) return false;
    const long long t = it / p.Kb;
    const long long t_begin = t * p.Kb, t_end = t_begin + p.Kb;
    const long long seg_end = t_end < it_end ? t_end : it_end;
    const long long first = cta_of(t_begin), last = cta_of(t_end - 1);
    u.tile = p.dp_waves * p.grid + static_cast<int>(t);
    u.kb0 = static_cast<int>(it - t_begin);
    u.kb1 = static_cast<int>(seg_end - t_begin);
    u.part = c - static_cast<int>(first);
    u.nparts = static_cast<int>(last - first + 1);
    it = seg_end;
    return true;
  }
};

constexpr int pow2_at_least(int v, int floor_) {
  int p = floor_;
  while (p < v) p <<= 1;
  return p;
}

template <int BN_, bool SWAP_, int STAGES_, int P_, int EPI_WARPS_>
struct Cfg {
  static constexpr int BN = BN_;
  static constexpr bool SWAP = SWAP_;
  static constexpr int STAGES = STAGES_;
  static constexpr int P = P_;
  static constexpr int EPI_WARPS = EPI_WARPS_;
  static constexpr int kThreads = (2 + EPI_WARPS) * 32;
  static constexpr int kGroups = EPI_WARPS / 4;  // column groups in the epilogue
  static constexpr int kCpt = BN / kGroups;      // columns per epilogue thread
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = pow2_at_least(P * BN, 32);
  static constexpr int kBarBytes = (2 * STAGES + 2 * P + 2) * 8 + 16;
  static constexpr int kSmemBytes = 1024 + STAGES * kStageBytes + kBarBytes;

  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
  static_assert(EPI_WARPS % 4 == 0, "epilogue warps come in warpgroups");
  static_assert(kCpt == 16 || kCpt % 32 == 0, "TMEM loads of 16 or 32 columns");
  static_assert(SWAP || kCpt == 128, "non-swapped tiles: one weight block per column group");
  static_assert(!SWAP || kGroups == 1, "swapped tiles: one column group");
  static_assert(P * BN <= 512, "TMEM has 512 columns");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ void tile_coords(const GemmParams& p, int tile, int& tl, int& tc) {
  tl = tile % p.tiles_lane;
  tc = tile / p.tiles_lane;
}

template <class C>
__device__ __forceinline__ void store_tile(const GemmParams& p, const float (&acc)[C::kCpt], int tl, int tc, int group,
                                           int row) {
  if constexpr (!C::SWAP) {
    const int m = tl * 128 + row;
    const int n0 = tc * C::BN + group * 128;
    if (m >= p.M) return;
    __nv_bfloat16* crow = p.c + static_cast<size_t>(m) * p.N;
#pragma unroll
    for (int v = 0; v < C::kCpt / 8; ++v) {
      const int n = n0 + v * 8;
      if (p.vec_store && n + 8 <= p.N) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(acc[v * 8 + 2 * e], acc[v * 8 + 2 * e + 1]);
          w[e] = *reinterpret_cast<const uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(crow + n) = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (n + e < p.N) crow[n + e] = __float2bfloat16_rn(acc[v * 8 + e]);
      }
    }
  } else {
    const int n = tl * 128 + row;
    if (n >= p.N) return;
#pragma unroll
    for (int j = 0; j < C::kCpt; ++j) {
      const int m = tc * C::BN + j;
      if (m < p.M) p.c[static_cast<size_t>(m) * p.N + n] = __float2bfloat16_rn(acc[j]);
    }
  }
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_lane, const __grid_constant__ CUtensorMap tmap_col,
                    const GemmParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::kStageBytes);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + C::P;
  uint64_t* drain = tempty + C::P;
  uint64_t* epi_bar = drain + 1;  // epilogue-only barrier for the stream-K fixup
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int q = 0; q < C::P; ++q) {
      mbar_init(&tfull[q], 1);
      mbar_init(&tempty[q], C::EPI_WARPS);
    }
    mbar_init(drain, 1);
    mbar_init(epi_bar, C::EPI_WARPS);
    *abort_flag = 0;
    *last_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_lane);
    tma_prefetch_desc(&tmap_col);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      Sched sch(prm, blockIdx.x);
      Unit u;
      int st = 0;
      uint32_t ph = 0;
      long long issued = 0;
      bool ok = true;
      while (ok && sch.next(u)) {
        int tl, tc;
        tile_coords(prm, u.tile, tl, tc);
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, prm.err, kDevErrTimeoutProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], C::kStageBytes);
          uint8_t* sa = smem + st * C::kStageBytes;
          tma_load_2d(sa, &tmap_lane, &full[st], kb * 128, tl * 128);
          tma_load_2d(sa + C::kABytes, &tmap_col, &full[st], kb * 128, tc * C::BN);
          ++issued;
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA exits.
        const long long n = issued < C::STAGES ? issued : C::STAGES;
        for (long long i = 0; i < n; ++i) {
          const long long idx = issued - 1 - i;
          mbar_wait(&full[idx % C::STAGES], static_cast<uint32_t>((idx / C::STAGES) & 1), nullptr, prm.err,
                    kDevErrTimeoutDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_e4m3_f32(128, C::BN);
      Sched sch(prm, blockIdx.x);
      Unit u;
      int st = 0, pb = 0;
      uint32_t ph = 0, pph = 0;
      bool ok = true;
      while (ok && sch.next(u)) {
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait(&full[st], ph, abort_flag, prm.err, kDevErrTimeoutMma) ||
              !mbar_wait(&tempty[pb], pph ^ 1u, abort_flag, prm.err, kDevErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(smem + st * C::kStageBytes);
          const uint64_t ad = sdesc_kmajor_sw128(a_addr);
          const uint64_t bd = sdesc_kmajor_sw128(a_addr + C::kABytes);
          const uint32_t d = tmem_base + static_cast<uint32_t>(pb * C::BN);
#pragma unroll
          for (int k = 0; k < 4; ++k)  // 32-byte K slices: start address advances by 32 B (2 x 16 B)
            mma_e4m3(d, ad + 2 * k, bd + 2 * k, kIdesc, k > 0 ? 1u : 0u);
          mma_commit(&empty[st]);
          mma_commit(&tfull[pb]);
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1u;
          }
          if (++pb == C::P) {
            pb = 0;
            pph ^= 1u;
          }
        }
      }
      // Wait for every MMA this thread issued before TMEM is released.
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, prm.err, kDevErrTimeoutDrain);
    }
  } else {
    // ---------------- promotion + epilogue ----------------
    const int ew = warp - 2;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int group = ew >> 2;     // column group
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr int kAsRegs = (C::kCpt + 31) / 32;

    // Epilogue-wide barrier on an mbarrier (bounded wait, unlike bar.sync, so a
    // warp that gave up cannot strand the others).
    uint32_t eph = 0;
    auto epi_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(epi_bar);
      const bool r = mbar_wait(epi_bar, eph, abort_flag, prm.err, kDevErrTimeoutEpilogue);
      eph ^= 1u;
      return r;
    };

    Sched sch(prm, blockIdx.x);
    Unit u;
    int pb = 0;
    uint32_t pph = 0;
    bool ok = true;
    while (ok && sch.next(u)) {
      int tl, tc;
      tile_coords(prm, u.tile, tl, tc);
      float acc[C::kCpt];
#pragma unroll
      for (int i = 0; i < C::kCpt; ++i) acc[i] = 0.0f;

      for (int kb = u.kb0; kb < u.kb1; ++kb) {
        // Scales of this K block, loaded before the wait to hide their latency.
        float sc_row = 0.0f;
        float sc_col[kAsRegs];
        if constexpr (!C::SWAP) {
          const int m = tl * 128 + row;
          const int nb = tc * C::kGroups + group;
          const float as = (m < prm.M) ? __ldg(prm.a_s + static_cast<size_t>(m) * prm.Kb + kb) : 0.0f;
          const float ws = (nb < prm.n_wblocks) ? __ldg(prm.w_s + static_cast<size_t>(nb) * prm.Kb + kb) : 0.0f;
          sc_row = as * ws;
        } else {
          const float ws = __ldg(prm.w_s + static_cast<size_t>(tl) * prm.Kb + kb);
#pragma unroll
          for (int i = 0; i < kAsRegs; ++i) {
            const int j = lane + 32 * i;
            const int m = tc * C::BN + j;
            sc_col[i] = (j < C::kCpt && m < prm.M) ? __ldg(prm.a_s + static_cast<size_t>(m) * prm.Kb + kb) * ws
                                                   : 0.0f;
          }
        }
        if (!mbar_wait(&tfull[pb], pph, abort_flag, prm.err, kDevErrTimeoutEpilogue)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t col0 = static_cast<uint32_t>(pb * C::BN + group * C::kCpt);
        if constexpr (C::kCpt == 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(t_lane + col0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float sc = C::SWAP ? __shfl_sync(0xFFFFFFFFu, sc_col[0], i) : sc_row;
            acc[i] = fmaf(__uint_as_float(v[i]), sc, acc[i]);
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < C::kCpt / 32; ++ch) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_lane + col0 + ch * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float sc = C::SWAP ? __shfl_sync(0xFFFFFFFFu, sc_col[ch], i) : sc_row;
              acc[ch * 32 + i] = fmaf(__uint_as_float(v[i]), sc, acc[ch * 32 + i]);
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[pb]);
        if (++pb == C::P) {
          pb = 0;
          pph ^= 1u;
        }
      }
      if (!ok) break;

      if (u.nparts == 1) {
        store_tile<C>(prm, acc, tl, tc, group, row);
      } else {
        // Stream-K fixup: publish this part, count arrivals, the last part sums.
        float* mine = prm.slots + static_cast<size_t>(2 * blockIdx.x + (u.part == 0 ? 1 : 0)) * (C::BN * 128);
#pragma unroll
        for (int i = 0; i < C::kCpt; ++i) __stcg(mine + (group * C::kCpt + i) * 128 + row, acc[i]);
        __threadfence();
        if (!epi_sync()) break;
        if (ew == 0 && lane == 0) {
          __threadfence();
          const int prev = atomicAdd(prm.counters + u.tile, 1);
          *last_flag = (prev == u.nparts - 1) ? 1 : 0;
        }
        if (!epi_sync()) break;
        if (*last_flag) {
          __threadfence();
          const int first = static_cast<int>(blockIdx.x) - u.part;
#pragma unroll
          for (int i = 0; i < C::kCpt; ++i) acc[i] = 0.0f;
          for (int q = 0; q < u.nparts; ++q) {
            const float* src = prm.slots + static_cast<size_t>(2 * (first + q) + (q == 0 ? 1 : 0)) * (C::BN * 128);
#pragma unroll
            for (int i = 0; i < C::kCpt; ++i) acc[i] += __ldcg(src + (group * C::kCpt + i) * 128 + row);
          }
          store_tile<C>(prm, acc, tl, tc, group, row);
          if (ew == 0 && lane == 0) prm.counters[u.tile] = 0;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// Tensor map of an e4m3 matrix [rows, K] (row-major, K % 128 == 0) read in
// boxes of 128 bytes x box_rows rows with 128-byte swizzling; rows past the
// end read as zeros.
bool make_kmajor_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Kernel variants. Non-swapped: BN = 256 (two epilogue warpgroups) or 128.
// Swapped (decode-sized M): BN = 16..128 token columns.
using CfgN256 = Cfg<256, false, 4, 2, 8>;
using CfgN128 = Cfg<128, false, 6, 4, 4>;
using CfgS16 = Cfg<16, true, 8, 8, 4>;
using CfgS32 = Cfg<32, true, 8, 8, 4>;
using CfgS64 = Cfg<64, true, 6, 4, 4>;
using CfgS128 = Cfg<128, true, 6, 4, 4>;

struct Plan {
  int bn;
  bool swap;
  int tiles_lane, tiles_col;
  int grid, dp_waves, sk_tiles;
  long long sk_iters;
};

Plan make_plan(int64_t M, int64_t N, int64_t K, int sm_count) {
  Plan pl{};
  const int64_t Kb = K / kBlock;
  if (M <= 128) {
    pl.swap = true;
    pl.bn = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
    pl.tiles_lane = static_cast<int>((N + 127) / 128);
    pl.tiles_col = static_cast<int>((M + pl.bn - 1) / pl.bn);
  } else {
    pl.swap = false;
    pl.bn = N <= 128 ? 128 : 256;
    pl.tiles_lane = static_cast<int>((M + 127) / 128);
    pl.tiles_col = static_cast<int>((N + pl.bn - 1) / pl.bn);
  }
  const long long tiles = static_cast<long long>(pl.tiles_lane) * pl.tiles_col;
  const int G = sm_count;
  if (tiles >= 2LL * G) {
    pl.grid = G;
    pl.dp_waves = static_cast<int>(tiles / G - 1);
    pl.sk_tiles = static_cast<int>(tiles - static_cast<long long>(pl.dp_waves) * G);
  } else {
    pl.dp_waves = 0;
    pl.sk_tiles = static_cast<int>(tiles);
    const long long iters = tiles * Kb;
    pl.grid = static_cast<int>(iters < G ? iters : G);
  }
  pl.sk_iters = static_cast<long long>(pl.sk_tiles) * Kb;
  return pl;
}

size_t align256(size_t v) { return (v + 255) & ~size_t{255}; }

size_t plan_workspace(const Plan& pl) {
  const size_t tiles = static_cast<size_t>(pl.tiles_lane) * pl.tiles_col;
  return align256(tiles * sizeof(int)) + static_cast<size_t>(2) * pl.grid * pl.bn * 128 * sizeof(float);
}

int sm_count_or_default() {
  const DevInfo* d;
  return current_device(&d) == FP8BLK_OK ? d->sm_count : 256;
}

template <class C>
int launch(const DevInfo* d, const CUtensorMap& ml, const CUtensorMap& mc, const GemmParams& prm,
           cudaStream_t stream) {
  static bool attr_done[64] = {};
  auto kern = fp8_gemm_kernel<C>;
  if (d->device >= 64 || !attr_done[d->device]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return FP8BLK_ERR_CUDA;
    if (d->device < 64) attr_done[d->device] = true;
  }
  kern<<<prm.grid, C::kThreads, C::kSmemBytes, stream>>>(ml, mc, prm);
  return launch_status();
}

}  // namespace

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 256;
  return plan_workspace(make_plan(M, N, K, sm_count_or_default()));
}

int gemm_run(const void* a, const float* a_s, const void* w, const float* w_s, void* c, int64_t M, int64_t N,
             int64_t K, int scale_fmt, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (scale_fmt != FP8BLK_SCALE_FP32 && scale_fmt != FP8BLK_SCALE_UE8M0) return FP8BLK_ERR_ARG;
  if (M < 0 || N < 0 || K < 0 || K % kBlock != 0) return FP8BLK_ERR_SHAPE;
  if (M > (int64_t{1} << 31) - 1 || N > (int64_t{1} << 31) - 1 || K > (int64_t{1} << 31) - 1)
    return FP8BLK_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8BLK_OK;
  if (!c) return FP8BLK_ERR_NULL;
  if (!is_aligned(c, 2)) return FP8BLK_ERR_ALIGN;
  if (K == 0) return cuda_status(cudaMemsetAsync(c, 0, static_cast<size_t>(M) * N * 2, stream));
  if (!a || !a_s || !w || !w_s) return FP8BLK_ERR_NULL;
  if (!is_aligned(a, 16) || !is_aligned(w, 16) || !is_aligned(a_s, 4) || !is_aligned(w_s, 4))
    return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  const Plan pl = make_plan(M, N, K, d->sm_count);
  const size_t need = plan_workspace(pl);
  if (!workspace || workspace_bytes < need) return FP8BLK_ERR_WORKSPACE;
  if (!is_aligned(workspace, 256)) return FP8BLK_ERR_ALIGN;

  GemmParams prm{};
  prm.a_s = a_s;
  prm.w_s = w_s;
  prm.c = static_cast<__nv_bfloat16*>(c);
  const size_t tiles = static_cast<size_t>(pl.tiles_lane) * pl.tiles_col;
  prm.counters = static_cast<int*>(workspace);
  prm.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(tiles * sizeof(int)));
  prm.err = d->err_word;
  prm.M = static_cast<int>(M);
  prm.N = static_cast<int>(N);
  prm.Kb = static_cast<int>(K / kBlock);
  prm.n_wblocks = static_cast<int>((N + 127) / 128);
  prm.tiles_lane = pl.tiles_lane;
  prm.tiles_col = pl.tiles_col;
  prm.grid = pl.grid;
  prm.dp_waves = pl.dp_waves;
  prm.sk_tiles = pl.sk_tiles;
  prm.sk_iters = pl.sk_iters;
  prm.vec_store = (N % 8 == 0 && is_aligned(c, 16)) ? 1 : 0;

  CUtensorMap ml, mc;
  const void* lane_src = pl.swap ? w : a;
  const void* col_src = pl.swap ? a : w;
  const uint64_t lane_rows = static_cast<uint64_t>(pl.swap ? N : M);
  const uint64_t col_rows = static_cast<uint64_t>(pl.swap ? M : N);
  if (!make_kmajor_map(&ml, lane_src, lane_rows, static_cast<uint64_t>(K), 128) ||
      !make_kmajor_map(&mc, col_src, col_rows, static_cast<uint64_t>(K), static_cast<uint32_t>(pl.bn)))
    return FP8BLK_ERR_CUDA;

  if (!pl.swap) {
    if (pl.bn == 256) return launch<CfgN256>(d, ml, mc, prm, stream);
    return launch<CfgN128>(d, ml, mc, prm, stream);
  }
  switch (pl.bn) {
    case 16: return launch<CfgS16>(d, ml, mc, prm, stream);
    case 32: return launch<CfgS32>(d, ml, mc, prm, stream);
    case 64: return launch<CfgS64>(d, ml, mc, prm, stream);
    default: return launch<CfgS128>(d, ml, mc, prm, stream);
  }
}

}  // namespace fp8blk

// ---------------------------------------------------------------------------
// fp8blk_gemm_noalloc: the GEMM with library-held scratch, for callers that
// cannot allocate device memory (see include/fp8blk.h). The scratch is a
// file-scope device array: every GPU that loads the library holds it until
// the process exits. Host code must not use the array's name as an address;
// the device address comes from cudaGetSymbolAddress, once per device.
// ---------------------------------------------------------------------------
namespace fp8blk {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FP8BLK_NOALLOC_SCRATCH_BYTES];

namespace {

struct NoAllocDevice {
  std::once_flag once;
  void* ptr;
  int status;
};
NoAllocDevice g_noalloc_dev[64];

// Device address of g_noalloc_scratch on device `dev` (which is current).
int noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= 64) return FP8BLK_ERR_CUDA;
  NoAllocDevice& nd = g_noalloc_dev[dev];
  std::call_once(nd.once, [&nd] {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    nd.ptr = p;
    nd.status = (e == cudaSuccess && p != nullptr) ? FP8BLK_OK : FP8BLK_ERR_CUDA;
  });
  *out = nd.ptr;
  return nd.status;
}

// Bytes at the start of a plan's workspace that hold the tile counters.
size_t plan_counter_bytes(const Plan& pl) {
  return align256(static_cast<size_t>(pl.tiles_lane) * pl.tiles_col * sizeof(int));
}

}  // namespace
}  // namespace fp8blk

extern "C" int fp8blk_gemm_noalloc(const void* a_e4m3, const float* a_s, const void* w_e4m3, const float* w_s,
                                   void* c_bf16, int64_t M, int64_t N, int64_t K, int scale_fmt,
                                   fp8blk_stream_t stream) {
  using namespace fp8blk;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int64_t lim = (int64_t{1} << 31) - 1;
  if (M > 0 && N > 0 && K > 0 && K % kBlock == 0 && M <= lim && N <= lim && K <= lim) {
    const DevInfo* d;
    if (int st = current_device(&d)) return st;
    const Plan pl = make_plan(M, N, K, d->sm_count);
    if (plan_workspace(pl) > FP8BLK_NOALLOC_SCRATCH_BYTES) return FP8BLK_ERR_TOO_LARGE;
    void* scratch = nullptr;
    if (int st = noalloc_scratch(d->device, &scratch)) return st;
    if (cudaMemsetAsync(scratch, 0, plan_counter_bytes(pl), cs) != cudaSuccess) return FP8BLK_ERR_CUDA;
    return gemm_run(a_e4m3, a_s, w_e4m3, w_s, c_bf16, M, N, K, scale_fmt, scratch, FP8BLK_NOALLOC_SCRATCH_BYTES, cs);
  }
  // Empty, zero-K and invalid problems need no scratch: same answers as fp8blk_gemm.
  return gemm_run(a_e4m3, a_s, w_e4m3, w_s, c_bf16, M, N, K, scale_fmt, nullptr, 0, cs);
}

extern "C" size_t fp8blk_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return fp8blk::gemm_workspace_bytes(M, N, K);
}

extern "C" int fp8blk_gemm(const void* a_e4m3, const float* a_s, const void* w_e4m3, const float* w_s, void* c_bf16,
                           int64_t M, int64_t N, int64_t K, int scale_fmt, void* workspace, size_t workspace_bytes,
                           fp8blk_stream_t stream) {
  return fp8blk::gemm_run(a_e4m3, a_s, w_e4m3, w_s, c_bf16, M, N, K, scale_fmt, workspace, workspace_bytes,
                          reinterpret_cast<cudaStream_t>(stream));
}
