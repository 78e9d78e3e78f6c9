// Block-scaled FP8 GEMM for sm_103a ("Administrator & Developer Guide", 8.5.3
// fp8_gemm_kernel, and 6.3 The FP8 path):
//
//   C[m, n] = sum_kb a_s[m, kb] * w_s[n/128, kb] * sum_{k in kb} a[m, k] w[n, k]
//
// Design (persistent, warp-specialised CTAs):
//   warp 0      TMA producer: per 128-wide K block, one 128x128 tile of the
//               "lane" operand and one BN x 128 tile of the "column" operand
//               into a STAGES-deep shared-memory ring (mbarrier full/empty);
//               the first STAGES weight tiles are requested before the
//               programmatic-dependent-launch wait.
//   warp 1      MMA issuer: the whole warp walks the schedule and waits; one
//               elected lane issues four tcgen05.mma kind::f8f6f4 (K = 32
//               each) per K block into a fresh TMEM partial (a ring of P
//               partials of BN fp32 columns), then tcgen05.commit to free the
//               smem stage and to publish the partial.
//   epilogue    promotion: tcgen05.ld each partial, multiply by the block's
//   warps       a_s * w_s and add into fp32 registers (the pages'
//               acc += dot(a, b) * a_s * b_s); at the end of a tile bf16
//               stores (dense large-M tiles: through a swizzled shared-memory
//               slab per warp and TMA boxes), or the SwiGLU + act_quant
//               epilogue, or rows scattered to slots (both through per-warp
//               slabs, eight rows per store instruction).
//   Large-M tiles (BN = 256, two column groups) run 12 warps: warps 0-3 give
//   registers to the two epilogue warpgroups (setmaxnreg 56 / 224).
//
// Operand roles. For M > 128 the activation rows are the MMA's M (TMEM lanes)
// and weight rows its N (columns), BN = 128 or 256. For decode-sized M <= 128
// the roles swap: 128 weight rows fill the MMA's M, so the weight scale is one
// number per CTA tile, and the M tokens (padded to BN = 16..128 by the TMA
// zero fill) are the columns, each with its own activation scale.
//
// Schedules (all deterministic).
//   - Large M, BN = 256: CTA pairs in clusters of 2 over adjacent 128-row lane
//     tiles; each CTA loads its own lane tile and one half of the weight tile,
//     multicast into both CTAs.
//   - Decode with at least SMs/2 weight tiles: whole tiles, one CTA per tile
//     up to one per SM, round-robin beyond.
//   - Decode with fewer tiles: split-K clusters of 2, 4 or 8 CTAs per tile,
//     partials reduced in rank order through distributed shared memory.
//   - Large M (and the pairs): tiles numbered lane-tile fastest (concurrent
//     tiles share column-operand tiles in L2), whole tiles round-robin over the
//     workers unless splitting K would shorten the busiest worker by more than
//     kStreamKSlackKb K blocks. Then the first dp_waves * workers tiles go
//     round-robin to whole workers and the rest are split stream-K: a tile cut
//     between workers is finished by whichever of them arrives last on its
//     counter, summing the fp32 partials in part order and storing bf16.
//     Small decode problems without split-K clusters take the same waves +
//     stream-K.
//   - Grouped (MoE) tiles: (group, column tile, 128-row tile), whole tiles
//     round-robin.
//
// Every mbarrier wait is bounded (2 s): on expiry the CTA records an error bit,
// stops issuing work, waits (bounded) for its own copies and MMAs in flight,
// frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "fp8blk.h"
#include "host.cuh"
#include "ptx.cuh"
#include "quotient.cuh"

namespace fp8blk {

// Epilogue modes.
enum : int {
  kEpiBf16 = 0,     // C[row, col] = bf16(acc)
  kEpiSwiGLU = 1,   // u = bf16(bf16(silu(bf16(h1))) * bf16(h3)), then act_quant of u -> e4m3 + scale
  kEpiScatter = 2,  // C[perm[row], col] = bf16(acc)
};

// Most grouped-GEMM groups (experts) the kernels take.
constexpr int kMaxGroups = 1024;

struct GemmParams {
  const float* a_s;    // [rows, Kb]
  const float* w_s;    // [weight blocks, Kb] (w1's scales in SwiGLU mode)
  const float* w3_s;   // SwiGLU: w3's scales
  __nv_bfloat16* c;    // bf16 output, row stride ldc
  uint8_t* uq;         // SwiGLU: e4m3 output, row stride ldc
  float* us;           // SwiGLU: scales of uq, row stride ldc / 128
  const int* perm;     // scatter: output row of every input row
  const int* grp_rows;    // grouped: first row of each group, [E + 1]
  const int* grp_mtiles;  // grouped: cumulative 128-row tiles of the groups, [E + 1]
  float* slots;        // stream-K partial slots, 2 per CTA, BN * 128 floats each ([col][lane])
  int* counters;       // one arrival counter per tile (zero between calls)
  unsigned* err;       // device error word
  int M;               // rows of the activation operand
  int N;               // output columns (grouped: per group)
  int Kb, n_wblocks;   // K / 128; weight row blocks (dense)
  int ldc;             // row stride of the output
  int E;               // grouped: number of groups; 0 for a dense GEMM
  int tiles_lane, tiles_col;
  int grid;            // CTAs
  int dp_waves;        // tiles [0, dp_waves * grid) run whole, round-robin
  int sk_tiles;        // the remaining tiles run stream-K
  long long sk_iters;  // sk_tiles * Kb
  int vec_store;       // C rows 16-byte aligned and N % 8 == 0
  int tma_store;       // kTmaStore tiles: C written by TMA through tmap_col2
  int vec_scales;      // Kb % 4 == 0 and the scale arrays 16-byte aligned: scales load four K blocks at a time
  int ue8m0;           // power-of-two scales for a fused act_quant (SwiGLU output, decode input)
  int whole_tiles;     // > 0: that many whole tiles, round-robin over the CTAs (no stream-K)
  int ksplit;          // > 1: clusters of ksplit CTAs share one tile, each a K slice, reduced in DSMEM
  const __nv_bfloat16* x;  // fused decode linear: the bf16 activation [M, Kb * 128]
  int trace_id;        // phase-trace builds only: which of 8 trace slots this launch fills
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
  int grouped_total;  // grouped GEMM: tile count read on the device (-1: dense)
  int krank;          // split-K clusters: this CTA's K slice

  __device__ Sched(const GemmParams& prm, int cta, int grouped_tiles = -1, int k_rank = 0)
      : p(prm), c(cta), j(0), grouped_total(grouped_tiles >= 0 ? grouped_tiles
                                                               : (prm.whole_tiles > 0 ? prm.whole_tiles : -1)),
        krank(k_rank) {
    it = static_cast<long long>(c) * p.sk_iters / p.grid;
    it_end = static_cast<long long>(c + 1) * p.sk_iters / p.grid;
  }
  // CTA whose stream-K range [c*S/G, (c+1)*S/G) holds iteration i. Every CTA
  // has a non-empty range because S >= G.
  __device__ long long cta_of(long long i) const { return ((i + 1) * p.grid - 1) / p.sk_iters; }

  __device__ bool next(Unit& u) {
    if (p.ksplit > 1) {  // split-K cluster: one tile per cluster, K slice `krank` of it
      if (j > 0) return false;
      u.tile = c;
      u.kb0 = static_cast<int>(static_cast<long long>(krank) * p.Kb / p.ksplit);
      u.kb1 = static_cast<int>(static_cast<long long>(krank + 1) * p.Kb / p.ksplit);
      u.part = 0;
      u.nparts = 1;
      ++j;
      return true;
    }
    if (grouped_total >= 0) {  // grouped: whole tiles, round-robin
      const long long t = c + static_cast<long long>(j) * p.grid;
      if (t >= grouped_total) return false;
      u.tile = static_cast<int>(t);
      u.kb0 = 0;
      u.kb1 = p.Kb;
      u.part = 0;
      u.nparts = 1;
      ++j;
      return true;
    }
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

// Plain (bf16-output, dense) non-swapped tiles: K blocks of scales per vector
// load in the promotion (1: one K block at a time, kAhead blocks ahead). The
// SwiGLU, scatter and grouped epilogues keep one K block at a time: their
// extra registers spill. Measured on the prefill GEMMs (4096 x 18432 x 7168,
// 4096 x 7168 x 18432): 519 / 508 us with 1, 506 / 496 us with 4.
#ifndef FP8BLK_SCALE_VEC
#define FP8BLK_SCALE_VEC 4
#endif

// TMEM columns per load (and per wait) in the register-split epilogue.

#ifndef FP8BLK_SPLIT_LD
#define FP8BLK_SPLIT_LD 64
#endif

template <int BN_, bool SWAP_, int STAGES_, int P_, int EPI_WARPS_, int MODE_ = kEpiBf16, bool GROUPED_ = false,
          bool FUSED_ = false, int CLUSTER_ = 1, bool MX_ = false>
struct Cfg {
  // MX: power-of-two (UE8M0) scales applied by the tensor core itself
  // (tcgen05.mma kind::mxf8f6f4.block_scale). The scale of a K block is the
  // same number for every 32-element MMA slice in it, so one UE8M0 scale per
  // operand row and slice gives exactly a_s * w_s * partial, and the fp32
  // accumulator stays in TMEM over the whole K range: no per-block promotion.
  // A scale-writer warpgroup (warps 4-7) turns the fp32 scales into UE8M0
  // bytes in a TMEM ring (16 columns per slot: 4 of activation-row scales, 8
  // of weight-row scales; each 32-bit column holds the scales of 4 K blocks,
  // chosen by the MMA's sf_id); the epilogue (warps 8-15) only drains the
  // finished accumulator.
  static constexpr bool MX = MX_;
  // CLUSTER = 2: two CTAs with adjacent 128-row lane tiles and the same column
  // tile form a cluster. Each loads its own lane tile and one half of the
  // shared column tile, multicast into both, so every CTA reads 2/3 of the
  // operand bytes per K block from L2 that a lone CTA would.
  static constexpr int CLUSTER = CLUSTER_;
  // FUSED: decode linear with act_quant inside -- the CTA quantises the bf16
  // activation itself into a resident shared-memory operand (all K blocks),
  // and only the weights stream through the stage ring.
  static constexpr bool FUSED = FUSED_;
  static constexpr int BN = BN_;
  static constexpr bool SWAP = SWAP_;
  static constexpr int STAGES = STAGES_;
  static constexpr int P = P_;
  static constexpr int EPI_WARPS = EPI_WARPS_;
  static constexpr int MODE = MODE_;
  static constexpr bool GROUPED = GROUPED_;
  // Weight rows one tile covers (SwiGLU: 128 rows of w1 and the same 128 of w3).
  static constexpr int w_rows() { return MODE == kEpiSwiGLU ? BN / 2 : BN; }
  // Extra shared memory: grouped tables (row offsets, cumulative tiles) and
  // the SwiGLU amax exchange between the two column groups (double-buffered).
  static constexpr int kGroupBytes = GROUPED ? 2 * (kMaxGroups + 4) * 4 : 0;
  static constexpr int kXchgBytes = MODE == kEpiSwiGLU ? 2 * 2 * 128 * 4 : 0;
  static constexpr int kGroups = EPI_WARPS / 4;  // column groups in the epilogue
  static constexpr int kCpt = BN / kGroups;      // columns per epilogue thread
  // Register split for large-M tiles (two column groups of 128): 12 warps, and
  // setmaxnreg moves registers from the first warpgroup (TMA producer, MMA
  // issuer, two idle warps) to the two epilogue warpgroups, whose threads hold
  // 128 accumulators next to 64 freshly loaded TMEM columns. The launch holds
  // kThreads x 168 registers; the split hands out exactly that many.
  static constexpr bool kSplitRegs = !SWAP && !FUSED && EPI_WARPS == 8 && kCpt == 128;
  static constexpr int kSfWarp0 = 4;                             // MX: first scale-writer warp
  static constexpr int kEpiWarp0 = MX ? 8 : kSplitRegs ? 4 : 2;  // first epilogue warp
  static constexpr int kThreads = (kEpiWarp0 + EPI_WARPS) * 32;
  static constexpr int kLaunchRegs = MX ? 128 : 168;
  static constexpr int kRegsLow = 56, kRegsHigh = MX ? 200 : 224;
  // MX scale ring: slots of 16 TMEM columns after the accumulator, 4 K blocks each.
  static constexpr int kSfSlots = MX ? 8 : 0;
  static constexpr int kSfCol0 = P * BN;
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = FUSED ? kABytes : kABytes + kBBytes;
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kTmemCols = pow2_at_least(P * BN + 16 * kSfSlots, 32);
  static constexpr int kBarBytes = (2 * STAGES + 2 * P + 3) * 8 + 16 + (2 * kSfSlots + (MX ? 1 : 0)) * 8;
  // MX: the scale writers' exchange of activation-row scale words, double-buffered.
  static constexpr int kSfxBytes = MX ? 2 * 128 * 4 : 0;
  // Dense bf16 tiles with activation rows as lanes store C through TMA: each
  // epilogue warp stages 32 rows x 64 columns (a 4 KB, 128-byte-swizzled box)
  // at a time after the stage ring.
  static constexpr bool kTmaStore = !SWAP && !FUSED && !GROUPED && MODE == kEpiBf16;
  // The SwiGLU (u codes) and scatter (rows in slot order) epilogues write
  // their rows through a 2 KB slab per warp instead (32 rows x 64 bytes),
  // four lanes per row, eight rows per store instruction. (Not the MX scatter
  // epilogue: its 200-register share cannot hold the staging next to the 128
  // accumulators.)
  static constexpr bool kSlabStore = !SWAP && (MODE == kEpiSwiGLU || (MODE == kEpiScatter && !MX));
  static constexpr int kOutSlab = kTmaStore ? 32 * 128 : kSlabStore ? 32 * 64 : 0;
  static constexpr int kOutStageBytes = EPI_WARPS * kOutSlab;
  static constexpr int kSmemBytes =
      1024 + kRingBytes + kOutStageBytes + kBarBytes + kGroupBytes + kXchgBytes + kSfxBytes;

  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
  static_assert(MODE == kEpiBf16 || !SWAP, "SwiGLU and scatter epilogues use activation rows as lanes");
  static_assert(MODE != kEpiSwiGLU || (BN == 256 && EPI_WARPS == 8), "SwiGLU: w1|w3 128+128 columns");
  static_assert(!GROUPED || !SWAP, "grouped GEMMs use activation rows as lanes");
  static_assert(!FUSED || (SWAP && BN <= 32 && MODE == kEpiBf16 && !GROUPED), "fused act_quant: decode tiles");
  static_assert(EPI_WARPS % 4 == 0, "epilogue warps come in warpgroups");
  static_assert(kCpt == 16 || kCpt % 32 == 0, "TMEM loads of 16 or 32 columns");
  static_assert(SWAP || kCpt == 128 || (kCpt == 64 && MODE != kEpiSwiGLU),
                "non-swapped tiles: a column group lies inside one weight block");
  static_assert(!SWAP || kGroups == 1, "swapped tiles: one column group");
  static_assert(P * BN <= 512, "TMEM has 512 columns");
  static_assert(kSfCol0 + 16 * kSfSlots <= 512, "TMEM has 512 columns");
  static_assert(!MX || (!SWAP && !FUSED && BN == 256 && P == 1 && EPI_WARPS == 8 && kSplitRegs),
                "MX: 128 x 256 tiles with activation rows as lanes, one accumulator");
  static_assert(!kSplitRegs || (kEpiWarp0 * 32 * kRegsLow + EPI_WARPS * 32 * kRegsHigh <= kThreads * kLaunchRegs &&
                                kThreads * kLaunchRegs <= 65536),
                "the register split must fit the registers the CTA is launched with");
  static_assert(CLUSTER == 1 || (CLUSTER == 2 && !SWAP && !GROUPED && !FUSED && BN == 256),
                "clusters pair the 128-row lane tiles of dense large-M GEMMs");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Where one output tile lives.
struct TileInfo {
  int lane_y;      // TMA row of the lane operand's 128-row tile
  int col_y;       // TMA row of the column operand's tile (w1/w3 row in SwiGLU mode)
  int lane_valid;  // lane rows of the tile that exist (activation rows, or weight rows when swapped)
  int wblock;      // global 128-row weight block of the tile's first weight row
  int col0;        // first output column (swapped: first token)
};

// Dense tiles run lane-tile fastest. Grouped tiles run (group, column tile,
// 128-row tile) with the row tile fastest, so the row tiles of one group that
// share a weight tile run side by side. rows/mtiles are the group tables in
// shared memory.
template <class C>
__device__ __forceinline__ TileInfo tile_info(const GemmParams& p, int tile, const int* rows, const int* mtiles,
                                              int rank) {
  TileInfo t;
  if constexpr (C::GROUPED) {
    int lo = 0, hi = p.E - 1;  // last group whose first tile is <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (mtiles[mid] * p.tiles_col <= tile) lo = mid;
      else hi = mid - 1;
    }
    const int e = lo;
    const int mt_e = mtiles[e + 1] - mtiles[e];
    const int local = tile - mtiles[e] * p.tiles_col;
    const int nt = local / mt_e, mt = local - nt * mt_e;
    t.lane_y = rows[e] + mt * 128;
    t.lane_valid = min(128, rows[e + 1] - t.lane_y);
    t.col_y = e * p.N + nt * C::w_rows();
    t.wblock = t.col_y / 128;
    t.col0 = nt * C::w_rows();
  } else {
    // Clusters: the schedule's lane index counts CTA pairs; `rank` picks the half.
    const int tl = (tile % p.tiles_lane) * C::CLUSTER + rank, tc = tile / p.tiles_lane;
    t.lane_y = tl * 128;
    if constexpr (C::SWAP) {
      t.lane_valid = min(128, p.N - t.lane_y);
      t.col_y = tc * C::BN;
      t.wblock = tl;
      t.col0 = tc * C::BN;
    } else {
      t.lane_valid = min(128, p.M - t.lane_y);
      t.col_y = tc * C::w_rows();
      t.wblock = t.col_y / 128;
      t.col0 = tc * C::w_rows();
    }
  }
  return t;
}

// Scale of a 128-element block for the fused act_quant (the act_quant rule:
// max(amax, 1e-4) / 448 as an IEEE division; ue8m0: rounded up to 2^k on the bits).
__device__ __forceinline__ float quant_block_scale(float amax, bool ue8m0) {
  float s = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
  if (ue8m0) {
    uint32_t b = __float_as_uint(s);
    if (b & 0x007FFFFFu) b = (b & 0x7F800000u) + 0x00800000u;
    s = __uint_as_float(b);
  }
  return s;
}

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

// A shared-memory counter written by one thread with release semantics and
// read with acquire semantics by others.
__device__ __forceinline__ void st_release_shared(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_shared(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// Waits until *p > k, bounded like mbar_wait: gives up after kWaitLimitNs (or
// once another role has given up), setting *abort and the error bit `code`.
__device__ __forceinline__ bool wait_count_above(const int* p, int k, volatile int* abort, unsigned* err,
                                                 unsigned code) {
  if (ld_acquire_shared(p) > k) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire_shared(p) > k) return true;
    if ((i & 63u) == 0) {
      if (abort && *abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        if (abort) *abort = 1;
        atomicOr(err, code);
        return false;
      }
    }
  }
}

// Coalesced row stores of one warp: lane i holds four 16-byte chunks of row i
// of the warp's 32. They go through `slab` (32 rows x 64 bytes; chunk c of row
// r at position (c + r / 2) % 4, so eight consecutive lanes cover all banks in
// both phases) and out eight rows per instruction, four lanes per row, to
// dst (this lane's row; null for a row that is not written). Every lane of
// the warp must call it.
__device__ __forceinline__ void warp_store_rows(uint8_t* slab, int lane, const uint4 (&v)[4], uint8_t* dst) {
  __syncwarp();  // the slab's previous contents have been read
#pragma unroll
  for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(slab + lane * 64 + (((c + (lane >> 1)) & 3) << 4)) = v[c];
  __syncwarp();
  const unsigned long long mine = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2), c = lane & 3;
    const unsigned long long d = __shfl_sync(0xFFFFFFFFu, mine, r);
    const uint4 val = *reinterpret_cast<const uint4*>(slab + r * 64 + (((c + (r >> 1)) & 3) << 4));
    if (d) *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(d) + c * 16) = val;
  }
}

// Writes one thread's finished accumulators: row `row` of the tile, the
// column group `group`. Returns false if an epilogue-wide wait gave up.
// kTmaStore tiles with p.tma_store: the whole warp (all 32 rows, valid or
// not) converts its rows 64 columns at a time into `slab` (row r's 16-byte
// chunk c at chunk c ^ (r % 8), the 128-byte swizzle) and one lane stores the
// box through `tmap_out`; rows past M and columns past N are clipped by the TMA.
template <class C, class Sync>
__device__ __forceinline__ bool finalize(const GemmParams& p, float (&acc)[C::kCpt], const TileInfo& t, int group,
                                         int row, float* xchg, uint32_t unit_parity, Sync&& epi_sync, uint8_t* slab,
                                         const CUtensorMap* tmap_out) {
  if constexpr (C::SWAP) {
    const int n = t.lane_y + row;
    if (row >= t.lane_valid) return true;  // rows past N
#pragma unroll
    for (int j = 0; j < C::kCpt; ++j) {
      const int m = t.col0 + j;
      if (m < p.M) p.c[static_cast<size_t>(m) * p.ldc + n] = __float2bfloat16_rn(acc[j]);
    }
    return true;
  } else if constexpr (C::MODE == kEpiSwiGLU) {
    // acc[0, 64): h1 of output columns col0 + 64 group + i; acc[64, 128): h3 of the same columns.
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float h1 = bf16_round(acc[i]);
      const float h3 = bf16_round(acc[64 + i]);
      const float g = bf16_round(__fdiv_rn(h1, 1.0f + expf(-h1)));
      const float u = bf16_round(g * h3);
      acc[i] = u;
      amax = fmaxf(amax, fabsf(u));
    }
    // The 128-column quantisation block is split over the two column groups:
    // exchange the half-block maxima through shared memory.
    float* x = xchg + unit_parity * 256;
    x[group * 128 + row] = amax;
    if (!epi_sync()) return false;
    amax = fmaxf(x[row], x[128 + row]);
    const float sc = quant_block_scale(amax, p.ue8m0 != 0);
    const float rc = __frcp_rn(sc);  // the block's quotients: see quotient.cuh
    // This row's 64 codes of the block (rows past the tile's valid rows are
    // computed and not written).
    uint4 q[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = v * 16 + e * 4;
        w[e] = pack_e4m3x4(div_by_scale(acc[i], sc, rc), div_by_scale(acc[i + 1], sc, rc),
                           div_by_scale(acc[i + 2], sc, rc), div_by_scale(acc[i + 3], sc, rc));
      }
      q[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    const bool valid = row < t.lane_valid;
    const size_t r = static_cast<size_t>(t.lane_y + row);
    warp_store_rows(slab, row & 31, q, valid ? p.uq + r * p.ldc + t.col0 + group * 64 : nullptr);
    if (valid && group == 0) p.us[r * (p.ldc / 128) + t.col0 / 128] = sc;
    return true;
  } else {
    if constexpr (C::kTmaStore) {
      if (p.tma_store) {
        const int lane = row & 31;
        const int y = t.lane_y + (row & ~31);             // the warp's first row
        const bool any_row = (row & ~31) < t.lane_valid;  // warp-uniform
#pragma unroll
        for (int h = 0; h < C::kCpt / 64; ++h) {
          const int x = t.col0 + group * C::kCpt + h * 64;
          if (lane == 0) bulk_wait_group_read0();  // the slab's previous box has been read
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 b =
                  __floats2bfloat162_rn(acc[h * 64 + c * 8 + 2 * e], acc[h * 64 + c * 8 + 2 * e + 1]);
              w[e] = *reinterpret_cast<const uint32_t*>(&b);
            }
            *reinterpret_cast<uint4*>(slab + lane * 128 + ((c ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();  // generic-proxy writes, read next by the TMA
          __syncwarp();
          if (lane == 0 && any_row && x < p.N) {
            tma_store_2d(tmap_out, slab, x, y);
            bulk_commit_group();
          }
        }
        return true;
      }
    }
    if constexpr (C::kSlabStore) {
      if (p.vec_store && t.col0 + C::BN <= p.N) {  // warp-uniform: whole 16-byte chunks, all columns inside N
        const bool valid = row < t.lane_valid;
        uint8_t* base = nullptr;
        if (valid) {
          const int r = t.lane_y + row;
          const size_t out_row = C::MODE == kEpiScatter ? static_cast<size_t>(__ldg(p.perm + r)) : static_cast<size_t>(r);
          base = reinterpret_cast<uint8_t*>(p.c + out_row * p.ldc + t.col0 + group * C::kCpt);
        }
#pragma unroll
        for (int q = 0; q < C::kCpt / 32; ++q) {  // 32 columns (64 bytes) per round
          uint4 v[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 b =
                  __floats2bfloat162_rn(acc[q * 32 + c * 8 + 2 * e], acc[q * 32 + c * 8 + 2 * e + 1]);
              w[e] = *reinterpret_cast<const uint32_t*>(&b);
            }
            v[c] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          warp_store_rows(slab, row & 31, v, base ? base + q * 64 : nullptr);
        }
        return true;
      }
    }
    if (row >= t.lane_valid) return true;
    const int r = t.lane_y + row;
    const size_t out_row = C::MODE == kEpiScatter ? static_cast<size_t>(__ldg(p.perm + r)) : static_cast<size_t>(r);
    const int n0 = t.col0 + group * C::kCpt;
    __nv_bfloat16* crow = p.c + out_row * p.ldc;
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
    return true;
  }
}

// Optional phase trace (compile with -DFP8BLK_TRACE): %globaltimer stamps per
// CTA at fixed points of each role, read back with fp8trace_read(). Not part
// of the library's interface; default builds contain none of it.
// Slots 16.. hold per-role sums of SM cycles (FP8BLK_PUT), e.g. time spent in
// one kind of wait.
#ifdef FP8BLK_TRACE
constexpr int kTraceSlots = 32;
__device__ unsigned long long g_trace[8 * 4096 * kTraceSlots];
#define FP8BLK_PUT(slot, value)                                                                          \
  do {                                                                                                   \
    if (blockIdx.x < 4096) g_trace[((prm.trace_id & 7) * 4096 + blockIdx.x) * kTraceSlots + (slot)] = (value); \
  } while (0)
#define FP8BLK_STAMP(slot) FP8BLK_PUT(slot, global_timer_ns())
// Per-K-block event timeline of CTA 0 in SM cycles: g_timeline[event][k-block].
constexpr int kTimelineLen = 1024;
__device__ long long g_timeline[16 * kTimelineLen];
#define FP8BLK_TL(ev, j)                                                                 \
  do {                                                                                   \
    if (blockIdx.x == 0 && (j) < kTimelineLen) g_timeline[(ev) * kTimelineLen + (j)] = clock64(); \
  } while (0)
#define FP8BLK_TIC(v) const long long v = clock64()
#define FP8BLK_TOC(sum, v) (sum) += clock64() - (v)
#else
#define FP8BLK_PUT(slot, value) do { } while (0)
#define FP8BLK_TL(ev, j) do { } while (0)
#define FP8BLK_STAMP(slot) do { } while (0)
#define FP8BLK_TIC(v) do { } while (0)
#define FP8BLK_TOC(sum, v) do { } while (0)
#endif

// Shared memory of the fused decode operand: Kb blocks of BN rows x 128
// e4m3, then Kb x BN fp32 scales.
__host__ __device__ constexpr size_t fused_extra_bytes(int Kb, int BN) {
  return static_cast<size_t>(Kb) * BN * 128 + ((static_cast<size_t>(Kb) * BN * 4 + 15) & ~size_t{15});
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_lane, const __grid_constant__ CUtensorMap tmap_col,
                    const __grid_constant__ CUtensorMap tmap_col2, const GemmParams prm) {
  // tmap_col2: the w3 operand (SwiGLU), or C as TMA stores see it (kTmaStore
  // tiles with prm.tma_store), else unused.
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  // Fused decode: the quantised activation (all K blocks, BN token rows each,
  // 128-byte swizzled like a TMA tile) and its scales follow the stage ring.
  uint8_t* out_stage = smem + C::kRingBytes;  // kTmaStore: one slab per epilogue warp
  uint8_t* act_smem = out_stage + C::kOutStageBytes;
  float* act_scale = reinterpret_cast<float*>(act_smem + static_cast<size_t>(prm.Kb) * C::BN * 128);
  uint8_t* tail = act_smem + (C::FUSED ? fused_extra_bytes(prm.Kb, C::BN) : 0);
  uint64_t* full = reinterpret_cast<uint64_t*>(tail);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + C::P;
  uint64_t* drain = tempty + C::P;
  uint64_t* epi_bar = drain + 1;    // epilogue-only barrier (stream-K fixup, SwiGLU amax exchange)
  // Fused decode: the number of K blocks of the activation operand already
  // quantised (written with release semantics after each pass, read with
  // acquire semantics by the MMA warp); an 8-byte slot of the barrier area.
  int* act_kb = reinterpret_cast<int*>(epi_bar + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;
  int* grp_rows = reinterpret_cast<int*>(tail + C::kBarBytes);
  int* grp_mtiles = grp_rows + (kMaxGroups + 4);
  float* xchg = reinterpret_cast<float*>(tail + C::kBarBytes + C::kGroupBytes);
  // MX scale ring: sf_full (the four scale writers have stored a slot),
  // sf_empty (the MMAs that read a slot have completed).
  uint64_t* sf_full = reinterpret_cast<uint64_t*>(tail + (2 * C::STAGES + 2 * C::P + 3) * 8 + 16);
  uint64_t* sf_empty = sf_full + C::kSfSlots;
  uint64_t* wr_bar = sf_empty + C::kSfSlots;  // the four scale writers, once per scale group
  uint32_t* sfx = reinterpret_cast<uint32_t*>(tail + C::kBarBytes + C::kGroupBytes + C::kXchgBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Cluster rank, and the index of the schedule this CTA (pair) walks.
  const int rank = C::CLUSTER > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  // Split-K clusters (swapped tiles only): ksplit CTAs per tile.
  const int ksplit = C::SWAP ? prm.ksplit : 1;
  const int krank = ksplit > 1 ? static_cast<int>(blockIdx.x) % ksplit : 0;
  const int worker = static_cast<int>(blockIdx.x) / (ksplit > 1 ? ksplit : C::CLUSTER);
  if (threadIdx.x == 0) FP8BLK_STAMP(0);
#ifdef FP8BLK_TRACE
  if (threadIdx.x == 0) {
    unsigned sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    FP8BLK_PUT(26, sm);
  }
#endif
  // The next kernel on the stream may begin its prologue (and its weight
  // loads) now; it waits for this one before touching anything we write.
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::CLUSTER);  // freed by the MMAs of every CTA that shares the stage
    }
    for (int q = 0; q < C::P; ++q) {
      mbar_init(&tfull[q], 1);
      mbar_init(&tempty[q], C::EPI_WARPS);
    }
    mbar_init(drain, 1);
    mbar_init(epi_bar, C::EPI_WARPS);
    *act_kb = 0;
    for (int q = 0; q < C::kSfSlots; ++q) {
      mbar_init(&sf_full[q], 4);
      mbar_init(&sf_empty[q], 1);
    }
    if constexpr (C::MX) mbar_init(wr_bar, 4);
    *abort_flag = 0;
    *last_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_lane);
    tma_prefetch_desc(&tmap_col);
    if constexpr (C::MODE == kEpiSwiGLU) tma_prefetch_desc(&tmap_col2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  int grouped_tiles = -1;
  if constexpr (C::GROUPED) {
    griddep_wait();  // the group tables come from the previous kernel
    for (int i = threadIdx.x; i <= prm.E; i += C::kThreads) {
      grp_rows[i] = __ldg(prm.grp_rows + i);
      grp_mtiles[i] = __ldg(prm.grp_mtiles + i);
    }
  }
  tc_fence_before_sync();
  // Clusters: no CTA multicasts into its peer before the peer's barriers exist.
  if constexpr (C::CLUSTER > 1) cluster_sync();
  else __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) FP8BLK_STAMP(1);
  if constexpr (C::GROUPED) grouped_tiles = grp_mtiles[prm.E] * prm.tiles_col;

  // Roles: warp 0 TMA producer, warp 1 MMA issuer, warps kEpiWarp0.. promotion
  // and epilogue. With the register split, each warpgroup sets its budget at
  // the head of its own branch, so the code it runs is compiled for it.
  if (warp < C::kEpiWarp0) {
  if constexpr (C::kSplitRegs) setmaxnreg_dec<C::kRegsLow>();
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // The weight operand is the lane operand when swapped, else the column one.
      auto load_weights = [&](int st, const TileInfo& t, int kb) {
        uint8_t* sa = smem + st * C::kStageBytes;
        if constexpr (C::SWAP) {
          tma_load_2d(sa, &tmap_lane, &full[st], kb * 128, t.lane_y);
        } else if constexpr (C::MODE == kEpiSwiGLU) {
          // Column rows [0,64) w1, [64,128) w3, [128,192) w1 + 64, [192,256) w3 + 64.
          uint8_t* sb = sa + C::kABytes;
          if constexpr (C::CLUSTER > 1) {  // rank r loads rows [128 r, 128 r + 128) into both CTAs
            const int off = rank * 64;
            tma_load_2d_multicast(sb + 2 * off * 128, &tmap_col, &full[st], kb * 128, t.col_y + off, 0x3);
            tma_load_2d_multicast(sb + (2 * off + 64) * 128, &tmap_col2, &full[st], kb * 128, t.col_y + off, 0x3);
          } else {
            tma_load_2d(sb, &tmap_col, &full[st], kb * 128, t.col_y);
            tma_load_2d(sb + 64 * 128, &tmap_col2, &full[st], kb * 128, t.col_y);
            tma_load_2d(sb + 128 * 128, &tmap_col, &full[st], kb * 128, t.col_y + 64);
            tma_load_2d(sb + 192 * 128, &tmap_col2, &full[st], kb * 128, t.col_y + 64);
          }
        } else if constexpr (C::CLUSTER > 1) {
          tma_load_2d_multicast(sa + C::kABytes + rank * 128 * 128, &tmap_col, &full[st], kb * 128,
                                t.col_y + rank * 128, 0x3);
        } else {
          tma_load_2d(sa + C::kABytes, &tmap_col, &full[st], kb * 128, t.col_y);
        }
      };
      auto load_acts = [&](int st, const TileInfo& t, int kb) {
        if constexpr (C::FUSED) return;  // the epilogue warps build the activation operand
        uint8_t* sa = smem + st * C::kStageBytes;
        if constexpr (C::SWAP) tma_load_2d(sa + C::kABytes, &tmap_col, &full[st], kb * 128, t.col_y);
        else tma_load_2d(sa, &tmap_lane, &full[st], kb * 128, t.lane_y);
      };
      constexpr uint32_t stage_tx = C::kStageBytes;
      // Weights do not depend on the previous kernel on the stream: the first
      // STAGES stages start loading them before the dependency wait; the
      // activations follow once the previous kernel has completed.
      int npre = 0;
      if constexpr (!C::GROUPED) {
        Sched pre(prm, worker, -1, krank);
        Unit u;
        while (npre < C::STAGES && pre.next(u)) {
          const TileInfo t = tile_info<C>(prm, u.tile, grp_rows, grp_mtiles, rank);
          for (int kb = u.kb0; kb < u.kb1 && npre < C::STAGES; ++kb) {
            mbar_arrive_expect_tx(&full[npre], stage_tx);
            load_weights(npre, t, kb);
            ++npre;
          }
        }
      }
      griddep_wait();
      FP8BLK_STAMP(2);
      Sched sch(prm, worker, grouped_tiles, krank);
      Unit u;
      int st = 0;
      uint32_t ph = 0;
      long long issued = 0;
      bool ok = true;
#ifdef FP8BLK_TRACE
      long long tw_empty = 0;
#endif
      while (ok && sch.next(u)) {
        const TileInfo t = tile_info<C>(prm, u.tile, grp_rows, grp_mtiles, rank);
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (issued < npre) {
            load_acts(st, t, kb);  // stage st == issued: weights already on their way
          } else {
            FP8BLK_TIC(t0);
            if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, prm.err, kDevErrTimeoutProducer)) {
              ok = false;
              break;
            }
            FP8BLK_TOC(tw_empty, t0);
            mbar_arrive_expect_tx(&full[st], stage_tx);
            load_weights(st, t, kb);
            load_acts(st, t, kb);
#ifdef FP8BLK_TRACE
            if (issued == C::STAGES) FP8BLK_STAMP(10);
            FP8BLK_STAMP(11);
#endif
          }
          FP8BLK_TL(0, issued);
          ++issued;
          if (++st == C::STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
#ifdef FP8BLK_TRACE
      FP8BLK_PUT(20, tw_empty);
#endif
      if constexpr (C::CLUSTER > 1) {
        // Wait until both CTAs' MMAs have released the last stages: their
        // multicast arrivals on this CTA's barriers have then all landed.
        const long long n = issued < C::STAGES ? issued : C::STAGES;
        for (long long i = 0; ok && i < n; ++i) {
          if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, prm.err, kDevErrTimeoutProducer)) ok = false;
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
    if constexpr (C::MX) {
    // ---------------- MMA issuer, tensor-core scaling ----------------
    // One accumulator per unit: the first MMA of the unit overwrites it, every
    // later one adds. A K block waits for its operands and, at the start of
    // each group of 4 K blocks, for its scale slot; the slot is released
    // after the group's MMAs, the accumulator after the unit's last.
    const bool leader = elect_one_sync();
    Sched sch(prm, worker, grouped_tiles, krank);
    Unit u;
    int st = 0, sfs = 0;
    uint32_t ph = 0, sfph = 0, tph = 0;
    bool ok = true;
    const uint32_t sf0 = tmem_base + static_cast<uint32_t>(C::kSfCol0);
    while (ok && sch.next(u)) {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tempty[0], tph ^ 1u, abort_flag, prm.err, kDevErrTimeoutMma))) {
        ok = false;
        break;
      }
      for (int kb = u.kb0; kb < u.kb1; ++kb) {
        const int g = kb - u.kb0;
        const bool last = kb + 1 == u.kb1;
        const bool slot_end = (g & 3) == 3 || last;
        bool w = mbar_wait(&full[st], ph, abort_flag, prm.err, kDevErrTimeoutMma);
        if ((g & 3) == 0) w = w && mbar_wait(&sf_full[sfs], sfph, abort_flag, prm.err, kDevErrTimeoutMma);
        if (!__all_sync(0xFFFFFFFFu, w)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_addr = smem_u32(smem + st * C::kStageBytes);
        const uint64_t ad = sdesc_kmajor_sw128(a_addr);
        const uint64_t bd = sdesc_kmajor_sw128(a_addr + C::kABytes);
        const uint32_t idesc = idesc_mx_e4m3(128, C::BN, static_cast<uint32_t>(g & 3));
        const uint32_t sfa = sf0 + static_cast<uint32_t>(sfs * 16);
        if (leader) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_mx_e4m3(tmem_base, ad + 2 * k, bd + 2 * k, idesc, sfa, sfa + 4, (g > 0 || k > 0) ? 1u : 0u);
          if constexpr (C::CLUSTER > 1) mma_commit_multicast(&empty[st], 0x3);
          else mma_commit(&empty[st]);
          if (slot_end) mma_commit(&sf_empty[sfs]);
          if (last) mma_commit(&tfull[0]);
        }
        __syncwarp();
        if (++st == C::STAGES) {
          st = 0;
          ph ^= 1u;
        }
        if (slot_end && ++sfs == C::kSfSlots) {
          sfs = 0;
          sfph ^= 1u;
        }
      }
      tph ^= 1u;
    }
    if (leader) {
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, prm.err, kDevErrTimeoutDrain);
    }
    __syncwarp();
    } else {
    // ---------------- MMA issuer ----------------
    // The whole warp walks the schedule and waits; one elected lane issues the
    // MMAs and commits, so the warp stays converged around the tcgen05 issue
    // (a loop run by a lone lane issues them far more slowly).
    const bool leader = elect_one_sync();
    constexpr uint32_t kIdesc = idesc_e4m3_f32(128, C::BN);
    Sched sch(prm, worker, grouped_tiles, krank);
    Unit u;
    int st = 0, pb = 0;
    uint32_t ph = 0, pph = 0;
    bool ok = true;
    // Every lane waits; a wait that gave up in any lane stops the whole warp.

#ifdef FP8BLK_TRACE
    long long tw_full = 0, tw_tmem = 0, n_kb = 0;
    FP8BLK_TIC(t_loop);
#endif
    while (ok && sch.next(u)) {
      for (int kb = u.kb0; kb < u.kb1; ++kb) {
        if constexpr (C::FUSED) {
          // K block kb of the activation operand has been quantised.
          if (!__all_sync(0xFFFFFFFFu, wait_count_above(act_kb, kb, abort_flag, prm.err, kDevErrTimeoutMma))) {
            ok = false;
            break;
          }
        }
        FP8BLK_TIC(t0);
        bool w = mbar_wait(&full[st], ph, abort_flag, prm.err, kDevErrTimeoutMma);
        FP8BLK_TOC(tw_full, t0);
#ifdef FP8BLK_TRACE
        if (leader) FP8BLK_TL(1, n_kb);
#endif
        FP8BLK_TIC(t1);
        w = w && mbar_wait(&tempty[pb], pph ^ 1u, abort_flag, prm.err, kDevErrTimeoutMma);
        FP8BLK_TOC(tw_tmem, t1);
        if (!__all_sync(0xFFFFFFFFu, w)) {
          ok = false;
          break;
        }
#ifdef FP8BLK_TRACE
        if (leader) {
          FP8BLK_TL(2, n_kb);
          if (st == 0 && ph == 0 && pb == 0) FP8BLK_STAMP(3);
          if (st == 0 && ph == 1) FP8BLK_STAMP(12);
        }
        ++n_kb;
#endif
        tc_fence_after_sync();
        const uint32_t a_addr = smem_u32(smem + st * C::kStageBytes);
        const uint64_t ad = sdesc_kmajor_sw128(a_addr);
        const uint64_t bd = C::FUSED ? sdesc_kmajor_sw128(smem_u32(act_smem + kb * (C::BN * 128)))
                                     : sdesc_kmajor_sw128(a_addr + C::kABytes);
        const uint32_t d = tmem_base + static_cast<uint32_t>(pb * C::BN);
        if (leader) {
#pragma unroll
          for (int k = 0; k < 4; ++k)  // 32-byte K slices: start address advances by 32 B (2 x 16 B)
            mma_e4m3(d, ad + 2 * k, bd + 2 * k, kIdesc, k > 0 ? 1u : 0u);
          if constexpr (C::CLUSTER > 1) mma_commit_multicast(&empty[st], 0x3);  // the stage is shared
          else mma_commit(&empty[st]);
          mma_commit(&tfull[pb]);
          FP8BLK_TL(3, n_kb - 1);
        }
        __syncwarp();
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
#ifdef FP8BLK_TRACE
    if (leader) {
      FP8BLK_STAMP(4);
      FP8BLK_PUT(16, tw_full);
      FP8BLK_PUT(17, tw_tmem);
      FP8BLK_PUT(18, n_kb);
      FP8BLK_PUT(19, clock64() - t_loop);
    }
#endif
    // Wait for every MMA the leader issued before TMEM is released.
    if (leader) {
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, prm.err, kDevErrTimeoutDrain);
    }
    __syncwarp();
    }
  } else if (warp >= C::kSfWarp0) {
    if constexpr (C::MX) {
      // ---------------- scale writer (MX) ----------------
      // For each group of 4 K blocks of a unit: the UE8M0 byte (the fp32
      // exponent field of a power-of-two scale) of every activation row's and
      // every weight row's scale, byte j for K block j of the group, stored
      // the same way into each of the four TMEM lane quarters: lane l, column
      // i holds operand row 32 i + l (columns 0-3 activation rows, 4-11 the
      // 256 weight rows, one weight block per 128 rows). K blocks past the
      // unit and rows past the matrix get 127 (a scale of 1).
      // Thread (quarter q, lane l) loads the scales of activation row 32 q + l
      // (one group ahead, so the loads overlap the previous group's stores);
      // the four warps exchange the packed row words through shared memory.
      // Lanes 0-7 load the tile's weight-block scales (block l / 4, K block
      // l % 4), packed by shuffles.
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;
      const uint32_t t_sf = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(C::kSfCol0);
      griddep_wait();  // the activation scales come from the previous kernel
      bool bad = false;
      auto ue8m0 = [&](float v) -> uint32_t {
        const uint32_t b = __float_as_uint(v);
        const uint32_t e = b >> 23;  // sign bit set: e >= 256
        bad |= (b & 0x007FFFFFu) != 0u || e == 0u || e >= 255u;
        return e & 0xFFu;
      };
      Sched sch(prm, worker, grouped_tiles, krank);
      Unit u;
      TileInfo t{};
      bool have = sch.next(u);
      if (have) t = tile_info<C>(prm, u.tile, grp_rows, grp_mtiles, rank);
      int k0 = have ? u.kb0 : 0;
      float ra[4], rw = 1.0f;
      auto fetch = [&]() {
        const int nk = u.kb1 - k0 < 4 ? u.kb1 - k0 : 4;
        const float* src = prm.a_s + static_cast<size_t>(t.lane_y + row) * prm.Kb + k0;
#pragma unroll
        for (int j = 0; j < 4; ++j) ra[j] = (row < t.lane_valid && j < nk) ? __ldg(src + j) : 1.0f;
        rw = 1.0f;
        if (lane < 8) {
          const int jb = lane & 3, blk = lane >> 2;
          // SwiGLU tiles: rows [0,64) w1, [64,128) w3, [128,192) w1, [192,256) w3, one block of each.
          const float* ws = (C::MODE == kEpiSwiGLU && blk) ? prm.w3_s : prm.w_s;
          const int nb = C::MODE == kEpiSwiGLU ? t.wblock : t.wblock + blk;
          if (jb < nk && (C::GROUPED || C::MODE == kEpiSwiGLU || nb < prm.n_wblocks))
            rw = __ldg(ws + static_cast<size_t>(nb) * prm.Kb + k0 + jb);
        }
      };
      if (have) fetch();
      int sfs = 0, xb = 0;
      uint32_t sfph = 0, xph = 0;
      bool ok = true;
      while (ok && have) {
        uint32_t wrow = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) wrow |= ue8m0(ra[j]) << (8 * j);
        const uint32_t wbyte = ue8m0(rw);
        // Advance to the next group and start its loads.
        k0 += 4;
        if (k0 >= u.kb1) {
          have = sch.next(u);
          if (have) {
            t = tile_info<C>(prm, u.tile, grp_rows, grp_mtiles, rank);
            k0 = u.kb0;
          }
        }
        if (have) fetch();
        // Exchange the row words (bounded mbarrier over the four warps).
        sfx[xb * 128 + row] = wrow;
        __syncwarp();
        if (lane == 0) mbar_arrive(wr_bar);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(wr_bar, xph, abort_flag, prm.err, kDevErrTimeoutEpilogue))) {
          ok = false;
          break;
        }
        xph ^= 1u;
        uint32_t wa[4], wb[8], blkw[2];
#pragma unroll
        for (int i = 0; i < 4; ++i) wa[i] = sfx[xb * 128 + 32 * i + lane];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          blkw[b] = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) blkw[b] |= __shfl_sync(0xFFFFFFFFu, wbyte, 4 * b + j) << (8 * j);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) wb[i] = blkw[C::MODE == kEpiSwiGLU ? ((i >> 1) & 1) : (i >> 2)];
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait(&sf_empty[sfs], sfph ^ 1u, abort_flag, prm.err, kDevErrTimeoutEpilogue))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        tmem_st_32x32b_x4(t_sf + static_cast<uint32_t>(sfs * 16), wa);
        tmem_st_32x32b_x8(t_sf + static_cast<uint32_t>(sfs * 16 + 4), wb);
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_full[sfs]);
        if (++sfs == C::kSfSlots) {
          sfs = 0;
          sfph ^= 1u;
        }
        xb ^= 1;
      }
      if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(prm.err, kDevErrBadScale);
    }
  }
  } else {
    if constexpr (C::kSplitRegs) setmaxnreg_inc<C::kRegsHigh>();
    // ---------------- promotion + epilogue ----------------
    const int ew = warp - C::kEpiWarp0;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int group = ew >> 2;     // column group
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr int kAsRegs = (C::kCpt + 31) / 32;
    uint8_t* out_slab = out_stage + ew * C::kOutSlab;  // kTmaStore: this warp's staging box
    if constexpr (C::kTmaStore) {
      if (prm.tma_store && lane == 0) tma_prefetch_desc(&tmap_col2);
    }

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

    if constexpr (C::FUSED) {
      // Rows M..BN-1 of the resident operand and their scales are zero; they
      // do not depend on x, so they are written before the dependency wait.
      const int et = threadIdx.x - C::kEpiWarp0 * 32;  // 0 .. 127
      const int pad_rows = C::BN - prm.M;
      for (int i = et; i < pad_rows * prm.Kb * 8; i += C::EPI_WARPS * 32) {
        const int r = prm.M + i / (prm.Kb * 8), rem = i % (prm.Kb * 8);
        const int kb = rem >> 3, chunk = rem & 7;
        *reinterpret_cast<uint4*>(act_smem + kb * (C::BN * 128) + (r >> 3) * 1024 + (r & 7) * 128 + chunk * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      for (int i = et; i < pad_rows * prm.Kb; i += C::EPI_WARPS * 32)
        act_scale[(i % prm.Kb) * C::BN + prm.M + i / prm.Kb] = 0.0f;
    }
    griddep_wait();  // activation scales and every output are the previous kernel's business
    if (threadIdx.x == C::kEpiWarp0 * 32) FP8BLK_STAMP(5);
    if constexpr (C::FUSED) {
      // act_quant of x [M, K] into the resident MMA operand: the act_quant rule
      // per (row, 128 columns) -- amax, max(amax, 1e-4) / 448 (ue8m0: rounded
      // up to 2^k), codes e4m3(x / s) -- one 128-element block per 16 lanes.
      // Layout: block kb at kb*BN*128, row m at (m / 8) * 1024 + (m % 8) * 128,
      // its 16-byte chunk c stored at chunk c ^ (m % 8) (the 128-byte swizzle
      // the descriptors name). Blocks go K block by K block (b = kb * M + m),
      // eight per pass (one per half-warp); after each pass the K blocks it
      // completed are published to the MMA warp, which starts on K block 0
      // while later ones are still being quantised.
      const int et = threadIdx.x - C::kEpiWarp0 * 32;  // 0 .. 127
      const int sub = et & 15, hw = et >> 4;
      const int total = prm.M * prm.Kb;
      const int K = prm.Kb * 128;
      // Up to kQb passes are loaded before any is used, so their L2/DRAM round
      // trips overlap.
      constexpr int kQb = 16;
      constexpr int kPass = C::EPI_WARPS * 2;  // half-warps
      for (int base = 0; base < total; base += kPass * kQb) {
        uint4 v[kQb];
#pragma unroll
        for (int q = 0; q < kQb; ++q) {
          const int b = base + q * kPass + hw;
          const int kb = b / prm.M, m = b - kb * prm.M;
          v[q] = b < total ? __ldg(reinterpret_cast<const uint4*>(prm.x + static_cast<size_t>(m) * K + kb * 128) +
                                   sub)
                           : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < kQb; ++q) {
          const int b = base + q * kPass + hw;
          if (base + q * kPass >= total) break;  // uniform over the epilogue: no block of this pass exists
          const bool valid = b < total;
          const int kb = valid ? b / prm.M : 0, m = valid ? b - kb * prm.M : 0;
          const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
          float f[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
          }
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
          for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off, 16));
          const float sc = quant_block_scale(amax, prm.ue8m0 != 0);
          const float rc = __frcp_rn(sc);  // the block's quotients: see quotient.cuh
          const uint32_t lo = pack_e4m3x4(div_by_scale(f[0], sc, rc), div_by_scale(f[1], sc, rc),
                                          div_by_scale(f[2], sc, rc), div_by_scale(f[3], sc, rc));
          const uint32_t hi = pack_e4m3x4(div_by_scale(f[4], sc, rc), div_by_scale(f[5], sc, rc),
                                          div_by_scale(f[6], sc, rc), div_by_scale(f[7], sc, rc));
          if (valid) {
            uint8_t* rowp = act_smem + kb * (C::BN * 128) + (m >> 3) * 1024 + (m & 7) * 128;
            *reinterpret_cast<uint2*>(rowp + (((sub >> 1) ^ (m & 7)) << 4) + (sub & 1) * 8) = make_uint2(lo, hi);
            if (sub == 0) act_scale[kb * C::BN + m] = sc;
          }
          fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
          named_barrier_sync(1, C::EPI_WARPS * 32);
          if (et == 0) {
            const int done = (base + (q + 1) * kPass) / prm.M;  // K blocks all of whose rows are written
            st_release_shared(act_kb, done < prm.Kb ? done : prm.Kb);
          }
        }
      }
      if (threadIdx.x == C::kEpiWarp0 * 32) FP8BLK_STAMP(6);
    }
    // Raw scale loads of one K block, issued kAhead blocks before their use so
    // that their L2 round trips overlap the MMAs of the blocks in between.
    constexpr int kColRegs = (C::SWAP && !C::FUSED) ? kAsRegs : 1;
    struct ScaleRaw {
      float a, w, w3;
      float col[kColRegs];
    };
    constexpr int kAhead = C::EPI_WARPS == 8 ? 3 : 4;
    auto load_scales = [&](const TileInfo& t, int kb, int kb_end) -> ScaleRaw {
      ScaleRaw r;
      r.a = r.w = r.w3 = 0.0f;
#pragma unroll
      for (int i = 0; i < kColRegs; ++i) r.col[i] = 0.0f;
      if (kb >= kb_end) return r;
      if constexpr (!C::SWAP) {
        if (row < t.lane_valid) r.a = __ldg(prm.a_s + static_cast<size_t>(t.lane_y + row) * prm.Kb + kb);
        if constexpr (C::MODE == kEpiSwiGLU) {
          r.w = __ldg(prm.w_s + static_cast<size_t>(t.wblock) * prm.Kb + kb);
          r.w3 = __ldg(prm.w3_s + static_cast<size_t>(t.wblock) * prm.Kb + kb);
        } else {
          const int nb = t.wblock + (group * C::kCpt) / 128;
          if (C::GROUPED || nb < prm.n_wblocks) r.w = __ldg(prm.w_s + static_cast<size_t>(nb) * prm.Kb + kb);
        }
      } else {
        // This lane's weight row: a slice can straddle two 128-row scale blocks.
        const int n = t.lane_y + row;
        if (n < prm.N) r.w = __ldg(prm.w_s + static_cast<size_t>(n >> 7) * prm.Kb + kb);
        if constexpr (!C::FUSED) {
#pragma unroll
          for (int i = 0; i < kColRegs; ++i) {
            const int j = lane + 32 * i;
            const int m = t.col0 + j;
            if (j < C::kCpt && m < prm.M) r.col[i] = __ldg(prm.a_s + static_cast<size_t>(m) * prm.Kb + kb);
          }
        }
      }
      return r;
    };

    // Non-swapped tiles: this thread's activation-row scales and the tile's
    // weight-block scales of kQ consecutive K blocks (a group), one vector
    // load each when the arrays allow it, the next group in flight while the
    // current one is used (the same a_s * w_s products as one K block at a time).
    constexpr int kQ = (C::MODE == kEpiBf16 && !C::GROUPED) ? FP8BLK_SCALE_VEC : 1;
    using QV = typename std::conditional<kQ == 4, float4, typename std::conditional<kQ == 2, float2, float>::type>::type;
    struct Quad {
      QV a, w, w3;
    };
    auto load_quad = [&](const TileInfo& t, int q) -> Quad {
      Quad r{};
      const int k0 = q * kQ;
      if (k0 >= prm.Kb) return r;
      auto ld4 = [&](const float* p) -> QV {
        if (prm.vec_scales) return __ldg(reinterpret_cast<const QV*>(p));
        QV v{};
        float* f = reinterpret_cast<float*>(&v);
#pragma unroll
        for (int i = 0; i < kQ; ++i) f[i] = k0 + i < prm.Kb ? __ldg(p + i) : 0.0f;
        return v;
      };
      if (row < t.lane_valid) r.a = ld4(prm.a_s + static_cast<size_t>(t.lane_y + row) * prm.Kb + k0);
      if constexpr (C::MODE == kEpiSwiGLU) {
        r.w = ld4(prm.w_s + static_cast<size_t>(t.wblock) * prm.Kb + k0);
        r.w3 = ld4(prm.w3_s + static_cast<size_t>(t.wblock) * prm.Kb + k0);
      } else {
        const int nb = t.wblock + (group * C::kCpt) / 128;
        if (C::GROUPED || nb < prm.n_wblocks) r.w = ld4(prm.w_s + static_cast<size_t>(nb) * prm.Kb + k0);
      }
      return r;
    };
    auto pick4 = [](const QV& v, int i) -> float {
      const float* f = reinterpret_cast<const float*>(&v);
      float r = f[0];
#pragma unroll
      for (int j = 1; j < kQ; ++j) r = i == j ? f[j] : r;
      return r;
    };

    Sched sch(prm, worker, grouped_tiles, krank);
    Unit u;
    int pb = 0;
    uint32_t pph = 0;
    uint32_t unit_parity = 0;
    bool ok = true;
#ifdef FP8BLK_TRACE
    long long tw_tfull = 0, t_busy = 0, t_fin = 0;
    int ekb = 0;
#endif
    while (ok && sch.next(u)) {
      const TileInfo t = tile_info<C>(prm, u.tile, grp_rows, grp_mtiles, rank);
      float acc[C::kCpt];
      if constexpr (C::MX) {
        // The unit's accumulator is complete in TMEM (scaled by the tensor
        // core): read this thread's 128 columns, then free it for the next unit.
        if (!mbar_wait(&tfull[0], pph, abort_flag, prm.err, kDevErrTimeoutEpilogue)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int h = 0; h < C::kCpt / 64; ++h) {
          uint32_t v[64];
          tmem_ld_32x32b_x64(t_lane + static_cast<uint32_t>(group * C::kCpt + h * 64), v);
#pragma unroll
          for (int i = 0; i < 64; ++i) acc[h * 64 + i] = __uint_as_float(v[i]);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[0]);
        pph ^= 1u;
      } else {
#pragma unroll
      for (int i = 0; i < C::kCpt; ++i) acc[i] = 0.0f;
      constexpr bool kPipe = C::SWAP || kQ == 1;
      ScaleRaw pipe[kPipe ? kAhead : 1];
      Quad qc{}, qn{};
      int qcur = u.kb0 / kQ;
      if constexpr (kPipe) {
#pragma unroll
        for (int d = 0; d < kAhead; ++d) pipe[d] = load_scales(t, u.kb0 + d, u.kb1);
      } else {
        qc = load_quad(t, qcur);
        qn = (qcur + 1) * kQ < u.kb1 ? load_quad(t, qcur + 1) : Quad{};
      }

      for (int kb = u.kb0; kb < u.kb1; ++kb) {
        // Scales of this K block: loaded kAhead blocks earlier (swapped tiles:
        // the shifting window `pipe`) or with its quad of four K blocks, the
        // next quad in flight; multiplied here. sc_lo applies to the first
        // half of the thread's columns, sc_hi to the second (they differ only
        // in SwiGLU mode: w1 vs w3 scales).
        ScaleRaw cur{};
        if constexpr (kPipe) {
          cur = pipe[0];
#pragma unroll
          for (int d = 0; d + 1 < kAhead; ++d) pipe[d] = pipe[d + 1];
          pipe[kAhead - 1] = load_scales(t, kb + kAhead, u.kb1);
        } else {
          if (kb / kQ != qcur) {
            qc = qn;
            ++qcur;
            qn = (qcur + 1) * kQ < u.kb1 ? load_quad(t, qcur + 1) : Quad{};
          }
          cur.a = pick4(qc.a, kb % kQ);
          cur.w = pick4(qc.w, kb % kQ);
          cur.w3 = pick4(qc.w3, kb % kQ);
        }
        float sc_lo = 0.0f, sc_hi = 0.0f;
        // Swapped tiles: sc_col[i] is the activation scale of token lane + 32 i
        // (shuffled to the thread that owns each column), w_row this thread's
        // own weight-row scale (rows of a slice can lie in two scale blocks).
        float sc_col[kAsRegs];
        const float w_row = cur.w;
        if constexpr (!C::SWAP) {
          sc_lo = cur.a * cur.w;
          sc_hi = C::MODE == kEpiSwiGLU ? cur.a * cur.w3 : sc_lo;
        } else {
#pragma unroll
          for (int i = 0; i < kAsRegs; ++i) {
            const int j = lane + 32 * i;
            if constexpr (C::FUSED)
              sc_col[i] = (j < C::kCpt) ? act_scale[kb * C::BN + j] : 0.0f;
            else
              sc_col[i] = cur.col[i < kColRegs ? i : 0];
          }
        }
        FP8BLK_TIC(t0);
        if (!mbar_wait(&tfull[pb], pph, abort_flag, prm.err, kDevErrTimeoutEpilogue)) {
          ok = false;
          break;
        }
        FP8BLK_TOC(tw_tfull, t0);
#ifdef FP8BLK_TRACE
        if (lane == 0 && ew == 0) FP8BLK_TL(4, ekb);
        if (lane == 0 && ew == C::EPI_WARPS - 1) FP8BLK_TL(6, ekb);
#endif
        FP8BLK_TIC(t1);
#ifdef FP8BLK_TRACE
        if (threadIdx.x == C::kEpiWarp0 * 32 && pb == 0 && pph == 0) FP8BLK_STAMP(7);
        if (threadIdx.x == C::kEpiWarp0 * 32 && kb == u.kb0 + C::STAGES) FP8BLK_STAMP(13);
#endif
        tc_fence_after_sync();
        const uint32_t col0 = static_cast<uint32_t>(pb * C::BN + group * C::kCpt);
        if constexpr (C::kSplitRegs) {
          // Two loads of 64 columns, one wait each; sc_lo scales the first 64
          // columns, sc_hi the second (w1 and w3 in SwiGLU mode).
#pragma unroll
          for (int h = 0; h < C::kCpt / FP8BLK_SPLIT_LD; ++h) {
            uint32_t v[FP8BLK_SPLIT_LD];
#if FP8BLK_SPLIT_LD == 64
            tmem_ld_32x32b_x64(t_lane + col0 + h * 64, v);
#else
            tmem_ld_32x32b_x32(t_lane + col0 + h * 32, v);
#endif
            const float sc = h * FP8BLK_SPLIT_LD < 64 ? sc_lo : sc_hi;
            const float2 sc2 = make_float2(sc, sc);
#pragma unroll
            for (int i = 0; i < FP8BLK_SPLIT_LD; i += 2) {
              const int j = h * FP8BLK_SPLIT_LD + i;
              const float2 r = __ffma2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), sc2,
                                          make_float2(acc[j], acc[j + 1]));
              acc[j] = r.x;
              acc[j + 1] = r.y;
            }
          }
        } else if constexpr (!C::SWAP && C::kCpt == 64) {
          // All 64 columns in one load and one wait, then packed f32x2 FMAs
          // (the same fp32 fma per element).
          uint32_t v[64];
          tmem_ld_32x32b_x64(t_lane + col0, v);
          const float2 sc2 = make_float2(sc_lo, sc_lo);
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            const float2 r = __ffma2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), sc2,
                                        make_float2(acc[i], acc[i + 1]));
            acc[i] = r.x;
            acc[i + 1] = r.y;
          }
        } else if constexpr (C::kCpt == 16 || C::EPI_WARPS == 8) {
          // 16-column loads: fewer live registers next to 128 accumulators
          // (ten warps leave 168 registers per thread).
#pragma unroll
          for (int ch = 0; ch < C::kCpt / 16; ++ch) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(t_lane + col0 + ch * 16, v);
            const float sc_h = (ch < C::kCpt / 32) ? sc_lo : sc_hi;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float sc =
                  C::SWAP ? __shfl_sync(0xFFFFFFFFu, sc_col[(ch * 16 + i) / 32], (ch * 16 + i) % 32) * w_row : sc_h;
              acc[ch * 16 + i] = fmaf(__uint_as_float(v[i]), sc, acc[ch * 16 + i]);
            }
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < C::kCpt / 32; ++ch) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_lane + col0 + ch * 32, v);
            const float sc_h = (ch < C::kCpt / 64) ? sc_lo : sc_hi;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float sc = C::SWAP ? __shfl_sync(0xFFFFFFFFu, sc_col[ch], i) * w_row : sc_h;
              acc[ch * 32 + i] = fmaf(__uint_as_float(v[i]), sc, acc[ch * 32 + i]);
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[pb]);
#ifdef FP8BLK_TRACE
        if (lane == 0 && ew == 0) FP8BLK_TL(5, ekb);
        if (lane == 0 && ew == C::EPI_WARPS - 1) FP8BLK_TL(7, ekb);
        ++ekb;
#endif
        FP8BLK_TOC(t_busy, t1);
        if (++pb == C::P) {
          pb = 0;
          pph ^= 1u;
        }
      }
      if (!ok) break;
      }
      FP8BLK_TIC(t2);
      if (ksplit > 1) {
        // Split-K cluster: park the partial in this CTA's (now idle) stage
        // ring as [column][lane]; the cluster reduces it after the roles end.
        float* part = reinterpret_cast<float*>(smem);
#pragma unroll
        for (int i = 0; i < C::kCpt; ++i) part[(group * C::kCpt + i) * 128 + row] = acc[i];
      } else if (u.nparts == 1) {
        ok = finalize<C>(prm, acc, t, group, row, xchg, unit_parity, epi_sync, out_slab, &tmap_col2);
      } else {
        // Stream-K fixup: publish this part, count arrivals, the last part sums.
        float* mine = prm.slots + static_cast<size_t>(2 * blockIdx.x + (u.part == 0 ? 1 : 0)) * (C::BN * 128);
#pragma unroll
        for (int i = 0; i < C::kCpt; ++i) __stcg(mine + (group * C::kCpt + i) * 128 + row, acc[i]);
        __threadfence();
        if (!epi_sync()) break;
        if (ew == 0 && lane == 0) {
          __threadfence();
          const int prev = atomicAdd(prm.counters + u.tile * C::CLUSTER + rank, 1);
          *last_flag = (prev == u.nparts - 1) ? 1 : 0;
        }
        if (!epi_sync()) break;
        if (*last_flag) {
          __threadfence();
          const int first = worker - u.part;
#pragma unroll
          for (int i = 0; i < C::kCpt; ++i) acc[i] = 0.0f;
          for (int q = 0; q < u.nparts; ++q) {
            const int cta = (first + q) * C::CLUSTER + rank;
            const float* src = prm.slots + static_cast<size_t>(2 * cta + (q == 0 ? 1 : 0)) * (C::BN * 128);
#pragma unroll
            for (int i = 0; i < C::kCpt; ++i) acc[i] += __ldcg(src + (group * C::kCpt + i) * 128 + row);
          }
          ok = finalize<C>(prm, acc, t, group, row, xchg, unit_parity, epi_sync, out_slab, &tmap_col2);
          if (ew == 0 && lane == 0) prm.counters[u.tile * C::CLUSTER + rank] = 0;
        }
      }
      FP8BLK_TOC(t_fin, t2);
      unit_parity ^= 1u;
    }
    if constexpr (C::kTmaStore) {
      if (lane == 0) bulk_wait_group0();  // every store written before the CTA exits
      __syncwarp();
    }
#ifdef FP8BLK_TRACE
    if (threadIdx.x == C::kEpiWarp0 * 32) {
      FP8BLK_PUT(21, tw_tfull);
      FP8BLK_PUT(22, t_busy);
      FP8BLK_PUT(23, t_fin);
    }
    if (threadIdx.x == C::kEpiWarp0 * 32 + 32 * 5) {  // a warp of the second column group
      FP8BLK_PUT(24, tw_tfull);
      FP8BLK_PUT(25, t_busy);
    }
#endif
  }

  if constexpr (C::SWAP) {
    if (ksplit > 1) {
      // Split-K reduction: CTA krank sums columns [krank, krank + 1) * BN / ksplit
      // of the tile over the ksplit partials, in rank order, and stores them.
      cluster_sync();  // every partial of the cluster is in shared memory
      if (warp >= C::kEpiWarp0) {
        const TileInfo t = tile_info<C>(prm, worker, grp_rows, grp_mtiles, 0);
        const int e = static_cast<int>(threadIdx.x) - C::kEpiWarp0 * 32;  // weight row of the tile
        const int n = t.lane_y + e;
        const int per = C::BN / ksplit;
        const float* part = reinterpret_cast<const float*>(smem);
        for (int jj = 0; jj < per; ++jj) {
          const int j = krank * per + jj;
          float sum = 0.0f;
          for (int q = 0; q < ksplit; ++q) sum += ld_shared_cluster_f32(part + j * 128 + e, static_cast<uint32_t>(q));
          const int m = t.col0 + j;
          if (m < prm.M && n < prm.N) prm.c[static_cast<size_t>(m) * prm.ldc + n] = __float2bfloat16_rn(sum);
        }
      }
      cluster_sync();  // no CTA leaves while a peer still reads its partial
    }
  }
  if (threadIdx.x == C::kEpiWarp0 * 32) FP8BLK_STAMP(8);
  tc_fence_before_sync();
  // Clusters: neither CTA leaves while its peer may still write its stages or
  // arrive on its barriers.
  if constexpr (C::CLUSTER > 1) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
  if (threadIdx.x == 0) FP8BLK_STAMP(9);
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

// 2-D bf16 output map for TMA stores: rows x cols (row stride cols * 2 bytes,
// a multiple of 16), boxes of 32 rows x 64 columns, 128-byte swizzled.
bool make_out_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Kernel variants. Non-swapped: BN = 256 (two epilogue warpgroups) or 128.
// Swapped (decode-sized M): BN = 16..128 token columns.
using CfgN256 = Cfg<256, false, 4, 2, 8>;
using CfgN256C2 = Cfg<256, false, 4, 2, 8, kEpiBf16, false, false, 2>;
// Large-M tiles of 128 x 128 with a four-deep TMEM ring and two column groups of
// 64: the promotion of one K block finishes while the next three are multiplied.
#ifndef FP8BLK_N128_STAGES
#define FP8BLK_N128_STAGES 6
#endif
using CfgN128E8 = Cfg<128, false, FP8BLK_N128_STAGES, 4, 8>;
// Large-M GEMMs run as CTA pairs (clusters of 2) unless built with
// -DFP8BLK_CLUSTER_PAIRS=0.
#ifndef FP8BLK_CLUSTER_PAIRS
#define FP8BLK_CLUSTER_PAIRS 1
#endif
#ifndef FP8BLK_DECODE_STAGES
#define FP8BLK_DECODE_STAGES 8
#endif
#ifndef FP8BLK_DECODE_P
#define FP8BLK_DECODE_P 8
#endif
#ifndef FP8BLK_SWAP_WHOLE_TILES
#define FP8BLK_SWAP_WHOLE_TILES 1
#endif
// Widest token tile that runs whole weight tiles (every swapped width: measured
// faster than stream-K at BN 16-128 for 86 to 768 weight tiles).
#ifndef FP8BLK_WHOLE_TILE_MAX_BN
#define FP8BLK_WHOLE_TILE_MAX_BN 128
#endif
#ifndef FP8BLK_DECODE_OCC
#define FP8BLK_DECODE_OCC 1
#endif
using CfgS16 = Cfg<16, true, FP8BLK_DECODE_STAGES, FP8BLK_DECODE_P, 4>;
using CfgS32 = Cfg<32, true, (FP8BLK_DECODE_STAGES > 10 ? 10 : FP8BLK_DECODE_STAGES), 8, 4>;
#ifndef FP8BLK_S64_STAGES
#define FP8BLK_S64_STAGES 6
#endif
using CfgS64 = Cfg<64, true, FP8BLK_S64_STAGES, 4, 4>;
using CfgS128 = Cfg<128, true, 6, 4, 4>;

// Fused w1/w3 GEMM with the SwiGLU + act_quant epilogue (dense and grouped),
// and the grouped GEMM whose rows are scattered back to token order.
using CfgSwiGLU = Cfg<256, false, 4, 2, 8, kEpiSwiGLU, false>;
using CfgSwiGLUC2 = Cfg<256, false, 4, 2, 8, kEpiSwiGLU, false, false, 2>;
using CfgSwiGLUGrouped = Cfg<256, false, 4, 2, 8, kEpiSwiGLU, true>;
using CfgScatterGrouped = Cfg<256, false, 4, 2, 8, kEpiScatter, true>;
// The same large-M tiles with power-of-two scales applied by the tensor core
// (one TMEM accumulator per tile, no promotion).
using CfgN256MX = Cfg<256, false, 4, 1, 8, kEpiBf16, false, false, 1, true>;
using CfgN256C2MX = Cfg<256, false, 4, 1, 8, kEpiBf16, false, false, 2, true>;
using CfgSwiGLUMX = Cfg<256, false, 4, 1, 8, kEpiSwiGLU, false, false, 1, true>;
using CfgSwiGLUC2MX = Cfg<256, false, 4, 1, 8, kEpiSwiGLU, false, false, 2, true>;
using CfgSwiGLUGroupedMX = Cfg<256, false, 4, 1, 8, kEpiSwiGLU, true, false, 1, true>;
using CfgScatterGroupedMX = Cfg<256, false, 4, 1, 8, kEpiScatter, true, false, 1, true>;

// UE8M0 scales take the tensor-core scaled kernels (MX) unless the call adds
// FP8BLK_SCALE_PROMOTE; that keeps the per-block promotion, which computes the
// same numbers in another summation order.
bool mx_for(int scale_fmt) { return scale_fmt_mx(scale_fmt); }
// Decode linear with the act_quant fused in (M <= 16): weights-only stages.
using CfgF16S8 = Cfg<16, true, 8, 8, 4, kEpiBf16, false, true>;
using CfgF16S4 = Cfg<16, true, 4, 8, 4, kEpiBf16, false, true>;

constexpr int kMaxDynSmem = 232448;
#ifndef FP8BLK_SMEM_CARVEOUT
#define FP8BLK_SMEM_CARVEOUT 100  // percent of the unified L1 / shared memory (-1: the driver's choice)
#endif

struct Plan {
  int bn;
  bool swap;
  int cluster;  // CTAs per schedule worker (2: lane-tile pairs); grid counts workers
  int ksplit;   // > 1: split-K clusters of that many CTAs per tile; grid counts CTAs
  int tiles_lane, tiles_col;
  int grid, dp_waves, sk_tiles;
  long long sk_iters;
  int whole_tiles;  // > 0: that many tiles, whole and round-robin (no stream-K, no counters)
};

// Arrival counters of the stream-K fixup: a fixed region at the start of
// every GEMM workspace, so that when one workspace serves GEMMs of different
// shapes, no plan's partial slots (which follow the region) overlap another
// plan's counters. A plan with more tiles than counters runs whole tiles.
constexpr size_t kCounterBytes = 64 * 1024;
constexpr long long kMaxCounters = static_cast<long long>(kCounterBytes / sizeof(int));

// Data-parallel waves while at least two full waves remain, stream-K for the rest.
void plan_schedule(Plan& pl, int64_t Kb, int sm_count) {
  const long long tiles = static_cast<long long>(pl.tiles_lane) * pl.tiles_col;
  const int G = sm_count;
  if (tiles * pl.cluster > kMaxCounters) {
    pl.grid = G;
    pl.dp_waves = 0;
    pl.sk_tiles = 0;
    pl.sk_iters = 0;
    pl.whole_tiles = static_cast<int>(tiles);
    return;
  }
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
}

// Dense large-M tiles: whole tiles round-robin over the workers unless
// splitting K (stream-K) shortens the busiest worker by more than
// kStreamKSlackKb K blocks; the stream-K fixup (partials to memory, arrival
// counters, the last part's reduction) costs about that much. Measured at
// 256-4096 rows: whole tiles 1.1-1.6x faster where the uneven last round is
// short (e.g. 512 x 7168 x 2048 21.1 -> 13.5 us), stream-K ahead where it
// saves 41 or more K blocks (2048 x 1536 x 7168, 4096 x 18432 x 7168).
constexpr long long kStreamKSlackKb = 32;

void plan_dense_schedule(Plan& pl, int64_t Kb, int workers) {
  const long long tiles = static_cast<long long>(pl.tiles_lane) * pl.tiles_col;
  const long long rounds = (tiles + workers - 1) / workers;
  // (More tiles than counters always run whole: plan_schedule. Below that the
  // products stay far inside 64 bits.)
  if (tiles * pl.cluster <= kMaxCounters && rounds * Kb * workers - tiles * Kb <= kStreamKSlackKb * workers) {
    pl.grid = static_cast<int>(tiles < workers ? tiles : workers);
    pl.dp_waves = 0;
    pl.sk_tiles = 0;
    pl.sk_iters = 0;
    pl.whole_tiles = static_cast<int>(tiles);
    return;
  }
  plan_schedule(pl, Kb, workers);
}

// Co-resident clusters of 2, 4 and 8 CTAs of the swapped kernel a plan would
// launch (index 1, 2, 3); zero where none fit.
struct SplitCaps {
  int clusters[4];
};

int swap_bn(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

// pair_workers: co-resident CTA pairs of the cluster kernel (0: no clusters).
// caps: split-K cluster capacity of the swapped kernel (null: no split-K).
Plan make_plan(int64_t M, int64_t N, int64_t K, int sm_count, int pair_workers, const SplitCaps* caps) {
  Plan pl{};
  pl.cluster = 1;
  pl.ksplit = 1;
  if (M <= 128) {
    pl.swap = true;
    pl.bn = swap_bn(M);
    pl.tiles_lane = static_cast<int>((N + 127) / 128);
    pl.tiles_col = static_cast<int>((M + pl.bn - 1) / pl.bn);
    const long long tiles = static_cast<long long>(pl.tiles_lane) * pl.tiles_col;
    if (FP8BLK_SWAP_WHOLE_TILES && pl.bn <= FP8BLK_WHOLE_TILE_MAX_BN && 2 * tiles >= sm_count) {
      // CTAs stream whole weight tiles, one per CTA up to one per SM and then
      // round-robin: no stream-K fixup, which costs a decode launch more than
      // an uneven last round of tiles (measured from 160 to 768 tiles).
      if (tiles <= sm_count) {
        pl.grid = static_cast<int>(tiles);
        pl.dp_waves = 1;
      } else {
        pl.grid = sm_count;
        pl.dp_waves = 0;
        pl.whole_tiles = static_cast<int>(tiles);
      }
      pl.sk_tiles = 0;
      pl.sk_iters = 0;
      return pl;
    }
    // Few weight tiles: a cluster of ks CTAs per tile, each one K slice, the
    // partials reduced in distributed shared memory (no global fixup).
    if (caps && 2 * tiles < sm_count) {
      const int64_t Kb = K / kBlock;
      for (int ks = 8, idx = 3; ks >= 2; ks >>= 1, --idx) {
        if (Kb >= 2 * ks && tiles * ks <= sm_count && tiles <= caps->clusters[idx]) {
          pl.ksplit = ks;
          pl.grid = static_cast<int>(tiles * ks);
          pl.dp_waves = 1;
          pl.sk_tiles = 0;
          pl.sk_iters = 0;
          return pl;
        }
      }
    }
    if (pl.bn <= 32) {
      plan_schedule(pl, K / kBlock, sm_count * FP8BLK_DECODE_OCC);
      return pl;
    }
  } else {
    pl.swap = false;
    // 128 x 128 tiles (four TMEM partials) where 128 x 256 tiles would be too
    // few to fill the machine twice, or too short (K <= 512) for two partials
    // to carry the MMA of the next tile past the current tile's epilogue.
    const int64_t tiles256 = ((M + 127) / 128) * ((N + 255) / 256);
    pl.bn = (N <= 128 || K / kBlock <= 4 || tiles256 < 2LL * sm_count) ? 128 : 256;
    pl.tiles_lane = static_cast<int>((M + 127) / 128);
    pl.tiles_col = static_cast<int>((N + pl.bn - 1) / pl.bn);
    if (pl.bn == 256 && pair_workers > 0) {
      pl.cluster = 2;
      pl.tiles_lane = (pl.tiles_lane + 1) / 2;
      plan_dense_schedule(pl, K / kBlock, pair_workers);
      return pl;
    }
    plan_dense_schedule(pl, K / kBlock, sm_count);
    return pl;
  }
  plan_schedule(pl, K / kBlock, sm_count);
  return pl;
}

// The fused w1/w3 GEMM: 128 activation rows x 128 output columns per tile
// (MMA N = 256: 128 columns of w1 and the same 128 of w3).
Plan make_swiglu_plan(int64_t M, int64_t inter, int64_t K, int sm_count, int pair_workers) {
  Plan pl{};
  pl.swap = false;
  pl.bn = 256;
  pl.cluster = pair_workers > 0 ? 2 : 1;
  pl.tiles_lane = static_cast<int>((M + 127) / 128);
  pl.tiles_lane = (pl.tiles_lane + pl.cluster - 1) / pl.cluster;
  pl.tiles_col = static_cast<int>(inter / 128);
  plan_dense_schedule(pl, K / kBlock, pair_workers > 0 ? pair_workers : sm_count);
  return pl;
}


// Scale rows of Kb floats load FP8BLK_SCALE_VEC at a time when every row of
// each array starts on that many floats' boundary.
int vec_scales_ok(int Kb, const float* a, const float* b, const float* c) {
  const int q = FP8BLK_SCALE_VEC;
  return q > 1 && Kb % q == 0 && is_aligned(a, 4u * q) && is_aligned(b, 4u * q) && is_aligned(c, 4u * q) ? 1 : 0;
}

// Workspace: the counter region (one arrival counter per output tile), then,
// for plans that cut tiles stream-K, two partial slots per CTA. Plans of whole
// tiles, weight slices or split-K clusters write no partial sums to memory.
size_t plan_counter_bytes(const Plan&) { return kCounterBytes; }

size_t plan_workspace(const Plan& pl) {
  const size_t slots = pl.sk_tiles > 0 ? static_cast<size_t>(2) * pl.grid * pl.cluster * pl.bn * 128 * sizeof(float) : 0;
  return plan_counter_bytes(pl) + slots;
}

template <class C>
int launch(const DevInfo* d, const CUtensorMap& ml, const CUtensorMap& mc, const CUtensorMap& mc2,
           const GemmParams& prm, cudaStream_t stream, size_t extra_smem = 0, int kcluster = 1) {
  static bool attr_done[64] = {};
  auto kern = fp8_gemm_kernel<C>;
  const int smem_attr = C::FUSED ? kMaxDynSmem : C::kSmemBytes;
  if (d->device >= 64 || !attr_done[d->device]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_attr) != cudaSuccess)
      return FP8BLK_ERR_CUDA;
    // All of the unified L1 / shared memory as shared memory: the kernels
    // stage through shared memory, and a CTA of the next launch can then sit
    // beside a running one wherever their shared memory fits.
    if (FP8BLK_SMEM_CARVEOUT >= 0 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, FP8BLK_SMEM_CARVEOUT) !=
            cudaSuccess)
      return FP8BLK_ERR_CUDA;
    if constexpr (C::kSplitRegs) {
      // setmaxnreg.inc would wait forever if the build gave the kernel fewer
      // registers per thread than the split hands out: refuse to launch.
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs < C::kLaunchRegs) return FP8BLK_ERR_CUDA;
    }
    if (d->device < 64) attr_done[d->device] = true;
  }
#ifdef FP8BLK_TRACE
  static int trace_counter = 0;
  const_cast<GemmParams&>(prm).trace_id = trace_counter++ & 7;
#endif
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(prm.grid * C::CLUSTER));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes + extra_smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C::CLUSTER > 1 ? C::CLUSTER : kcluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (C::CLUSTER > 1 || kcluster > 1) ? 2 : 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, ml, mc, mc2, prm));
}

// How many clusters of C fit on the device at once (0 if none, or if clusters
// are disabled): the persistent schedule's worker count. Cached per device.
template <class C>
int cluster_workers(const DevInfo* d) {
  if (!FP8BLK_CLUSTER_PAIRS) return 0;
  static int cached[64] = {};
  if (d->device < 64 && cached[d->device] != 0) return cached[d->device] > 0 ? cached[d->device] : 0;
  int n = 0;
  auto kern = fp8_gemm_kernel<C>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(d->sm_count));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      n = 0;
      cudaGetLastError();  // the query's error is not the caller's
    }
  }
  if (d->device < 64) cached[d->device] = n > 0 ? n : -1;
  return n > 0 ? n : 0;
}

// Co-resident clusters of `size` CTAs of kernel C (0 if none or on error).
template <class C>
int max_clusters(const DevInfo* d, int size) {
  auto kern = fp8_gemm_kernel<C>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((d->sm_count / size) * size));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <class C>
SplitCaps split_caps_of(const DevInfo* d) {
  SplitCaps c{};
  c.clusters[1] = max_clusters<C>(d, 2);
  c.clusters[2] = max_clusters<C>(d, 4);
  c.clusters[3] = max_clusters<C>(d, 8);
  return c;
}

// Split-K capacity of the swapped kernel for M tokens, cached per device.
const SplitCaps* split_caps(const DevInfo* d, int64_t M) {
  static SplitCaps cache[64][4];
  static bool done[64][4] = {};
  const int bn = swap_bn(M);
  const int bi = bn == 16 ? 0 : bn == 32 ? 1 : bn == 64 ? 2 : 3;
  if (d->device >= 64) return nullptr;
  if (!done[d->device][bi]) {
    cache[d->device][bi] = bi == 0 ? split_caps_of<CfgS16>(d)
                           : bi == 1 ? split_caps_of<CfgS32>(d)
                           : bi == 2 ? split_caps_of<CfgS64>(d)
                                     : split_caps_of<CfgS128>(d);
    done[d->device][bi] = true;
  }
  return &cache[d->device][bi];
}

}  // namespace

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 256;
  const DevInfo* d;
  if (current_device(&d) != FP8BLK_OK) return plan_workspace(make_plan(M, N, K, 256, 0, nullptr));
  return plan_workspace(make_plan(M, N, K, d->sm_count, cluster_workers<CfgN256C2>(d), split_caps(d, M)));
}

// The argument checks of fp8_gemm, in order: FP8BLK_OK when they pass (an
// empty problem, M == 0 or N == 0, passes without its pointers being looked
// at; K == 0 needs only c).
int gemm_check_args(const void* a, const float* a_s, const void* w, const float* w_s, const void* c, int64_t M,
                    int64_t N, int64_t K, int scale_fmt) {
  if (!scale_fmt_valid(scale_fmt)) return FP8BLK_ERR_ARG;
  if (M < 0 || N < 0 || K < 0 || K % kBlock != 0) return FP8BLK_ERR_SHAPE;
  if (M > (int64_t{1} << 31) - 1 || N > (int64_t{1} << 31) - 1 || K > (int64_t{1} << 31) - 1)
    return FP8BLK_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8BLK_OK;
  if (!c) return FP8BLK_ERR_NULL;
  if (!is_aligned(c, 2)) return FP8BLK_ERR_ALIGN;
  if (K == 0) return FP8BLK_OK;
  if (!a || !a_s || !w || !w_s) return FP8BLK_ERR_NULL;
  if (!is_aligned(a, 16) || !is_aligned(w, 16) || !is_aligned(a_s, 4) || !is_aligned(w_s, 4))
    return FP8BLK_ERR_ALIGN;
  return FP8BLK_OK;
}

int decode_gemm_run(const DevInfo* dev, const void* a, const float* a_s, const void* w, const float* w_s, void* c,
                    int64_t M, int64_t N, int64_t K, cudaStream_t stream, bool* used);

int gemm_run(const void* a, const float* a_s, const void* w, const float* w_s, void* c, int64_t M, int64_t N,
             int64_t K, int scale_fmt, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (int st = gemm_check_args(a, a_s, w, w_s, c, M, N, K, scale_fmt)) return st;
  if (M == 0 || N == 0) return FP8BLK_OK;
  if (K == 0) return cuda_status(cudaMemsetAsync(c, 0, static_cast<size_t>(M) * N * 2, stream));
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  const Plan pl = make_plan(M, N, K, d->sm_count, cluster_workers<CfgN256C2>(d), split_caps(d, M));
  const size_t need = plan_workspace(pl);
  if (!workspace || workspace_bytes < need) return FP8BLK_ERR_WORKSPACE;
  if (!is_aligned(workspace, 256)) return FP8BLK_ERR_ALIGN;
  // Up to 16 tokens, when a CTA's weight slice fits in shared memory: the
  // slice-per-SM decode kernel (no workspace used).
  {
    bool used = false;
    const int st = decode_gemm_run(d, a, a_s, w, w_s, c, M, N, K, stream, &used);
    if (st || used) return st;
  }

  GemmParams prm{};
  prm.a_s = a_s;
  prm.w_s = w_s;
  prm.c = static_cast<__nv_bfloat16*>(c);
  prm.counters = static_cast<int*>(workspace);
  prm.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan_counter_bytes(pl));
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
  prm.whole_tiles = pl.whole_tiles;
  prm.ksplit = pl.ksplit;
  prm.vec_store = (N % 8 == 0 && is_aligned(c, 16)) ? 1 : 0;
  prm.vec_scales = vec_scales_ok(prm.Kb, a_s, w_s, w_s);
  prm.ldc = static_cast<int>(N);

  CUtensorMap ml, mc;
  const void* lane_src = pl.swap ? w : a;
  const void* col_src = pl.swap ? a : w;
  const uint64_t lane_rows = static_cast<uint64_t>(pl.swap ? N : M);
  const uint64_t col_rows = static_cast<uint64_t>(pl.swap ? M : N);
  // Cluster pairs load the column tile in two 128-row halves.
  const uint32_t col_box = static_cast<uint32_t>(pl.cluster == 2 ? 128 : pl.bn);
  if (!make_kmajor_map(&ml, lane_src, lane_rows, static_cast<uint64_t>(K), 128) ||
      !make_kmajor_map(&mc, col_src, col_rows, static_cast<uint64_t>(K), col_box))
    return FP8BLK_ERR_CUDA;

  if (!pl.swap) {
    const bool mx = mx_for(scale_fmt);
    // C through TMA stores: boxes of 32 rows x 64 columns, rows of N bf16.
    CUtensorMap mo = mc;
    if (prm.vec_store && make_out_map(&mo, c, static_cast<uint64_t>(M), static_cast<uint64_t>(N))) prm.tma_store = 1;
    if (pl.cluster == 2)
      return mx ? launch<CfgN256C2MX>(d, ml, mc, mo, prm, stream) : launch<CfgN256C2>(d, ml, mc, mo, prm, stream);
    if (pl.bn == 256)
      return mx ? launch<CfgN256MX>(d, ml, mc, mo, prm, stream) : launch<CfgN256>(d, ml, mc, mo, prm, stream);
    return launch<CfgN128E8>(d, ml, mc, mo, prm, stream);
  }
  switch (pl.bn) {
    case 16: return launch<CfgS16>(d, ml, mc, mc, prm, stream, 0, pl.ksplit);
    case 32: return launch<CfgS32>(d, ml, mc, mc, prm, stream, 0, pl.ksplit);
    case 64: return launch<CfgS64>(d, ml, mc, mc, prm, stream, 0, pl.ksplit);
    default: return launch<CfgS128>(d, ml, mc, mc, prm, stream, 0, pl.ksplit);
  }
}

namespace {

bool scale_fmt_ok(int f) { return scale_fmt_valid(f); }

}  // namespace

// Decode FP8 linear (M <= 16) in one kernel: act_quant of x inside the GEMM
// CTAs, whole 128-row weight tiles per CTA. Sets *used = false (and launches
// nothing) when the shape does not fit the fused kernel's shared memory; the
// caller then runs act_quant + fp8_gemm.
namespace {

// Which fused kernel takes the shape: 0 (8 weight stages), 1 (4 stages), or
// -1 (none: the resident activation operand does not fit).
int linear_fused_variant(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || M > 16 || N < 1 || K < kBlock || K % kBlock || N > (int64_t{1} << 31) - 1 || K > (int64_t{1} << 24))
    return -1;
  const size_t extra = fused_extra_bytes(static_cast<int>(K / kBlock), 16);
  return CfgF16S8::kSmemBytes + extra <= kMaxDynSmem ? 0 : CfgF16S4::kSmemBytes + extra <= kMaxDynSmem ? 1 : -1;
}

}  // namespace

bool linear_fused_fits(int64_t M, int64_t N, int64_t K) { return linear_fused_variant(M, N, K) >= 0; }

int linear_fused_run(const void* x, const void* w, const float* w_s, void* y, int64_t M, int64_t N, int64_t K,
                     int scale_fmt, cudaStream_t stream, bool* used) {
  *used = false;
  if (!scale_fmt_ok(scale_fmt)) return FP8BLK_ERR_ARG;
  const int variant = linear_fused_variant(M, N, K);
  if (variant < 0) return FP8BLK_OK;
  if (!x || !w || !w_s || !y) return FP8BLK_ERR_NULL;
  if (!is_aligned(x, 16) || !is_aligned(w, 16) || !is_aligned(w_s, 4) || !is_aligned(y, 2)) return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  const int Kb = static_cast<int>(K / kBlock);
  const size_t extra = fused_extra_bytes(Kb, 16);
  GemmParams prm{};
  prm.w_s = w_s;
  prm.c = static_cast<__nv_bfloat16*>(y);
  prm.x = static_cast<const __nv_bfloat16*>(x);
  prm.err = d->err_word;
  prm.M = static_cast<int>(M);
  prm.N = static_cast<int>(N);
  prm.Kb = Kb;
  prm.n_wblocks = static_cast<int>((N + 127) / 128);
  prm.ldc = static_cast<int>(N);
  prm.tiles_lane = prm.n_wblocks;
  prm.tiles_col = 1;
  prm.whole_tiles = prm.n_wblocks;
  prm.grid = prm.n_wblocks < d->sm_count ? prm.n_wblocks : d->sm_count;
  prm.ue8m0 = scale_fmt_ue8m0(scale_fmt);
  CUtensorMap ml;
  if (!make_kmajor_map(&ml, w, static_cast<uint64_t>(N), static_cast<uint64_t>(K), 128)) return FP8BLK_ERR_CUDA;
  *used = true;
  return variant == 0 ? launch<CfgF16S8>(d, ml, ml, ml, prm, stream, extra)
                      : launch<CfgF16S4>(d, ml, ml, ml, prm, stream, extra);
}

size_t swiglu_workspace_bytes(int64_t M, int64_t inter, int64_t K) {
  if (M <= 0 || inter <= 0 || K <= 0) return 256;
  const DevInfo* d;
  if (current_device(&d) != FP8BLK_OK) return plan_workspace(make_swiglu_plan(M, inter, K, 256, 0));
  return plan_workspace(make_swiglu_plan(M, inter, K, d->sm_count, cluster_workers<CfgSwiGLUC2>(d)));
}

// u = act_quant(bf16(silu(bf16(x w1^T))) * bf16(x w3^T)) in one kernel.
int swiglu_run(const void* xq, const float* xs, const void* w1, const float* w1s, const void* w3, const float* w3s,
               void* uq, float* us, int64_t M, int64_t inter, int64_t K, int scale_fmt, void* workspace,
               size_t workspace_bytes, cudaStream_t stream) {
  if (!scale_fmt_ok(scale_fmt)) return FP8BLK_ERR_ARG;
  const int64_t lim = (int64_t{1} << 31) - 1;
  if (M < 0 || inter < 0 || K <= 0 || K % kBlock || inter % kBlock || M > lim || inter > lim || K > lim)
    return FP8BLK_ERR_SHAPE;
  if (M == 0 || inter == 0) return FP8BLK_OK;
  if (!xq || !xs || !w1 || !w1s || !w3 || !w3s || !uq || !us) return FP8BLK_ERR_NULL;
  if (!is_aligned(xq, 16) || !is_aligned(w1, 16) || !is_aligned(w3, 16) || !is_aligned(uq, 16) ||
      !is_aligned(xs, 4) || !is_aligned(w1s, 4) || !is_aligned(w3s, 4) || !is_aligned(us, 4))
    return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  const Plan pl = make_swiglu_plan(M, inter, K, d->sm_count, cluster_workers<CfgSwiGLUC2>(d));
  if (!workspace || workspace_bytes < plan_workspace(pl)) return FP8BLK_ERR_WORKSPACE;
  if (!is_aligned(workspace, 256)) return FP8BLK_ERR_ALIGN;
  GemmParams prm{};
  prm.a_s = xs;
  prm.w_s = w1s;
  prm.w3_s = w3s;
  prm.uq = static_cast<uint8_t*>(uq);
  prm.us = us;
  prm.counters = static_cast<int*>(workspace);
  prm.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan_counter_bytes(pl));
  prm.err = d->err_word;
  prm.M = static_cast<int>(M);
  prm.N = static_cast<int>(inter);
  prm.Kb = static_cast<int>(K / kBlock);
  prm.n_wblocks = static_cast<int>(inter / kBlock);
  prm.ldc = static_cast<int>(inter);
  prm.tiles_lane = pl.tiles_lane;
  prm.tiles_col = pl.tiles_col;
  prm.grid = pl.grid;
  prm.dp_waves = pl.dp_waves;
  prm.sk_tiles = pl.sk_tiles;
  prm.sk_iters = pl.sk_iters;
  prm.whole_tiles = pl.whole_tiles;
  prm.ue8m0 = scale_fmt_ue8m0(scale_fmt);
  prm.vec_scales = 0;  // one K block at a time in the SwiGLU epilogue
  CUtensorMap ml, m1, m3;
  if (!make_kmajor_map(&ml, xq, static_cast<uint64_t>(M), static_cast<uint64_t>(K), 128) ||
      !make_kmajor_map(&m1, w1, static_cast<uint64_t>(inter), static_cast<uint64_t>(K), 64) ||
      !make_kmajor_map(&m3, w3, static_cast<uint64_t>(inter), static_cast<uint64_t>(K), 64))
    return FP8BLK_ERR_CUDA;
  if (mx_for(scale_fmt))
    return pl.cluster == 2 ? launch<CfgSwiGLUC2MX>(d, ml, m1, m3, prm, stream)
                           : launch<CfgSwiGLUMX>(d, ml, m1, m3, prm, stream);
  if (pl.cluster == 2) return launch<CfgSwiGLUC2>(d, ml, m1, m3, prm, stream);
  return launch<CfgSwiGLU>(d, ml, m1, m3, prm, stream);
}

// Grouped fused w1/w3 GEMM over rows sorted by group: group e owns rows
// [grp_rows[e], grp_rows[e+1]) of xg and weight rows [e*inter, (e+1)*inter)
// of w1 and w3. grp_rows / grp_mtiles are device arrays of E + 1 entries.
int grouped_swiglu_run(const void* xg, const float* xgs, const void* w1, const float* w1s, const void* w3,
                       const float* w3s, void* uq, float* us, int64_t rows, int64_t E, int64_t inter, int64_t K,
                       const int* grp_rows, const int* grp_mtiles, int scale_fmt, cudaStream_t stream) {
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  GemmParams prm{};
  prm.a_s = xgs;
  prm.w_s = w1s;
  prm.w3_s = w3s;
  prm.uq = static_cast<uint8_t*>(uq);
  prm.us = us;
  prm.grp_rows = grp_rows;
  prm.grp_mtiles = grp_mtiles;
  prm.err = d->err_word;
  prm.M = static_cast<int>(rows);
  prm.N = static_cast<int>(inter);
  prm.Kb = static_cast<int>(K / kBlock);
  prm.ldc = static_cast<int>(inter);
  prm.E = static_cast<int>(E);
  prm.tiles_col = static_cast<int>(inter / 128);
  prm.grid = d->sm_count;
  prm.ue8m0 = scale_fmt_ue8m0(scale_fmt);
  prm.vec_scales = 0;
  CUtensorMap ml, m1, m3;
  if (!make_kmajor_map(&ml, xg, static_cast<uint64_t>(rows), static_cast<uint64_t>(K), 128) ||
      !make_kmajor_map(&m1, w1, static_cast<uint64_t>(E * inter), static_cast<uint64_t>(K), 64) ||
      !make_kmajor_map(&m3, w3, static_cast<uint64_t>(E * inter), static_cast<uint64_t>(K), 64))
    return FP8BLK_ERR_CUDA;
  if (mx_for(scale_fmt)) return launch<CfgSwiGLUGroupedMX>(d, ml, m1, m3, prm, stream);
  return launch<CfgSwiGLUGrouped>(d, ml, m1, m3, prm, stream);
}

// Grouped GEMM (w2) whose output row r goes to out[perm[r]]: group e's rows
// times weight rows [e*dim, (e+1)*dim) of w2 [E*dim, inter]; dim % 256 == 0.
int grouped_scatter_run(const void* uq, const float* us, const void* w2, const float* w2s, void* out,
                        const int* perm, int64_t rows, int64_t E, int64_t dim, int64_t inter, const int* grp_rows,
                        const int* grp_mtiles, int scale_fmt, cudaStream_t stream) {
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  GemmParams prm{};
  prm.a_s = us;
  prm.w_s = w2s;
  prm.c = static_cast<__nv_bfloat16*>(out);
  prm.perm = perm;
  prm.grp_rows = grp_rows;
  prm.grp_mtiles = grp_mtiles;
  prm.err = d->err_word;
  prm.M = static_cast<int>(rows);
  prm.N = static_cast<int>(dim);
  prm.Kb = static_cast<int>(inter / kBlock);
  prm.ldc = static_cast<int>(dim);
  prm.E = static_cast<int>(E);
  prm.tiles_col = static_cast<int>(dim / 256);
  prm.grid = d->sm_count;
  prm.vec_store = (dim % 8 == 0 && is_aligned(out, 16)) ? 1 : 0;
  prm.vec_scales = 0;
  CUtensorMap ml, mc;
  if (!make_kmajor_map(&ml, uq, static_cast<uint64_t>(rows), static_cast<uint64_t>(inter), 128) ||
      !make_kmajor_map(&mc, w2, static_cast<uint64_t>(E * dim), static_cast<uint64_t>(inter), 256))
    return FP8BLK_ERR_CUDA;
  if (mx_for(scale_fmt)) return launch<CfgScatterGroupedMX>(d, ml, mc, mc, prm, stream);
  return launch<CfgScatterGrouped>(d, ml, mc, mc, prm, stream);
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

}  // namespace
}  // namespace fp8blk

extern "C" int fp8blk_gemm_noalloc(const void* a_e4m3, const float* a_s, const void* w_e4m3, const float* w_s,
                                   void* c_bf16, int64_t M, int64_t N, int64_t K, int scale_fmt,
                                   fp8blk_stream_t stream) {
  using namespace fp8blk;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // fp8blk_gemm's argument checks come first, so a rejected call returns the
  // same status as fp8blk_gemm would and neither clears nor launches anything.
  if (int st = gemm_check_args(a_e4m3, a_s, w_e4m3, w_s, c_bf16, M, N, K, scale_fmt)) return st;
  // Empty and zero-K problems need no scratch.
  if (M == 0 || N == 0 || K == 0)
    return gemm_run(a_e4m3, a_s, w_e4m3, w_s, c_bf16, M, N, K, scale_fmt, nullptr, 0, cs);
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  const Plan pl = make_plan(M, N, K, d->sm_count, cluster_workers<CfgN256C2>(d), split_caps(d, M));
  if (plan_workspace(pl) > FP8BLK_NOALLOC_SCRATCH_BYTES) return FP8BLK_ERR_TOO_LARGE;
  void* scratch = nullptr;
  if (int st = noalloc_scratch(d->device, &scratch)) return st;
  if (cudaMemsetAsync(scratch, 0, plan_counter_bytes(pl), cs) != cudaSuccess) return FP8BLK_ERR_CUDA;
  return gemm_run(a_e4m3, a_s, w_e4m3, w_s, c_bf16, M, N, K, scale_fmt, scratch, FP8BLK_NOALLOC_SCRATCH_BYTES, cs);
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

#ifdef FP8BLK_TRACE
// Phase-trace reader (trace builds only): copies n stamps (kTraceSlots per CTA) to host.
extern "C" __attribute__((visibility("default"))) int fp8trace_read(unsigned long long* host, int n) {
  return cudaMemcpyFromSymbol(host, fp8blk::g_trace, sizeof(unsigned long long) * n) == cudaSuccess ? 0 : 1;
}
extern "C" __attribute__((visibility("default"))) int fp8trace_timeline(long long* host) {
  return cudaMemcpyFromSymbol(host, fp8blk::g_timeline, sizeof(fp8blk::g_timeline)) == cudaSuccess ? 0 : 1;
}
extern "C" __attribute__((visibility("default"))) int fp8trace_clear(void) {
  static unsigned long long zeros[8 * 4096 * fp8blk::kTraceSlots];
  return cudaMemcpyToSymbol(fp8blk::g_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : 1;
}
#endif
