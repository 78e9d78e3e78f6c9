// MLA "absorb" projections with the FP8 wkv_b weight ("Administrator &
// Developer Guide", 8.3 steps 5 and 7): per head h,
//   qk: out[t, h, c] = sum_d q_nope[t, h, d] * W[h (dn + dv) + d, c]        (K = dn, N = C)
//   v:  out[t, h, d] = sum_c x[t, h, c]      * W[h (dn + dv) + dn + d, c]   (K = C,  N = dv)
// where W is wkv_b as weight_dequant gives it (bf16 of the fp32 code times its
// 128 x 128 block scale, 8.5.2), activations and outputs are bf16, and the
// sum is fp32 (a bf16 product accumulated in fp32).
//
// The tensor cores take bf16 x bf16 (tcgen05.mma kind::f16, both operands
// bf16): the FP8 weight tile is TMA-loaded as bytes, dequantised row by row by
// four warps into a bf16 128-byte-swizzled tile in shared memory, and fed to
// the MMA next to the TMA-loaded bf16 activation tile. W's rows are the N
// dimension for v (a K-major operand) and the K dimension for qk (W keeps its
// layout and is read as an MN-major operand, so no transpose). Persistent
// CTAs, one per SM, walk the tiles of (head, 128-token tile, 128-column
// tile); a tile's fp32 accumulator stays in TMEM over its whole K (no
// per-block promotion: the block scale is inside the dequantised weight), in
// one of two buffers, so a tile's stores overlap the next tile's loads,
// dequantisation and MMAs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fp8blk.h"
#include "host.cuh"
#include "ptx.cuh"

namespace fp8blk {
namespace {

// Warps: 0 activation TMA, 1 MMA, 2-5 and 11-14 dequant, 6-9 epilogue, 10 weight TMA.
constexpr int kMlaThreads = 480;
constexpr int kDequantWarps = 8;
constexpr int kAHalf = 128 * 128;                // 128 rows x 64 bf16 (one 128-byte swizzled half)
constexpr int kATile = 2 * kAHalf;               // 128 token rows x 128 bf16
constexpr int kB8Tile = 128 * 128;               // 128 x 128 e4m3
constexpr int kB16Tile = 2 * kAHalf;             // the dequantised weight tile, K-major, two halves
// The epilogue's staging tile: per epilogue warp, its 32 output rows x 128
// bf16 as two 64-column halves of 32 rows x 128 bytes, 128-byte swizzled (the
// TMA store's box).
constexpr int kOutHalf = 32 * 128;
constexpr int kOutWarp = 2 * kOutHalf;
constexpr int kOutBytes = 4 * kOutWarp;
// Three rings, one entry per (tile, K block) step: activation tiles (freed by
// the MMAs), e4m3 weight tiles (freed once dequantised) and bf16 weight tiles
// (freed by the MMAs). The weight stream runs ahead of the MMAs by up to
// kWRing + kBRing steps, the activation stream by kARing.
constexpr int kARing = 3, kWRing = 2, kBRing = 2;
constexpr int kOffW = kARing * kATile;
constexpr int kOffB = kOffW + kWRing * kB8Tile;
constexpr int kOffO = kOffB + kBRing * kB16Tile;
constexpr int kOffBar = kOffO + kOutBytes;
constexpr int kNumBars = 2 * (kARing + kWRing + kBRing) + 4 + 1;
constexpr int kMlaSmem = 1024 + kOffBar + kNumBars * 8 + 16;
static_assert(kMlaSmem <= 232448, "shared memory per CTA");
constexpr unsigned kDevErrTimeoutMla = 1u << 6;

// Shared-memory matrix descriptor for an MN-major operand tile with 128-byte
// swizzling: each 128-byte row holds 64 consecutive M/N elements (16-bit) of
// one K index, 8 K rows form a 1024-byte swizzle atom; `lbo` is the byte
// stride between 64-element blocks along M/N, `sbo` the byte stride between
// 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// The issuing thread's bulk stores, all but the most recent group, have read
// their shared-memory sources.
__device__ __forceinline__ void bulk_wait_group_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// kind::f16 instruction descriptor: f32 accumulator, A and B both bf16 (one
// value sets both format fields), A K-major, B K-major or (b_mn) MN-major
// (bit 16), an M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool b_mn) {
  constexpr uint32_t kBf16 = 1;
  return (1u << 4) | (kBf16 << 7) | (kBf16 << 10) | (b_mn ? 1u << 16 : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one 32-byte (16 x bf16) K slice.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct MlaParams {
  const float* ws;        // wkv_b block scales [H (dn + dv) / 128, C / 128]
  __nv_bfloat16* out;     // qk: [T, H, C]; v: [T, H, dv]
  unsigned* err;
  int T, H, C;
  int v_mode;             // 0: qk, 1: v
  int kb_count;           // K blocks of 128: qk 1, v C / 128
  int n_tiles, m_tiles;   // column tiles (qk C / 128, v 1), 128-token tiles
};

// Byte offset of 16-byte chunk q (elements 8q .. 8q + 7) of row r of a bf16
// tile of 128 rows x 128 elements, 128-byte swizzled: two halves of 64
// elements (128-byte rows), 8-row atoms of 1024 bytes, chunk c of row r stored
// at chunk c ^ (r % 8). For the v projection the rows are N and the elements
// K (a K-major operand); for qk the rows are K and the elements N (an
// MN-major operand with 16 KB between the halves and 1 KB between 8-row
// groups).
__device__ __forceinline__ uint32_t b16_chunk_offset(int r, int q) {
  return static_cast<uint32_t>((q >> 3) * kAHalf + (r >> 3) * 1024 + (r & 7) * 128 + (((q & 7) ^ (r & 7)) << 4));
}

// Two e4m3 codes (the first in the low byte) times the block scale, as bf16x2.
__device__ __forceinline__ uint32_t dequant_pack2(uint32_t pair, float s) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair & 0xFFFFu), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  const __nv_bfloat162 r = __floats2bfloat162_rn(__fmul_rn(f.x, s), __fmul_rn(f.y, s));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Persistent CTAs: CTA c takes tiles c, c + grid, ... of (head, 128-token
// tile, 128-column tile), head-major, each KB K blocks long, as steps j =
// (its i-th tile) * KB + kb. The MMA accumulates a tile in one of two TMEM
// buffers, so the epilogue drains tile i while the loads, dequantisation and
// MMAs of tile i + 1 go on.
//
// Launched with programmatic stream serialization: the weight tiles and
// scales may be read while the previous kernel on the stream still runs; the
// activations are loaded, and the output written, after it has completed.
__global__ void __launch_bounds__(kMlaThreads, 1)
    mla_absorb_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_o, const MlaParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* out_stage = smem + kOffO;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* a_empty = a_full + kARing;
  uint64_t* w_full = a_empty + kARing;
  uint64_t* w_empty = w_full + kWRing;
  uint64_t* b_full = w_empty + kWRing;
  uint64_t* b_empty = b_full + kBRing;
  uint64_t* tfull = b_empty + kBRing;  // [2]: accumulator buffer complete
  uint64_t* tempty = tfull + 2;        // [2]: accumulator buffer drained
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = prm.kb_count;
  const int kdim = prm.v_mode ? prm.C : 128;  // the activation's per-head width
  const int per_head = prm.n_tiles * prm.m_tiles;
  const int ntiles = prm.H * per_head;
  const int grid = static_cast<int>(gridDim.x);
  const int my_tiles = static_cast<int>(blockIdx.x) < ntiles ? (ntiles - 1 - static_cast<int>(blockIdx.x)) / grid + 1 : 0;
  const long long nsteps = static_cast<long long>(my_tiles) * KB;
  auto tile_of = [&](int i, int& h, int& mt, int& nt) {
    const int tt = static_cast<int>(blockIdx.x) + i * grid;
    h = tt / per_head;
    const int r = tt - h * per_head;
    mt = r / prm.n_tiles;
    nt = r - mt * prm.n_tiles;
  };
  // Parity of the n-th completion (n >= 0) of a ring entry used every `depth` steps.
  auto use_parity = [](long long j, int depth) { return static_cast<uint32_t>((j / depth) & 1); };

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kARing; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kWRing; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], kDequantWarps);
    }
    for (int s = 0; s < kBRing; ++s) {
      mbar_init(&b_full[s], kDequantWarps);
      mbar_init(&b_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 || warp == 10) {
    // ---------------- TMA producers: activations (warp 0), weights (warp 10) ----------------
    if (lane == 0) {
      const bool act = warp == 0;
      const int depth = act ? kARing : kWRing;
      uint64_t* full = act ? a_full : w_full;
      uint64_t* empty = act ? a_empty : w_empty;
      if (act) {
        tma_prefetch_desc(&tmap_a);
        griddep_wait();  // the activations come from the previous kernel
      } else {
        tma_prefetch_desc(&tmap_w);
      }
      long long j = 0;
      for (; j < nsteps; ++j) {
        const int i = static_cast<int>(j / KB), kb = static_cast<int>(j - static_cast<long long>(i) * KB);
        int h, mt, nt;
        tile_of(i, h, mt, nt);
        const int st = static_cast<int>(j % depth);
        if (j >= depth &&
            !mbar_wait(&empty[st], use_parity(j, depth) ^ 1u, abort_flag, prm.err, kDevErrTimeoutMla))
          break;
        if (act) {
          uint8_t* sa = smem + st * kATile;
          mbar_arrive_expect_tx(&full[st], kATile);
          const int ax = h * kdim + kb * 128;
          tma_load_2d(sa, &tmap_a, &full[st], ax, mt * 128);
          tma_load_2d(sa + kAHalf, &tmap_a, &full[st], ax + 64, mt * 128);
        } else {
          uint8_t* sw = smem + kOffW + st * kB8Tile;
          mbar_arrive_expect_tx(&full[st], kB8Tile);
          if (prm.v_mode) tma_load_2d(sw, &tmap_w, &full[st], kb * 128, h * 256 + 128);
          else tma_load_2d(sw, &tmap_w, &full[st], nt * 128, h * 256);
        }
      }
      // No copy may still be landing when the CTA exits.
      for (long long q = j - 1; q >= 0 && q >= j - depth; --q)
        mbar_wait(&full[q % depth], use_parity(q, depth), nullptr, prm.err, kDevErrTimeoutMla);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    const bool leader = elect_one_sync();
    constexpr uint32_t kIdescK = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t kIdescMN = idesc_bf16_f32(128, 128, true);
    long long j = 0;
    bool ok = true;
    for (int i = 0; ok && i < my_tiles; ++i) {
      const int b = i & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tempty[b], static_cast<uint32_t>(((i >> 1) & 1) ^ 1), abort_flag,
                                             prm.err, kDevErrTimeoutMla))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t d = tmem_base + static_cast<uint32_t>(b * 128);
      for (int kb = 0; kb < KB; ++kb, ++j) {
        const int sa = static_cast<int>(j % kARing), sb = static_cast<int>(j % kBRing);
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait(&a_full[sa], use_parity(j, kARing), abort_flag, prm.err, kDevErrTimeoutMla) &&
                            mbar_wait(&b_full[sb], use_parity(j, kBRing), abort_flag, prm.err, kDevErrTimeoutMla))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_addr = smem_u32(smem + sa * kATile);
        const uint32_t b_addr = smem_u32(smem + kOffB + sb * kB16Tile);
        if (leader) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint64_t ad = sdesc_kmajor_sw128(a_addr + half * kAHalf);
            const uint64_t bd = sdesc_kmajor_sw128(b_addr + half * kAHalf);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // 16 K per MMA. A (and B for v): 32 bytes along the K-major row,
              // the descriptor's start address advances by 2 x 16 B. B for qk:
              // 16 K rows, two 1 KB groups of the MN-major tile.
              const uint32_t acc = (kb | half | k) != 0 ? 1u : 0u;
              if (prm.v_mode)
                mma_bf16(d, ad + 2 * k, bd + 2 * k, kIdescK, acc);
              else
                mma_bf16(d, ad + 2 * k, sdesc_mnmajor_sw128(b_addr + (half * 4 + k) * 2048, kAHalf, 1024), kIdescMN,
                         acc);
            }
          }
          mma_commit(&a_empty[sa]);
          mma_commit(&b_empty[sb]);
          if (kb == KB - 1) mma_commit(&tfull[b]);
        }
        __syncwarp();
      }
    }
    if (leader) {  // every MMA done before TMEM is released
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, prm.err, kDevErrTimeoutMla);
    }
    __syncwarp();
  } else if (warp < 6 || warp > 10) {
    // ---------------- weight dequantisation ----------------
    // Row r of the e4m3 tile becomes row r of the bf16 tile: for v, row r is
    // output column d = r (N) over 128 c (K); for qk, row r is d = r (K) over
    // 128 output columns c (N). Two warps share each row range (one on each
    // half of the row), one pair per SM sub-partition.
    const int dw = warp < 6 ? warp - 2 : warp - 7;  // 0..7
    const int r = (dw & 3) * 32 + lane;
    const int c_lo = (dw >> 2) * 4;
    const int cblocks = prm.C / 128;
    for (long long j = 0; j < nsteps; ++j) {
      const int i = static_cast<int>(j / KB), kb = static_cast<int>(j - static_cast<long long>(i) * KB);
      int h, mt, nt;
      tile_of(i, h, mt, nt);
      const int sw = static_cast<int>(j % kWRing), sb = static_cast<int>(j % kBRing);
      // qk: W rows h*256 + d, columns nt*128 + c; v: rows h*256 + 128 + d, columns kb*128 + c.
      const float s = prm.v_mode ? __ldg(prm.ws + static_cast<size_t>(2 * h + 1) * cblocks + kb)
                                 : __ldg(prm.ws + static_cast<size_t>(2 * h) * cblocks + nt);
      if (!__all_sync(0xFFFFFFFFu,
                      mbar_wait(&w_full[sw], use_parity(j, kWRing), abort_flag, prm.err, kDevErrTimeoutMla) &&
                          (j < kBRing || mbar_wait(&b_empty[sb], use_parity(j, kBRing) ^ 1u, abort_flag, prm.err,
                                                   kDevErrTimeoutMla))))
        break;
      const uint8_t* b8 = smem + kOffW + sw * kB8Tile;
      uint8_t* b16 = smem + kOffB + sb * kB16Tile;
      // The e4m3 tile is 128-byte swizzled by the TMA: 16-byte chunk c of row
      // r (16 elements) sits at chunk c ^ (r % 8).
#pragma unroll
      for (int c = c_lo; c < c_lo + 4; ++c) {
        const uint4 raw = *reinterpret_cast<const uint4*>(b8 + r * 128 + ((c ^ (r & 7)) << 4));
        *reinterpret_cast<uint4*>(b16 + b16_chunk_offset(r, 2 * c)) =
            make_uint4(dequant_pack2(raw.x, s), dequant_pack2(raw.x >> 16, s), dequant_pack2(raw.y, s),
                       dequant_pack2(raw.y >> 16, s));
        *reinterpret_cast<uint4*>(b16 + b16_chunk_offset(r, 2 * c + 1)) =
            make_uint4(dequant_pack2(raw.z, s), dequant_pack2(raw.z >> 16, s), dequant_pack2(raw.w, s),
                       dequant_pack2(raw.w >> 16, s));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&w_empty[sw]);  // the e4m3 tile is read
      fence_proxy_async_smem();                   // generic-proxy writes, read next by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&b_full[sb]);
    }
  } else {
    // ---------------- epilogue ----------------
    // Each warp drains its 32 TMEM lanes (tokens) into its own staging slab,
    // then one lane stores the slab with two TMA boxes of 32 rows x 64 columns.
    griddep_wait();  // no output is written before the previous kernel has completed
    const int quarter = warp & 3;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const int nout = prm.v_mode ? 128 : prm.C;
    uint8_t* slab = out_stage + quarter * kOutWarp;
    for (int i = 0; i < my_tiles; ++i) {
      const int b = i & 1;
      int h, mt, nt;
      tile_of(i, h, mt, nt);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tfull[b], static_cast<uint32_t>((i >> 1) & 1), abort_flag, prm.err,
                                             kDevErrTimeoutMla)))
        break;
      tc_fence_after_sync();
      const int y = mt * 128 + quarter * 32;
      const int x = h * nout + nt * 128;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // Each half of the slab is committed as its own bulk group (one per
        // half and tile, empty where nothing is stored); groups complete in
        // order, so with at most one pending, the store that last used this
        // half has read it.
        if (lane == 0) bulk_wait_group_read_le1();
        __syncwarp();
#pragma unroll
        for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(b * 128 + c0), v);
          if (c0 == 96) {  // the buffer's last columns are in registers: free it for tile i + 2
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
          }
          uint8_t* row = slab + half * kOutHalf + lane * 128;
#pragma unroll
          for (int g = 0; g < 4; ++g) {  // 16-byte chunk ((c0 % 64) / 8 + g) of the row, at chunk ^ (lane % 8)
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 bb =
                  __floats2bfloat162_rn(__uint_as_float(v[g * 8 + 2 * e]), __uint_as_float(v[g * 8 + 2 * e + 1]));
              w4[e] = *reinterpret_cast<const uint32_t*>(&bb);
            }
            const int chunk = ((c0 & 63) >> 3) + g;
            *reinterpret_cast<uint4*>(row + ((chunk ^ (lane & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
        fence_proxy_async_smem();  // the slab's generic-proxy writes, read next by the TMA
        __syncwarp();
        if (lane == 0) {
          // Rows past T inside the box are clipped by the TMA; a quarter wholly
          // past T stores nothing but still commits its (empty) group, so that
          // every half of every tile owns exactly one group.
          if (y < prm.T) tma_store_2d(&tmap_o, slab + half * kOutHalf, x + half * 64, y);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group0();  // every store written before the CTA exits
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 256);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
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

// 2-D row-major tensor map: rows x cols elements, boxes of box_cols x box_rows.
bool make_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int esize, uint64_t rows,
                 uint64_t cols, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * static_cast<uint64_t>(esize)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int mla_run(const void* in, const void* w, const float* ws, void* out, int64_t T, int64_t H, int64_t dn, int64_t dv,
            int64_t C, int v_mode, cudaStream_t stream) {
  if (T < 0 || H < 1 || dn != 128 || dv != 128 || C < 128 || C % 128 || H * (dn + dv) > (int64_t{1} << 31) - 1 ||
      T > (int64_t{1} << 31) - 1 || T * H * C > (int64_t{1} << 40))
    return FP8BLK_ERR_SHAPE;
  if (T == 0) return FP8BLK_OK;
  if (!in || !w || !ws || !out) return FP8BLK_ERR_NULL;
  if (!is_aligned(in, 16) || !is_aligned(w, 16) || !is_aligned(out, 16) || !is_aligned(ws, 4)) return FP8BLK_ERR_ALIGN;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  static bool attr_done[64] = {};
  if (d->device >= 64 || !attr_done[d->device]) {
    if (cudaFuncSetAttribute(mla_absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmem) !=
        cudaSuccess)
      return FP8BLK_ERR_CUDA;
    if (d->device < 64) attr_done[d->device] = true;
  }
  const int64_t kdim = v_mode ? C : dn;
  const int64_t nout = v_mode ? dv : C;
  // The e4m3 tile is read a row per thread: 128-byte swizzled so a warp's
  // 16-byte reads spread over the banks.
  CUtensorMap ma, mw, mo;
  if (!make_map_2d(&ma, in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(T),
                   static_cast<uint64_t>(H * kdim), 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&mw, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(H * (dn + dv)),
                   static_cast<uint64_t>(C), 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&mo, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(T),
                   static_cast<uint64_t>(H * nout), 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
    return FP8BLK_ERR_CUDA;
  MlaParams prm{};
  prm.ws = ws;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.err = d->err_word;
  prm.T = static_cast<int>(T);
  prm.H = static_cast<int>(H);
  prm.C = static_cast<int>(C);
  prm.v_mode = v_mode;
  prm.kb_count = static_cast<int>(kdim / 128);
  prm.n_tiles = v_mode ? 1 : static_cast<int>(C / 128);
  prm.m_tiles = static_cast<int>((T + 127) / 128);
  const int64_t tiles = H * prm.m_tiles * prm.n_tiles;
  if (tiles > (int64_t{1} << 31) - 1) return FP8BLK_ERR_SHAPE;
  // Persistent: one CTA per SM (the rings' shared memory), at most one per tile.
  const int grid = static_cast<int>(tiles < d->sm_count ? tiles : d->sm_count);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kMlaThreads);
  cfg.dynamicSmemBytes = kMlaSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, mla_absorb_kernel, ma, mw, mo, prm));
}

}  // namespace
}  // namespace fp8blk

using namespace fp8blk;

extern "C" int fp8blk_mla_absorb_qk(const void* q_nope_bf16, const void* wkv_b_e4m3, const float* wkv_b_s,
                                    void* out_bf16, int64_t T, int64_t H, int64_t dn, int64_t dv, int64_t C,
                                    fp8blk_stream_t stream) {
  return mla_run(q_nope_bf16, wkv_b_e4m3, wkv_b_s, out_bf16, T, H, dn, dv, C, 0,
                 reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fp8blk_mla_absorb_v(const void* x_bf16, const void* wkv_b_e4m3, const float* wkv_b_s, void* out_bf16,
                                   int64_t T, int64_t H, int64_t dn, int64_t dv, int64_t C, fp8blk_stream_t stream) {
  return mla_run(x_bf16, wkv_b_e4m3, wkv_b_s, out_bf16, T, H, dn, dv, C, 1, reinterpret_cast<cudaStream_t>(stream));
}
