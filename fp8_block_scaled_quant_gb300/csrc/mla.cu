// MLA "absorb" projections with the FP8 wkv_b weight ("Administrator &
// Developer Guide", 8.3 steps 5 and 7): per head h,
//   qk: out[t, h, c] = sum_d q_nope[t, h, d] * W[h (dn + dv) + d, c]        (K = dn, N = C)
//   v:  out[t, h, d] = sum_c x[t, h, c]      * W[h (dn + dv) + dn + d, c]   (K = C,  N = dv)
// where W is wkv_b as weight_dequant gives it (bf16 of the fp32 code times its
// 128 x 128 block scale, 8.5.2), activations and outputs are bf16, and the
// sum is fp32 (a bf16 product accumulated in fp32).
//
// The tensor cores take bf16 x bf16 (tcgen05.mma kind::f16, both operands
// bf16): the FP8 weight tile is TMA-loaded as bytes, dequantised by four warps
// into a bf16 K-major 128-byte-swizzled tile in shared memory (transposed in
// the qk case, where W's rows are the K dimension), and fed to the MMA next to
// the TMA-loaded bf16 activation tile. One CTA per (head, 128-token tile,
// 128-column tile); the fp32 accumulator stays in TMEM over the whole K
// (no per-block promotion: the block scale is inside the dequantised weight).
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

constexpr int kMlaThreads = 192;                 // warp 0 TMA, warp 1 MMA, warps 2-5 dequant + epilogue
constexpr int kAHalf = 128 * 128;                // 128 rows x 64 bf16 (one 128-byte swizzled half)
constexpr int kATile = 2 * kAHalf;               // 128 token rows x 128 bf16
constexpr int kB8Tile = 128 * 128;               // 128 x 128 e4m3, unswizzled rows of 128 bytes
constexpr int kB16Tile = 2 * kAHalf;             // the dequantised weight tile, K-major, two halves
constexpr int kMlaStageBytes = kATile + kB8Tile + kB16Tile;
// Stages: one for qk (a single K block, so two CTAs fit on an SM), two for v.
__host__ __device__ constexpr int mla_smem(int stages) { return 1024 + stages * kMlaStageBytes + (3 * stages + 2) * 8 + 16; }
constexpr unsigned kDevErrTimeoutMla = 1u << 6;

// kind::f16 instruction descriptor: f32 accumulator, A and B both bf16 (one
// value sets both format fields), both K-major, an M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  constexpr uint32_t kBf16 = 1;
  return (1u << 4) | (kBf16 << 7) | (kBf16 << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
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

// Byte offset of element (row r, k) of a K-major bf16 tile of 128 rows x 128
// k: two halves of 64 k (128-byte rows), 8-row atoms of 1024 bytes, 16-byte
// chunk c of row r stored at chunk c ^ (r % 8).
__device__ __forceinline__ uint32_t b16_chunk_offset(int r, int q) {  // q: 16-byte chunk 0..15 (8 k each)
  return static_cast<uint32_t>((q >> 3) * kAHalf + (r >> 3) * 1024 + (r & 7) * 128 + (((q & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t dequant_pack2(uint8_t a, uint8_t b, float s) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
      static_cast<__nv_fp8x2_storage_t>(static_cast<uint16_t>(a) | (static_cast<uint16_t>(b) << 8)), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  const __nv_bfloat162 r = __floats2bfloat162_rn(__fmul_rn(f.x, s), __fmul_rn(f.y, s));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <int kMlaStages>
__global__ void __launch_bounds__(kMlaThreads, 1)
    mla_absorb_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                      const MlaParams prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kMlaStages * kMlaStageBytes);
  uint64_t* bready = full + kMlaStages;
  uint64_t* empty = bready + kMlaStages;
  uint64_t* tfull = empty + kMlaStages;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bid = static_cast<int>(blockIdx.x);
  const int nt = bid % prm.n_tiles;
  const int mt = (bid / prm.n_tiles) % prm.m_tiles;
  const int h = bid / (prm.n_tiles * prm.m_tiles);
  const int KB = prm.kb_count;
  const int kdim = prm.v_mode ? prm.C : 128;  // the activation's per-head width

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMlaStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&bready[s], 4);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmap_a);
      tma_prefetch_desc(&tmap_w);
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int st = kb % kMlaStages;
        if (kb >= kMlaStages &&
            !mbar_wait(&empty[st], ((kb / kMlaStages) & 1) ^ 1u, abort_flag, prm.err, kDevErrTimeoutMla))
          break;
        uint8_t* sa = smem + st * kMlaStageBytes;
        mbar_arrive_expect_tx(&full[st], kATile + kB8Tile);
        const int ax = h * kdim + kb * 128;
        tma_load_2d(sa, &tmap_a, &full[st], ax, mt * 128);
        tma_load_2d(sa + kAHalf, &tmap_a, &full[st], ax + 64, mt * 128);
        if (prm.v_mode) tma_load_2d(sa + kATile, &tmap_w, &full[st], kb * 128, h * 256 + 128);
        else tma_load_2d(sa + kATile, &tmap_w, &full[st], nt * 128, h * 256);
        ++issued;
      }
      // No copy may still be landing when the CTA exits.
      for (int i = issued - 1; i >= 0 && i >= issued - kMlaStages; --i)
        mbar_wait(&full[i % kMlaStages], static_cast<uint32_t>((i / kMlaStages) & 1), nullptr, prm.err,
                  kDevErrTimeoutMla);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    const bool leader = elect_one_sync();
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128);
    for (int kb = 0; kb < KB; ++kb) {
      const int st = kb % kMlaStages;
      const bool w =
          mbar_wait(&bready[st], static_cast<uint32_t>((kb / kMlaStages) & 1), abort_flag, prm.err, kDevErrTimeoutMla);
      if (!__all_sync(0xFFFFFFFFu, w)) break;
      tc_fence_after_sync();
      const uint32_t a_addr = smem_u32(smem + st * kMlaStageBytes);
      const uint32_t b_addr = a_addr + kATile + kB8Tile;
      if (leader) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint64_t ad = sdesc_kmajor_sw128(a_addr + half * kAHalf);
          const uint64_t bd = sdesc_kmajor_sw128(b_addr + half * kAHalf);
#pragma unroll
          for (int k = 0; k < 4; ++k)  // 16 bf16 = 32 bytes per MMA: the start address advances by 2 x 16 B
            mma_bf16(tmem_base, ad + 2 * k, bd + 2 * k, kIdesc, (kb | half | k) != 0 ? 1u : 0u);
        }
        mma_commit(&empty[st]);
        if (kb == KB - 1) mma_commit(tfull);
      }
      __syncwarp();
    }
    if (leader) {  // every MMA done before TMEM is released
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, prm.err, kDevErrTimeoutMla);
    }
    __syncwarp();
  } else {
    // ---------------- weight dequant, then the epilogue ----------------
    const int n = (warp - 2) * 32 + lane;  // the dequantised tile's row (MMA N index)
    const int cblocks = prm.C / 128;
    bool ok = true;
    for (int kb = 0; kb < KB; ++kb) {
      const int st = kb % kMlaStages;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[st], static_cast<uint32_t>((kb / kMlaStages) & 1), abort_flag,
                                             prm.err, kDevErrTimeoutMla))) {
        ok = false;
        break;
      }
      const uint8_t* b8 = smem + st * kMlaStageBytes + kATile;
      uint8_t* b16 = smem + st * kMlaStageBytes + kATile + kB8Tile;
      // qk: W rows h*256 + d (d = K), columns nt*128 + n; v: rows h*256 + 128 + n, columns kb*128 + k.
      const float s = prm.v_mode ? __ldg(prm.ws + static_cast<size_t>(2 * h + 1) * cblocks + kb)
                                 : __ldg(prm.ws + static_cast<size_t>(2 * h) * cblocks + nt);
#pragma unroll 4
      for (int q = 0; q < 16; ++q) {  // 8 k per 16-byte chunk
        uint8_t v8[8];
        if (prm.v_mode) {
          const uint2 raw = *reinterpret_cast<const uint2*>(b8 + n * 128 + q * 8);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v8[i] = static_cast<uint8_t>(raw.x >> (8 * i));
            v8[4 + i] = static_cast<uint8_t>(raw.y >> (8 * i));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) v8[i] = b8[(q * 8 + i) * 128 + n];  // column n of rows k: the transpose
        }
        const uint4 packed = make_uint4(dequant_pack2(v8[0], v8[1], s), dequant_pack2(v8[2], v8[3], s),
                                        dequant_pack2(v8[4], v8[5], s), dequant_pack2(v8[6], v8[7], s));
        *reinterpret_cast<uint4*>(b16 + b16_chunk_offset(n, q)) = packed;
      }
      fence_proxy_async_smem();  // generic-proxy writes, read next by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&bready[st]);
    }
    if (ok && __all_sync(0xFFFFFFFFu, mbar_wait(tfull, 0, abort_flag, prm.err, kDevErrTimeoutMla))) {
      tc_fence_after_sync();
      const int quarter = warp & 3;
      const int r = mt * 128 + quarter * 32 + lane;  // token
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      const int nout = prm.v_mode ? 128 : prm.C;
      __nv_bfloat16* dst = prm.out + (static_cast<size_t>(r) * prm.H + h) * nout + nt * 128;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(c0), v);
        if (r < prm.T) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 b =
                  __floats2bfloat162_rn(__uint_as_float(v[g * 8 + 2 * e]), __uint_as_float(v[g * 8 + 2 * e + 1]));
              w4[e] = *reinterpret_cast<const uint32_t*>(&b);
            }
            *reinterpret_cast<uint4*>(dst + c0 + g * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 128);
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
    if (cudaFuncSetAttribute(mla_absorb_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, mla_smem(1)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(mla_absorb_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, mla_smem(2)) !=
            cudaSuccess)
      return FP8BLK_ERR_CUDA;
    if (d->device < 64) attr_done[d->device] = true;
  }
  const int64_t kdim = v_mode ? C : dn;
  CUtensorMap ma, mw;
  if (!make_map_2d(&ma, in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(T),
                   static_cast<uint64_t>(H * kdim), 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&mw, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(H * (dn + dv)),
                   static_cast<uint64_t>(C), 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
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
  const int64_t grid = H * prm.m_tiles * prm.n_tiles;
  if (grid > (int64_t{1} << 31) - 1) return FP8BLK_ERR_SHAPE;
  if (v_mode) mla_absorb_kernel<2><<<static_cast<unsigned>(grid), kMlaThreads, mla_smem(2), stream>>>(ma, mw, prm);
  else mla_absorb_kernel<1><<<static_cast<unsigned>(grid), kMlaThreads, mla_smem(1), stream>>>(ma, mw, prm);
  return launch_status();
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
