// Library-wide entry points: device checks, the device error word, status
// names, and the FP8 linear layer ("Administrator & Developer Guide", 6.3:
// with gemm_impl "fp8", linear() quantises its input with act_quant and calls
// fp8_gemm) on device and on host buffers.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fp8blk.h"
#include "host.cuh"

namespace fp8blk {

// Error word written by kernels that gave up waiting (one per device context).
__device__ unsigned g_device_error_word;

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
int act_quant_launch(const void* x_bf16, int64_t M, int64_t K, void* q_e4m3, float* s, int scale_fmt,
                     cudaStream_t stream, bool trigger);
int linear_fused_run(const void* x, const void* w, const float* w_s, void* y, int64_t M, int64_t N, int64_t K,
                     int scale_fmt, cudaStream_t stream, bool* used);
int gemm_run(const void* a, const float* a_s, const void* w, const float* w_s, void* c, int64_t M, int64_t N,
             int64_t K, int scale_fmt, void* workspace, size_t workspace_bytes, cudaStream_t stream);
bool decode_gemm_fits(int64_t M, int64_t N, int64_t K, int sm_count);
bool linear_fused_fits(int64_t M, int64_t N, int64_t K);

namespace {

constexpr int kMaxDevices = 64;
DevInfo g_info[kMaxDevices];
int g_status[kMaxDevices];
std::once_flag g_once[kMaxDevices];

void init_device(int dev) {
  DevInfo& d = g_info[dev];
  d.device = dev;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    g_status[dev] = FP8BLK_ERR_CUDA;
    return;
  }
  d.sm_count = prop.multiProcessorCount;
  d.cc_major = prop.major;
  d.cc_minor = prop.minor;
  d.smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
  d.smem_per_sm = static_cast<int>(prop.sharedMemPerMultiprocessor);
  if (prop.major != 10 || prop.minor != 3) {
    g_status[dev] = FP8BLK_ERR_ARCH;
    return;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) {
    g_status[dev] = FP8BLK_ERR_CUDA;
    return;
  }
  d.err_word = static_cast<unsigned*>(p);
  g_status[dev] = FP8BLK_OK;
}

size_t align256(size_t v) { return (v + 255) & ~size_t{255}; }

#ifndef FP8BLK_FUSED_LINEAR_MAX_M
#define FP8BLK_FUSED_LINEAR_MAX_M 2
#endif
constexpr int64_t kFusedLinearMaxM = FP8BLK_FUSED_LINEAR_MAX_M;

}  // namespace

int current_device(const DevInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8BLK_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FP8BLK_ERR_CUDA;
  std::call_once(g_once[dev], init_device, dev);
  *out = &g_info[dev];
  return g_status[dev];
}

}  // namespace fp8blk

using namespace fp8blk;

extern "C" const char* fp8blk_status_string(int status) {
  switch (status) {
    case FP8BLK_OK: return "ok";
    case FP8BLK_ERR_NULL: return "null pointer";
    case FP8BLK_ERR_SHAPE: return "invalid shape (K must be a multiple of 128 where required)";
    case FP8BLK_ERR_ALIGN: return "misaligned pointer";
    case FP8BLK_ERR_WORKSPACE: return "workspace missing or too small";
    case FP8BLK_ERR_ARCH: return "device is not sm_103 (GB300)";
    case FP8BLK_ERR_TIMEOUT: return "a kernel gave up waiting";
    case FP8BLK_ERR_CUDA: return "CUDA runtime error";
    case FP8BLK_ERR_ARG: return "invalid argument";
    case FP8BLK_ERR_TOO_LARGE:
      return "problem needs more scratch than the built-in buffer of fp8blk_gemm_noalloc (use fp8blk_gemm)";
    default: return "unknown status";
  }
}

extern "C" int fp8blk_version(void) { return 100; }

extern "C" int fp8blk_last_device_error(fp8blk_stream_t stream, unsigned* bits) {
  if (!bits) return FP8BLK_ERR_NULL;
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8BLK_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, d->err_word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FP8BLK_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(d->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return FP8BLK_ERR_CUDA;
  }
  *bits = v;
  return v ? FP8BLK_ERR_TIMEOUT : FP8BLK_OK;
}

// Workspace of the linear layer: [GEMM workspace][x_q e4m3 M*K][x_s fp32 M*K/128],
// each part 256-byte aligned. The GEMM workspace comes first so that its tile
// counters sit at the same offset whatever the shape: one workspace can serve
// layers of different shapes.
extern "C" size_t fp8blk_linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return 0;
  return align256(gemm_workspace_bytes(M, N, K)) + align256(static_cast<size_t>(M) * K) +
         align256(static_cast<size_t>(M) * (K / kBlock) * 4);
}

extern "C" int fp8blk_linear(const void* x_bf16, const void* w_e4m3, const float* w_s, void* y_bf16, int64_t M,
                             int64_t N, int64_t K, int scale_fmt, void* workspace, size_t workspace_bytes,
                             fp8blk_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || K % kBlock != 0) return FP8BLK_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8BLK_OK;
  // M <= 2: act_quant runs inside the GEMM kernel (one launch), unless the
  // slice-per-SM decode GEMM takes the shape (act_quant + that kernel is the
  // faster pair). For larger M the in-kernel act_quant (every CTA quantises
  // all of x) costs more than the launch it saves, so act_quant is a kernel
  // of its own.
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  if (M <= kFusedLinearMaxM && !decode_gemm_fits(M, N, K, d->sm_count)) {
    bool used = false;
    const int st = linear_fused_run(x_bf16, w_e4m3, w_s, y_bf16, M, N, K, scale_fmt,
                                    reinterpret_cast<cudaStream_t>(stream), &used);
    if (st || used) return st;
  }
  if (!workspace) return FP8BLK_ERR_WORKSPACE;
  if (!is_aligned(workspace, 256)) return FP8BLK_ERR_ALIGN;
  const size_t need = fp8blk_linear_workspace_bytes(M, N, K);
  if (workspace_bytes < need) return FP8BLK_ERR_WORKSPACE;
  uint8_t* gws = static_cast<uint8_t*>(workspace);
  const size_t gbytes = align256(gemm_workspace_bytes(M, N, K));
  uint8_t* xq = gws + gbytes;
  float* xs = reinterpret_cast<float*>(xq + align256(static_cast<size_t>(M) * K));
  if (int st = act_quant_launch(x_bf16, M, K, xq, xs, scale_fmt, reinterpret_cast<cudaStream_t>(stream), true))
    return st;
  return gemm_run(xq, xs, w_e4m3, w_s, y_bf16, M, N, K, scale_fmt, gws, gbytes,
                  reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fp8blk_linear_kernels(int64_t M, int64_t N, int64_t K, int* kernels) {
  if (!kernels) return FP8BLK_ERR_NULL;
  if (M < 0 || N < 0 || K < 0 || K % kBlock != 0) return FP8BLK_ERR_SHAPE;
  if (M == 0 || N == 0 || K == 0) {
    *kernels = 0;
    return FP8BLK_OK;
  }
  const DevInfo* d;
  if (int st = current_device(&d)) return st;
  *kernels = (M <= kFusedLinearMaxM && !decode_gemm_fits(M, N, K, d->sm_count) && linear_fused_fits(M, N, K)) ? 1 : 2;
  return FP8BLK_OK;
}

// Host variant: [linear workspace][x bf16 M*K][y bf16 M*N] (the linear
// workspace first, for the same reason).
extern "C" size_t fp8blk_linear_host_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return 0;
  return align256(fp8blk_linear_workspace_bytes(M, N, K)) + align256(static_cast<size_t>(M) * K * 2) +
         align256(static_cast<size_t>(M) * N * 2);
}

extern "C" int fp8blk_linear_host(const void* x_host, const void* w_e4m3, const float* w_s, void* y_host,
                                  int64_t M, int64_t N, int64_t K, int scale_fmt, void* workspace,
                                  size_t workspace_bytes, fp8blk_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || K % kBlock != 0) return FP8BLK_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8BLK_OK;
  if (!x_host || !y_host) return FP8BLK_ERR_NULL;
  if (!workspace) return FP8BLK_ERR_WORKSPACE;
  if (!is_aligned(workspace, 256)) return FP8BLK_ERR_ALIGN;
  if (workspace_bytes < fp8blk_linear_host_workspace_bytes(M, N, K)) return FP8BLK_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* lws = static_cast<uint8_t*>(workspace);
  const size_t lbytes = align256(fp8blk_linear_workspace_bytes(M, N, K));
  const size_t xb = static_cast<size_t>(M) * K * 2, yb = static_cast<size_t>(M) * N * 2;
  uint8_t* xd = lws + lbytes;
  uint8_t* yd = xd + align256(xb);
  // Pinned host buffers the device can address (every page-locked allocation
  // on a unified-address system such as a Grace + GB300 node): the layer reads
  // x from and writes y to them directly over the chip-to-chip link, with no
  // staging copies, so its kernels stay one chain of dependent launches.
  void* xm = nullptr;
  void* ym = nullptr;
  if (cudaHostGetDevicePointer(&xm, const_cast<void*>(x_host), 0) == cudaSuccess &&
      cudaHostGetDevicePointer(&ym, y_host, 0) == cudaSuccess && is_aligned(xm, 16) && is_aligned(ym, 16))
    return fp8blk_linear(xm, w_e4m3, w_s, ym, M, N, K, scale_fmt, lws, lbytes, stream);
  cudaGetLastError();  // an unregistered buffer is not an error here: copy it instead
  if (K > 0 && cudaMemcpyAsync(xd, x_host, xb, cudaMemcpyHostToDevice, cs) != cudaSuccess) return FP8BLK_ERR_CUDA;
  if (int st = fp8blk_linear(xd, w_e4m3, w_s, yd, M, N, K, scale_fmt, lws, lbytes, stream))
    return st;
  if (cudaMemcpyAsync(y_host, yd, yb, cudaMemcpyDeviceToHost, cs) != cudaSuccess) return FP8BLK_ERR_CUDA;
  return FP8BLK_OK;
}
