// Host-side helpers shared by the library's translation units: per-device
// information (SM count, compute capability, the device error word), status
// mapping and argument checks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8blk.h"

namespace fp8blk {

constexpr int kBlock = 128;

struct DevInfo {
  int device;
  int sm_count;
  int cc_major;
  int cc_minor;
  int smem_optin;      // max dynamic shared memory per block (opt-in)
  int smem_per_sm;     // shared memory per SM (all resident blocks together)
  unsigned* err_word;  // device address of this device's error word
};

// Fills *out with the current device's info (cached per device). Returns
// FP8BLK_ERR_CUDA if the runtime fails, FP8BLK_ERR_ARCH unless the device is
// compute capability 10.3 (sm_103).
int current_device(const DevInfo** out);

inline bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// scale_fmt arguments: FP8BLK_SCALE_FP32, FP8BLK_SCALE_UE8M0, or UE8M0 with
// FP8BLK_SCALE_PROMOTE (keep the per-block promotion in the GEMMs).
inline bool scale_fmt_valid(int f) {
  return f == FP8BLK_SCALE_FP32 || f == FP8BLK_SCALE_UE8M0 || f == (FP8BLK_SCALE_UE8M0 | FP8BLK_SCALE_PROMOTE);
}
inline bool scale_fmt_ue8m0(int f) { return (f & ~FP8BLK_SCALE_PROMOTE) == FP8BLK_SCALE_UE8M0; }
// The GEMM lets the tensor core apply the scales (block-scaled MMA) where its
// tiles allow it: UE8M0 scales without FP8BLK_SCALE_PROMOTE.
inline bool scale_fmt_mx(int f) { return f == FP8BLK_SCALE_UE8M0; }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8BLK_OK : FP8BLK_ERR_CUDA; }

inline int launch_status() { return cuda_status(cudaGetLastError()); }

}  // namespace fp8blk
