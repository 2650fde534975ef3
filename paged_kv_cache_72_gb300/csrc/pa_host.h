// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Device attributes of the current device, cached per device.
struct DeviceInfo {
  int device;
  int sm_count;
  int smem_per_sm;      // bytes of shared memory per SM
  int smem_per_block;   // opt-in maximum per block
};
int current_device_info(DeviceInfo* info);

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point so
// that the library does not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool is_pow2(long long x) { return x > 0 && (x & (x - 1)) == 0; }

inline int ilog2(long long x) {
  int r = 0;
  while ((1LL << r) < x) ++r;
  return r;
}

// Kernel launch status -> library status.
inline int launch_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

}  // namespace pa
