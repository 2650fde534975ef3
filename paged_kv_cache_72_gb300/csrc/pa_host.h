// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

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

// Records the CUDA error behind a PA_ERR_CUDA (per host thread) so that
// pa_strerror can name it.
void note_cuda_error(int code, const char* where);

// Kernel launch status -> library status.
inline int launch_status(cudaError_t e, const char* where = "kernel launch") {
  if (e == cudaSuccess) return PA_OK;
  note_cuda_error((int)e, where);
  return PA_ERR_CUDA;
}

// Launches `kern` with programmatic stream serialization allowed: the kernel
// may start while its predecessor in the stream drains, and calls
// grid_dep_wait before reading any input.  Returns the launch status.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Clears an error left by an earlier, already reported runtime call so that
// the check after the next launch sees only that launch.
inline void clear_stale_error() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) note_cuda_error((int)e, "an earlier runtime call (cleared)");
}

}  // namespace pa
