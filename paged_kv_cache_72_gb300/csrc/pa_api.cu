// Library-wide entry points: error reporting, version, device attributes and
// the tensor-map encoder lookup.
#include <stdio.h>

#include <mutex>

#include "pa_host.h"

namespace pa {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices];
std::mutex g_mu;
}  // namespace

int current_device_info(DeviceInfo* info) {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return launch_status(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_have[dev]) {
    DeviceInfo d{};
    d.device = dev;
    cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (!e) e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (!e) e = cudaDeviceGetAttribute(&d.smem_per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e) return launch_status(e, "cudaDeviceGetAttribute");
    g_info[dev] = d;
    g_have[dev] = true;
  }
  *info = g_info[dev];
  return PA_OK;
}

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

namespace {
thread_local char g_err_msg[256];
}  // namespace

void note_cuda_error(int code, const char* where) {
  if (code >= 1000)  // a driver-API result (tensor-map encoding)
    snprintf(g_err_msg, sizeof(g_err_msg), "CUDA call failed (%s: CUresult %d)", where,
             code - 1000);
  else
    snprintf(g_err_msg, sizeof(g_err_msg), "CUDA call failed (%s: %s: %s)", where,
             cudaGetErrorName((cudaError_t)code), cudaGetErrorString((cudaError_t)code));
}

}  // namespace pa

extern "C" {

int pa_get_error(int32_t* err_word, pa_stream stream, int32_t* flags) {
  if (flags) *flags = 0;
  if (!err_word) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, err_word, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (host != 0) {
    if (cudaMemsetAsync(err_word, 0, sizeof(int32_t), s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  }
  if (flags) *flags = host;
  return host ? PA_ERR_DEVICE_INDEX : PA_OK;
}

const char* pa_strerror(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_WORKSPACE: return "decode workspace too small";
    case PA_ERR_CUDA: return pa::g_err_msg[0] ? pa::g_err_msg : "CUDA call failed";
    case PA_ERR_DEVICE_INDEX: return "a kernel reported an out-of-range index";
    default: return "unknown status";
  }
}

int pa_version(void) { return 100; }

}  // extern "C"
