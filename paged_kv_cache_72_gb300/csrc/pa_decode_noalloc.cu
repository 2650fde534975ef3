// pa_decode_noalloc: paged decode attention for callers that cannot allocate
// device memory.
//
// pa_decode needs a workspace for the partial softmax states of contexts that
// are split across thread blocks, and expects the caller to allocate it.  Some
// callers cannot: a runtime whose device memory is already reserved in full by
// another allocator (a framework's pool that owns the free memory), a plain C
// host program with no device allocator of its own, or a latency-critical
// decode loop that cannot afford cudaMalloc's implicit device synchronization
// and unpredictable cost.  This entry point runs the same kernels with their
// workspace in a fixed array that lives in the library's own device memory.
//
// The array is a file-scope static __device__ buffer of PA_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  In host
// code the array's name is only a host-side stand-in, so its device address is
// looked up with cudaGetSymbolAddress, once per device (and again if that
// device's context was reset and re-created), with that device current, the
// first time the entry point runs there.
#include <mutex>

#include "pa_host.h"

namespace pa {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
struct ScratchAddr {
  void* ptr;
  unsigned long long ctx_id;   // the context the address belongs to (0: unknown)
};
ScratchAddr g_scratch[kMaxScratchDevices];
std::mutex g_scratch_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// A process-unique id of the current context, or 0 where the driver cannot
// give one.  A device reset destroys the context and the next runtime call
// creates a new one, with a new id, in which the array may sit elsewhere.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_decode_scratch on the current device.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return launch_status(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxScratchDevices) return PA_ERR_CUDA;
  // cudaSetDevice on the current device makes its primary context current,
  // creating it if a reset destroyed it, so that its id can be read
  if (cudaError_t e = cudaSetDevice(dev)) return launch_status(e, "cudaSetDevice");
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& s = g_scratch[dev];
  if (!s.ptr || s.ctx_id != ctx) {
    void* p = nullptr;
    if (cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch))
      return launch_status(e, "cudaGetSymbolAddress");
    if (!p) return PA_ERR_CUDA;
    s.ptr = p;
    s.ctx_id = ctx;
  }
  *out = s.ptr;
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int32_t table_stride,
                                 const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int64_t num_blocks, int32_t dtype, float scale, void* out,
                                 int32_t flags, int32_t num_ctas, int32_t* err_word,
                                 pa_stream stream) {
  size_t need = 0;
  if (int rc = pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                                        flags, num_ctas, &need))
    return rc;
  // the fixed buffer is too small for this grid and group size
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (int rc = pa::scratch_address(&scratch)) return rc;
  // The workspace starts with the split contexts' piece counters, which must
  // be zero when the decode starts.  The array is zero at load and every call
  // that runs to its end leaves them at zero, but the array keeps whatever the
  // last call left, so they are cleared here, on the call's stream, and no
  // earlier call's state can reach this one.  The partial-state records after
  // them are written before they are read within one call.
  if (cudaError_t e = cudaMemsetAsync(scratch, 0, (size_t)PA_DECODE_MAX_CTAS * sizeof(uint32_t),
                                      static_cast<cudaStream_t>(stream)))
    return pa::launch_status(e, "cudaMemsetAsync");
  return pa_decode(q, k_cache, v_cache, block_tables, table_stride, seq_lens, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, dtype, scale, out,
                   scratch, (size_t)PA_NOALLOC_SCRATCH_BYTES, flags, num_ctas, err_word, stream);
}
