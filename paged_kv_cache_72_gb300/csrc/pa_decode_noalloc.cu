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
// looked up with cudaGetSymbolAddress, once per device, with that device
// current, the first time the entry point runs on it.
#include <mutex>

#include "pa_host.h"

namespace pa {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
void* g_scratch_addr[kMaxScratchDevices];
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxScratchDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
  // The kernels write every workspace word they later read within the same
  // call (each thread block writes its bookkeeping before the merge kernel
  // reads it), so nothing left over from an earlier call needs clearing.
  return pa_decode(q, k_cache, v_cache, block_tables, table_stride, seq_lens, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, dtype, scale, out,
                   scratch, (size_t)PA_NOALLOC_SCRATCH_BYTES, flags, num_ctas, err_word, stream);
}
