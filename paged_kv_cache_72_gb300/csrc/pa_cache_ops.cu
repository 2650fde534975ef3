// Slot mapping, slot-mapped cache write and copy-on-write block copy.
//
// "vLLM Framework and Inference Engine Design", section "How is vLLM's KV cache
// paged?", bullet "Writing": when a token's K and V are computed, a small
// kernel stores them at slot block_table[floor(t/B)] * B + (t mod B); the list
// of these slots is the slot mapping.  Section "What operations can cause
// memory fragmentation, and how does vLLM avoid it?": a shared block is copied
// only when a sequence needs to write into it.
//
// The slot mapping, the 16-bit cache write and the block copy are pure data
// movement (16-byte vector copies, bit-exact).  The E4M3 cache write quantizes
// ("vLLM Framework and Inference Engine Design", section "How can one
// customize the tokenizer, cache strategy, or scheduler strategy?",
// kv_cache_dtype="fp8"; our reading: code = e4m3(float32(x) / scale), round to
// nearest even, saturating).
#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {

__global__ void slot_mapping_kernel(const int32_t* __restrict__ bt, int stride, int num_seqs,
                                    const int32_t* __restrict__ tok_seq,
                                    const int32_t* __restrict__ tok_pos, long long n, int log2B,
                                    long long num_blocks, int64_t* __restrict__ slots,
                                    int32_t* err) {
  grid_dep_wait();
  grid_dep_launch();
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n;
       k += (long long)gridDim.x * blockDim.x) {
    const int i = tok_seq[k];
    const int t = tok_pos[k];
    int64_t s = -1;
    if (i < 0 || i >= num_seqs || t < 0 || (long long)t >= ((long long)stride << log2B)) {
      set_error(err, PA_DEVERR_POSITION);
    } else {
      const int p = bt[(size_t)i * stride + (t >> log2B)];
      if (p < 0 || (long long)p >= num_blocks) {
        set_error(err, PA_DEVERR_BLOCK_ID);
      } else {
        s = ((int64_t)p << log2B) + (t & ((1 << log2B) - 1));
      }
    }
    slots[k] = s;
  }
}

// One block per new token: its K row [H_kv][D] and V row are each contiguous
// in the input and at the destination slot.
__global__ void cache_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                   const int64_t* __restrict__ slots, int vecs_per_row,
                                   long long num_slots, uint4* __restrict__ kc,
                                   uint4* __restrict__ vc, int32_t* err) {
  grid_dep_wait();
  grid_dep_launch();
  const long long tok = blockIdx.x;
  const long long s = slots[tok];
  if (s < 0) return;
  if (s >= num_slots) {
    if (threadIdx.x == 0) set_error(err, PA_DEVERR_SLOT);
    return;
  }
  const uint4* ks = k + tok * vecs_per_row;
  const uint4* vs = v + tok * vecs_per_row;
  uint4* kd = kc + s * vecs_per_row;
  uint4* vd = vc + s * vecs_per_row;
  for (int e = threadIdx.x; e < vecs_per_row; e += blockDim.x) {
    const uint4 a = __ldg(ks + e);
    const uint4 b = __ldg(vs + e);
    kd[e] = a;
    vd[e] = b;
  }
}

// The slot of new token tok, with the checks of slot_mapping_kernel: -1 (and
// an error bit) for a bad sequence index, position or table entry.
__device__ __forceinline__ long long token_slot(const int32_t* __restrict__ bt, int stride,
                                                int num_seqs, const int32_t* __restrict__ tok_seq,
                                                const int32_t* __restrict__ tok_pos, long long tok,
                                                int log2B, long long num_blocks, int32_t* err) {
  const int i = tok_seq[tok];
  const int t = tok_pos[tok];
  if (i < 0 || i >= num_seqs || t < 0 || (long long)t >= ((long long)stride << log2B)) {
    set_error(err, PA_DEVERR_POSITION);
    return -1;
  }
  const int p = bt[(size_t)i * stride + (t >> log2B)];
  if (p < 0 || (long long)p >= num_blocks) {
    set_error(err, PA_DEVERR_BLOCK_ID);
    return -1;
  }
  return ((long long)p << log2B) + (t & ((1 << log2B) - 1));
}

// Slot mapping and cache write in one launch: one CTA per new token.  Thread
// 0 finds the token's slot from its (sequence, position) and the block table,
// with the checks of slot_mapping_kernel, and writes it to slots when given;
// meanwhile every thread loads its first vectors of the token's K and V rows,
// which are then stored at the slot.  Saves the second kernel's start and its
// read of the slots.
__global__ void cache_write_mapped_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                          const int32_t* __restrict__ bt, int stride, int num_seqs,
                                          const int32_t* __restrict__ tok_seq,
                                          const int32_t* __restrict__ tok_pos, int log2B,
                                          long long num_blocks, int vecs_per_row,
                                          uint4* __restrict__ kc, uint4* __restrict__ vc,
                                          int64_t* __restrict__ slots, int32_t* err) {
  __shared__ long long s_slot;
  grid_dep_wait();
  grid_dep_launch();
  const long long tok = blockIdx.x;
  const uint4* ks = k + tok * vecs_per_row;
  const uint4* vs = v + tok * vecs_per_row;
  const int e0 = threadIdx.x;
  uint4 a0 = make_uint4(0u, 0u, 0u, 0u), b0 = a0;
  if (e0 < vecs_per_row) {
    a0 = __ldg(ks + e0);
    b0 = __ldg(vs + e0);
  }
  if (threadIdx.x == 0) {
    const long long sl = token_slot(bt, stride, num_seqs, tok_seq, tok_pos, tok, log2B,
                                    num_blocks, err);
    if (slots) slots[tok] = sl;
    s_slot = sl;
  }
  __syncthreads();
  const long long sl = s_slot;
  if (sl < 0) return;
  uint4* kd = kc + sl * vecs_per_row;
  uint4* vd = vc + sl * vecs_per_row;
  if (e0 < vecs_per_row) {
    kd[e0] = a0;
    vd[e0] = b0;
  }
  for (int e = e0 + blockDim.x; e < vecs_per_row; e += blockDim.x) {
    kd[e] = __ldg(ks + e);
    vd[e] = __ldg(vs + e);
  }
}

// E4M3 cache write: one block per new token; each thread turns 8 16-bit
// elements (16 bytes) of the token's K and V rows into 8 codes (8 bytes).
template <bool kBF16>
__global__ void cache_write_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                       const int64_t* __restrict__ slots, int vecs_per_row,
                                       long long num_slots, uint2* __restrict__ kc,
                                       uint2* __restrict__ vc, float k_scale, float v_scale,
                                       int32_t* err) {
  grid_dep_wait();
  grid_dep_launch();
  const long long tok = blockIdx.x;
  const long long s = slots[tok];
  if (s < 0) return;
  if (s >= num_slots) {
    if (threadIdx.x == 0) set_error(err, PA_DEVERR_SLOT);
    return;
  }
  auto quantize8 = [](const uint4 x, float scale) -> uint2 {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack2<kBF16>(w[i]);
      c[i] = f32x2_to_e4m3x2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
    }
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  };
  const uint4* ks = k + tok * vecs_per_row;
  const uint4* vs = v + tok * vecs_per_row;
  uint2* kd = kc + s * vecs_per_row;
  uint2* vd = vc + s * vecs_per_row;
  for (int e = threadIdx.x; e < vecs_per_row; e += blockDim.x) {
    kd[e] = quantize8(__ldg(ks + e), k_scale);
    vd[e] = quantize8(__ldg(vs + e), v_scale);
  }
}

// The E4M3 cache write with its slot mapping in one launch, as
// cache_write_mapped_kernel does for 16-bit pools.
template <bool kBF16>
__global__ void cache_write_fp8_mapped_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int32_t* __restrict__ bt,
    int stride, int num_seqs, const int32_t* __restrict__ tok_seq,
    const int32_t* __restrict__ tok_pos, int log2B, long long num_blocks, int vecs_per_row,
    uint2* __restrict__ kc, uint2* __restrict__ vc, float k_scale, float v_scale,
    int64_t* __restrict__ slots, int32_t* err) {
  __shared__ long long s_slot;
  grid_dep_wait();
  grid_dep_launch();
  const long long tok = blockIdx.x;
  const uint4* ks = k + tok * vecs_per_row;
  const uint4* vs = v + tok * vecs_per_row;
  const int e0 = threadIdx.x;
  uint4 a0 = make_uint4(0u, 0u, 0u, 0u), b0 = a0;
  if (e0 < vecs_per_row) {
    a0 = __ldg(ks + e0);
    b0 = __ldg(vs + e0);
  }
  if (threadIdx.x == 0) {
    const long long sl = token_slot(bt, stride, num_seqs, tok_seq, tok_pos, tok, log2B,
                                    num_blocks, err);
    if (slots) slots[tok] = sl;
    s_slot = sl;
  }
  __syncthreads();
  const long long sl = s_slot;
  if (sl < 0) return;
  auto quantize8 = [](const uint4 x, float scale) -> uint2 {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack2<kBF16>(w[i]);
      c[i] = f32x2_to_e4m3x2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
    }
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  };
  uint2* kd = kc + sl * vecs_per_row;
  uint2* vd = vc + sl * vecs_per_row;
  if (e0 < vecs_per_row) {
    kd[e0] = quantize8(a0, k_scale);
    vd[e0] = quantize8(b0, v_scale);
  }
  for (int e = e0 + blockDim.x; e < vecs_per_row; e += blockDim.x) {
    kd[e] = quantize8(__ldg(ks + e), k_scale);
    vd[e] = quantize8(__ldg(vs + e), v_scale);
  }
}

// Pair validation for the block copy and the block swap, in time linear in
// the number of pairs.  Each thread block owns a contiguous range of at most
// kPairsPerCta pairs.  It puts its own pairs' dst blocks in a hash table in
// shared memory (key and local index in one 64-bit word, open addressing),
// then reads every pair of the list once and looks its src and its dst up:
//   * a dst that is some pair's src (block copy only: both sides address the
//     same pool) makes the owning pair invalid;
//   * a dst that is another pair's dst makes both invalid;
//   * a src or dst outside its pool makes the pair invalid.
// The grid is bounded by a small multiple of the SM count, so the whole check
// reads the list once per thread block: O(num_pairs) per block, with no
// device memory beyond the inputs.
constexpr int kPairsPerCta = 512;
constexpr int kPairHash = 1024;              // table slots (power of two, twice the pairs)
constexpr unsigned long long kHashEmpty = ~0ull;

__device__ __forceinline__ unsigned pair_hash(int key) {
  return ((unsigned)key * 2654435761u) >> (32 - 10);   // kPairHash = 2^10
}

// Marks bad[i] for the invalid pairs among the m pairs from p0; the caller
// syncs after.  table: kPairHash words of shared memory.
__device__ __forceinline__ void validate_pairs(const int32_t* __restrict__ pairs, int num_pairs,
                                               int p0, int m, long long src_blocks,
                                               long long dst_blocks, bool dst_may_be_src,
                                               unsigned long long* table, unsigned char* bad) {
  for (int i = threadIdx.x; i < kPairHash; i += blockDim.x) table[i] = kHashEmpty;
  for (int i = threadIdx.x; i < m; i += blockDim.x) bad[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const int src = pairs[2 * (p0 + i)], dst = pairs[2 * (p0 + i) + 1];
    if (src < 0 || (long long)src >= src_blocks || dst < 0 || (long long)dst >= dst_blocks) {
      bad[i] = 1;
      continue;
    }
    const unsigned long long word = ((unsigned long long)(unsigned)dst << 32) | (unsigned)i;
    for (unsigned h = pair_hash(dst);; h = (h + 1) & (kPairHash - 1)) {
      const unsigned long long prev = atomicCAS(&table[h], kHashEmpty, word);
      if (prev == kHashEmpty) break;
      if ((int)(prev >> 32) == dst) {   // two own pairs share a dst
        bad[i] = 1;
        bad[(unsigned)prev] = 1;
        break;
      }
    }
  }
  __syncthreads();
  auto find = [&](int key) -> int {   // local index of the own pair with dst == key, or -1
    for (unsigned h = pair_hash(key);; h = (h + 1) & (kPairHash - 1)) {
      const unsigned long long w = table[h];
      if (w == kHashEmpty) return -1;
      if ((int)(w >> 32) == key) return (int)(unsigned)w;
    }
  };
  for (int j = threadIdx.x; j < num_pairs; j += blockDim.x) {
    const int sj = pairs[2 * j], dj = pairs[2 * j + 1];
    if (dst_may_be_src) {
      const int a = find(sj);   // an own dst that is pair j's src
      if (a >= 0) bad[a] = 1;
    }
    const int b = find(dj);     // an own dst that is pair j's dst too
    if (b >= 0 && p0 + b != j) bad[b] = 1;
  }
}

// Copies the valid pairs among the m pairs from p0, K and V blocks, in 16-byte
// vectors, four loads in flight per thread.
__device__ __forceinline__ void copy_valid_pairs(const int32_t* __restrict__ pairs, int p0, int m,
                                                 int vecs_per_block, const unsigned char* bad,
                                                 const uint4* src_k, const uint4* src_v,
                                                 uint4* dst_k, uint4* dst_v) {
  for (int i = 0; i < m; ++i) {
    if (bad[i]) continue;
    const long long src = pairs[2 * (p0 + i)], dst = pairs[2 * (p0 + i) + 1];
    const uint4* sk = src_k + src * vecs_per_block;
    const uint4* sv = src_v + src * vecs_per_block;
    uint4* dk = dst_k + dst * vecs_per_block;
    uint4* dv = dst_v + dst * vecs_per_block;
    const int n = 2 * vecs_per_block;
    int e = threadIdx.x;
    for (; e + 3 * (int)blockDim.x < n; e += 4 * blockDim.x) {
      uint4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int f = e + u * blockDim.x;
        x[u] = f < vecs_per_block ? sk[f] : sv[f - vecs_per_block];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int f = e + u * blockDim.x;
        if (f < vecs_per_block) dk[f] = x[u];
        else dv[f - vecs_per_block] = x[u];
      }
    }
    for (; e < n; e += blockDim.x) {
      if (e < vecs_per_block) dk[e] = sk[e];
      else dv[e - vecs_per_block] = sv[e - vecs_per_block];
    }
  }
}

// Copy-on-write block copy: thread block b owns pairs [b * per_cta, ...).  A
// pair is copied only if it is in range, its dst appears once among the dsts
// and is no pair's src.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const int32_t* __restrict__ pairs,
                                                          int num_pairs, int per_cta,
                                                          long long num_blocks, int vecs_per_block,
                                                          uint4* kc, uint4* vc, int32_t* err) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ unsigned long long table[kPairHash];
  __shared__ unsigned char bad[kPairsPerCta];
  __shared__ int any_bad;
  const int p0 = blockIdx.x * per_cta;
  const int m = min(per_cta, num_pairs - p0);
  if (m <= 0) return;
  validate_pairs(pairs, num_pairs, p0, m, num_blocks, num_blocks, true, table, bad);
  if (threadIdx.x == 0) any_bad = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < m; i += blockDim.x)
    if (bad[i]) any_bad = 1;
  __syncthreads();
  if (threadIdx.x == 0 && any_bad) set_error(err, PA_DEVERR_COPY_PAIR);
  copy_valid_pairs(pairs, p0, m, vecs_per_block, bad, kc, vc, kc, vc);
}

// Block swap between the device pool and a pinned host pool ("vLLM anatomy",
// section "Memory Pressure and Preemption": swapping moves physical blocks from
// GPU memory to the CPU's memory and back).  Thread block b owns pairs
// [b * per_cta, ...) and copies them in 16-byte vectors; the host pool is
// addressed through its mapped device address, so any number of blocks moves
// in one launch (over NVLink-C2C on a Grace-Blackwell node).  A pair is copied
// only if both blocks are in range and its dst appears once among the dsts.
__global__ void __launch_bounds__(256) swap_blocks_kernel(
    const int32_t* __restrict__ pairs, int num_pairs, int per_cta, long long src_blocks,
    long long dst_blocks, int vecs_per_block, const uint4* __restrict__ src_k,
    const uint4* __restrict__ src_v, uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
    int32_t* err) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ unsigned long long table[kPairHash];
  __shared__ unsigned char bad[kPairsPerCta];
  __shared__ int any_bad;
  const int p0 = blockIdx.x * per_cta;
  const int m = min(per_cta, num_pairs - p0);
  if (m <= 0) return;
  validate_pairs(pairs, num_pairs, p0, m, src_blocks, dst_blocks, false, table, bad);
  if (threadIdx.x == 0) any_bad = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < m; i += blockDim.x)
    if (bad[i]) any_bad = 1;
  __syncthreads();
  if (threadIdx.x == 0 && any_bad) set_error(err, PA_DEVERR_COPY_PAIR);
  copy_valid_pairs(pairs, p0, m, vecs_per_block, bad, src_k, src_v, dst_k, dst_v);
}

// Pairs per thread block for a list of n pairs: at most kPairsPerCta, and
// enough blocks (two per SM) to keep the copies spread over the GPU.
static int pairs_per_cta(int n, int sm_count) {
  const int target_ctas = 2 * sm_count;
  int per = (n + target_ctas - 1) / target_ctas;
  if (per < 1) per = 1;
  if (per > kPairsPerCta) per = kPairsPerCta;
  return per;
}

static bool shape_ok(int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                     bool allow_fp8 = false) {
  return (head_dim == 64 || head_dim == 128) && num_kv_heads > 0 && is_pow2(block_size) &&
         block_size <= 256 &&
         (dtype == PA_F16 || dtype == PA_BF16 || (allow_fp8 && dtype == PA_FP8_E4M3));
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_slot_mapping(const int32_t* block_tables, int32_t table_stride, int32_t num_seqs,
                    const int32_t* token_seq, const int32_t* token_pos, int64_t num_tokens,
                    int32_t block_size, int64_t num_blocks, int64_t* slot_mapping,
                    int32_t* err_word, pa_stream stream) {
  if (num_tokens < 0 || num_seqs < 0 || table_stride < 0 || num_blocks < 0)
    return PA_ERR_INVALID_ARG;
  if (!is_pow2(block_size)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!block_tables || !token_seq || !token_pos || !slot_mapping) return PA_ERR_INVALID_ARG;
  DeviceInfo di;
  if (int rc = current_device_info(&di)) return rc;
  const int threads = 256;
  long long blocks = (num_tokens + threads - 1) / threads;
  if (blocks > (long long)di.sm_count * 16) blocks = (long long)di.sm_count * 16;
  clear_stale_error();
  return launch_status(launch_pdl(slot_mapping_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                                  static_cast<cudaStream_t>(stream), block_tables,
                                  (int)table_stride, (int)num_seqs, token_seq, token_pos,
                                  (long long)num_tokens, ilog2(block_size), (long long)num_blocks,
                                  slot_mapping, err_word),
                       "slot mapping launch");
}

int pa_cache_write(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                   void* k_cache, void* v_cache, int64_t num_blocks, int32_t block_size,
                   int32_t num_kv_heads, int32_t head_dim, int32_t dtype, int32_t* err_word,
                   pa_stream stream) {
  if (num_tokens < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  if (!shape_ok(block_size, num_kv_heads, head_dim, dtype)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (num_tokens > 0x7fffffffLL) return PA_ERR_INVALID_ARG;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int vecs = num_kv_heads * head_dim * 2 / 16;
  const int threads = vecs >= 256 ? 256 : (vecs >= 128 ? 128 : 64);
  clear_stale_error();
  return launch_status(launch_pdl(cache_write_kernel, dim3((unsigned)num_tokens), dim3(threads), 0,
                                  static_cast<cudaStream_t>(stream),
                                  static_cast<const uint4*>(k), static_cast<const uint4*>(v),
                                  slot_mapping, vecs, num_blocks * (long long)block_size,
                                  static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                                  err_word),
                       "cache write launch");
}

int pa_cache_write_mapped(const void* k, const void* v, const int32_t* block_tables,
                          int32_t table_stride, int32_t num_seqs, const int32_t* token_seq,
                          const int32_t* token_pos, int64_t num_tokens, void* k_cache,
                          void* v_cache, int64_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                          int64_t* slot_mapping, int32_t* err_word, pa_stream stream) {
  if (num_tokens < 0 || num_seqs < 0 || table_stride < 0 || num_blocks < 0)
    return PA_ERR_INVALID_ARG;
  if (!shape_ok(block_size, num_kv_heads, head_dim, dtype)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (num_tokens > 0x7fffffffLL) return PA_ERR_INVALID_ARG;
  if (!k || !v || !block_tables || !token_seq || !token_pos || !k_cache || !v_cache)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int vecs = num_kv_heads * head_dim * 2 / 16;
  const int threads = vecs >= 256 ? 256 : (vecs >= 128 ? 128 : 64);
  clear_stale_error();
  return launch_status(
      launch_pdl(cache_write_mapped_kernel, dim3((unsigned)num_tokens), dim3(threads), 0,
                 static_cast<cudaStream_t>(stream), static_cast<const uint4*>(k),
                 static_cast<const uint4*>(v), block_tables, (int)table_stride, (int)num_seqs,
                 token_seq, token_pos, ilog2(block_size), (long long)num_blocks, vecs,
                 static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping,
                 err_word),
      "slot-mapped cache write launch");
}

int pa_copy_blocks(const int32_t* src_dst_pairs, int32_t num_pairs, void* k_cache, void* v_cache,
                   int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                   int32_t head_dim, int32_t dtype, int32_t* err_word, pa_stream stream) {
  if (num_pairs < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  if (!shape_ok(block_size, num_kv_heads, head_dim, dtype, true)) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (num_pairs > 65535) return PA_ERR_INVALID_ARG;
  if (!src_dst_pairs || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
  const int eb = dtype == PA_FP8_E4M3 ? 1 : 2;
  const long long vecs = (long long)block_size * num_kv_heads * head_dim * eb / 16;
  if (vecs > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  DeviceInfo di;
  if (int rc = current_device_info(&di)) return rc;
  const int per = pairs_per_cta(num_pairs, di.sm_count);
  const unsigned ctas = (unsigned)((num_pairs + per - 1) / per);
  clear_stale_error();
  return launch_status(launch_pdl(copy_blocks_kernel, dim3(ctas), dim3(256), 0,
                                  static_cast<cudaStream_t>(stream), src_dst_pairs,
                                  (int)num_pairs, per, (long long)num_blocks, (int)vecs,
                                  static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                                  err_word),
                       "block copy launch");
}

int pa_swap_blocks(const int32_t* src_dst_pairs, int32_t num_pairs, int32_t direction,
                   void* dev_k, void* dev_v, int64_t dev_num_blocks, void* host_k, void* host_v,
                   int64_t host_num_blocks, int32_t block_size, int32_t num_kv_heads,
                   int32_t head_dim, int32_t dtype, int32_t* err_word, pa_stream stream) {
  if (num_pairs < 0 || dev_num_blocks < 0 || host_num_blocks < 0) return PA_ERR_INVALID_ARG;
  if (direction != PA_SWAP_OUT && direction != PA_SWAP_IN) return PA_ERR_INVALID_ARG;
  if (!shape_ok(block_size, num_kv_heads, head_dim, dtype, true)) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (num_pairs > 65535) return PA_ERR_INVALID_ARG;
  if (!src_dst_pairs || !dev_k || !dev_v || !host_k || !host_v) return PA_ERR_INVALID_ARG;
  if (!aligned16(dev_k) || !aligned16(dev_v) || !aligned16(host_k) || !aligned16(host_v))
    return PA_ERR_INVALID_ARG;
  // the device-side addresses of the host pool (pinned and mapped memory, or
  // pageable memory where the GPU reads the host's page tables)
  void* hk = nullptr;
  void* hv = nullptr;
  if (cudaHostGetDevicePointer(&hk, host_k, 0) != cudaSuccess ||
      cudaHostGetDevicePointer(&hv, host_v, 0) != cudaSuccess) {
    cudaGetLastError();   // not addressable from the GPU: the caller's error, not a sticky one
    return PA_ERR_INVALID_ARG;
  }
  const int eb = dtype == PA_FP8_E4M3 ? 1 : 2;
  const long long vecs = (long long)block_size * num_kv_heads * head_dim * eb / 16;
  if (vecs > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  const bool out = direction == PA_SWAP_OUT;
  DeviceInfo di;
  if (int rc = current_device_info(&di)) return rc;
  const int per = pairs_per_cta(num_pairs, di.sm_count);
  const unsigned ctas = (unsigned)((num_pairs + per - 1) / per);
  clear_stale_error();
  const cudaError_t e = launch_pdl(
      swap_blocks_kernel, dim3(ctas), dim3(256), 0,
      static_cast<cudaStream_t>(stream), src_dst_pairs, (int)num_pairs, per,
      (long long)(out ? dev_num_blocks : host_num_blocks),
      (long long)(out ? host_num_blocks : dev_num_blocks), (int)vecs,
      static_cast<const uint4*>(out ? dev_k : hk), static_cast<const uint4*>(out ? dev_v : hv),
      static_cast<uint4*>(out ? hk : dev_k), static_cast<uint4*>(out ? hv : dev_v), err_word);
  return launch_status(e, "block swap launch");
}

int pa_cache_write_fp8(const void* k, const void* v, int32_t src_dtype,
                       const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                       void* v_cache, int64_t num_blocks, int32_t block_size,
                       int32_t num_kv_heads, int32_t head_dim, float k_scale, float v_scale,
                       int32_t* err_word, pa_stream stream) {
  if (num_tokens < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  if (!shape_ok(block_size, num_kv_heads, head_dim, src_dtype)) return PA_ERR_UNSUPPORTED;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale > 3.0e38f || v_scale > 3.0e38f)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (num_tokens > 0x7fffffffLL) return PA_ERR_INVALID_ARG;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int vecs = num_kv_heads * head_dim / 8;   // 16-byte input vectors per row
  const int threads = vecs >= 256 ? 256 : (vecs >= 128 ? 128 : 64);
  clear_stale_error();
  const long long num_slots = num_blocks * (long long)block_size;
  cudaError_t e =
      src_dtype == PA_BF16
          ? launch_pdl(cache_write_fp8_kernel<true>, dim3((unsigned)num_tokens), dim3(threads), 0,
                       static_cast<cudaStream_t>(stream), static_cast<const uint4*>(k),
                       static_cast<const uint4*>(v), slot_mapping, vecs, num_slots,
                       static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), k_scale,
                       v_scale, err_word)
          : launch_pdl(cache_write_fp8_kernel<false>, dim3((unsigned)num_tokens), dim3(threads), 0,
                       static_cast<cudaStream_t>(stream), static_cast<const uint4*>(k),
                       static_cast<const uint4*>(v), slot_mapping, vecs, num_slots,
                       static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), k_scale,
                       v_scale, err_word);
  return launch_status(e, "E4M3 cache write launch");
}

int pa_cache_write_fp8_mapped(const void* k, const void* v, int32_t src_dtype,
                              const int32_t* block_tables, int32_t table_stride, int32_t num_seqs,
                              const int32_t* token_seq, const int32_t* token_pos,
                              int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                              int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                              float k_scale, float v_scale, int64_t* slot_mapping,
                              int32_t* err_word, pa_stream stream) {
  if (num_tokens < 0 || num_seqs < 0 || table_stride < 0 || num_blocks < 0)
    return PA_ERR_INVALID_ARG;
  if (!shape_ok(block_size, num_kv_heads, head_dim, src_dtype)) return PA_ERR_UNSUPPORTED;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale > 3.0e38f || v_scale > 3.0e38f)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (num_tokens > 0x7fffffffLL) return PA_ERR_INVALID_ARG;
  if (!k || !v || !block_tables || !token_seq || !token_pos || !k_cache || !v_cache)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int vecs = num_kv_heads * head_dim / 8;   // 16-byte input vectors per row
  const int threads = vecs >= 256 ? 256 : (vecs >= 128 ? 128 : 64);
  clear_stale_error();
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int log2B = ilog2(block_size);
  cudaError_t e =
      src_dtype == PA_BF16
          ? launch_pdl(cache_write_fp8_mapped_kernel<true>, dim3((unsigned)num_tokens),
                       dim3(threads), 0, s, static_cast<const uint4*>(k),
                       static_cast<const uint4*>(v), block_tables, (int)table_stride,
                       (int)num_seqs, token_seq, token_pos, log2B, (long long)num_blocks, vecs,
                       static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), k_scale,
                       v_scale, slot_mapping, err_word)
          : launch_pdl(cache_write_fp8_mapped_kernel<false>, dim3((unsigned)num_tokens),
                       dim3(threads), 0, s, static_cast<const uint4*>(k),
                       static_cast<const uint4*>(v), block_tables, (int)table_stride,
                       (int)num_seqs, token_seq, token_pos, log2B, (long long)num_blocks, vecs,
                       static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), k_scale,
                       v_scale, slot_mapping, err_word);
  return launch_status(e, "slot-mapped E4M3 cache write launch");
}

}  // extern "C"
