/*
 * pa.h -- C ABI of the paged KV-cache library (GB300, sm_103a).
 *
 * The data-parallel hot path of PagedAttention: slot mapping, the slot-mapped
 * cache write, the copy-on-write block copy and single-query decode attention
 * over a block-paged KV pool, with its split-context reduce.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "vLLM Framework and Inference Engine Design" (vineetganti.com)
 *   [P3] "vLLM anatomy: high-throughput LLM inference" (karya-semi.vercel.app)
 *   [P5] "vLLM" (bibekananda.in)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All data pointers are DEVICE pointers, owned by the caller.  The library
 *    allocates no device memory and keeps no per-call state.  Buffers must be
 *    16-byte aligned.
 *  - KV pool, one per layer and per K/V ([P1] "What is the essence of vLLM's
 *    PagedAttention?"; "How is vLLM's KV cache paged?"): a contiguous array
 *        cache[num_blocks][block_size][num_kv_heads][head_dim]
 *    of 16-bit elements (PA_F16: IEEE binary16, PA_BF16: bfloat16).
 *  - Block tables: int32 [num_seqs][table_stride], row i lists the physical
 *    blocks of sequence i in logical order; entries past
 *    ceil(seq_lens[i] / block_size) are never read.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Host-detectable errors return a PA_ERR_* status before
 *    anything is launched.  Bad indices met on the device never fault and never
 *    trap: the access is skipped, a PA_DEVERR_* bit is OR-ed into *err_word
 *    (an int32 device word, may be NULL), and pa_get_error() reports it.
 *  - Supported shapes: head_dim in {64, 128}; block_size a power of two in
 *    [1, 256] ([2, 256] for pa_decode and pa_gather_kv); num_q_heads a
 *    multiple of num_kv_heads with group G = num_q_heads / num_kv_heads in
 *    [1, 16].
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
#define PA_F16 0
#define PA_BF16 1
/* E4M3 KV-cache codes (pools only; see pa_cache_write_fp8 / pa_decode_fp8) */
#define PA_FP8_E4M3 2

/* status codes returned by the entry points */
#define PA_OK 0
#define PA_ERR_INVALID_ARG 1   /* null pointer, negative size, misaligned buffer, bad shape */
#define PA_ERR_UNSUPPORTED 2   /* shape outside the compiled kernels */
#define PA_ERR_WORKSPACE 3     /* decode workspace smaller than pa_decode_workspace_size() */
#define PA_ERR_CUDA 4          /* a CUDA runtime or driver call failed */
#define PA_ERR_DEVICE_INDEX 5  /* pa_get_error(): a kernel reported a PA_DEVERR_* bit */

/* bits a kernel ORs into *err_word */
#define PA_DEVERR_SLOT 0x1       /* slot_mapping entry >= num_blocks * block_size */
#define PA_DEVERR_BLOCK_ID 0x2   /* block-table entry outside [0, num_blocks) */
#define PA_DEVERR_SEQ_LEN 0x4    /* seq_len < 0 or > table_stride * block_size */
#define PA_DEVERR_COPY_PAIR 0x8  /* copy pair out of range, repeated dst, or dst that is a src */
#define PA_DEVERR_TIMEOUT 0x10   /* a pipeline wait passed its bound; the result is invalid */
#define PA_DEVERR_POSITION 0x20  /* slot mapping: sequence index or position outside its table */

/* pa_swap_blocks directions */
#define PA_SWAP_OUT 0   /* device pool -> host pool */
#define PA_SWAP_IN 1    /* host pool -> device pool */

/* pa_decode flags */
#define PA_DECODE_AUTO 0
#define PA_DECODE_SIMT 1  /* CUDA-core kernel (group size 1 only) */
#define PA_DECODE_MMA 2   /* tensor-core kernel (any supported group size) */
/* OR-ed into the flags of pa_decode, pa_decode_window and pa_decode_fp8: the
 * caller promises that seq_lens and block_tables are complete before the
 * preceding kernel in the stream starts (as a serving step's metadata is).
 * The decode then reads them while that kernel drains, under programmatic
 * dependent launch; q, the pools, out and the workspace are still touched
 * only after it completes. */
#define PA_DECODE_TABLES_READY 0x100

typedef void* pa_stream; /* cudaStream_t */

/*
 * pa_slot_mapping -- flat cache slot of each new token.
 * [P1] "How is vLLM's KV cache paged?", bullet "Writing": a token at position t
 * of a sequence is stored at slot block_table[floor(t/B)] * B + (t mod B).
 *   block_tables  int32 [num_seqs][table_stride]
 *   token_seq     int32 [num_tokens]  sequence index of each new token
 *   token_pos     int32 [num_tokens]  its position t within the sequence
 *   slot_mapping  int64 [num_tokens]  output
 * A token whose sequence index is outside [0, num_seqs) or whose position is
 * outside the table row gets slot -1 and sets PA_DEVERR_POSITION; a table entry
 * outside [0, num_blocks) gives slot -1 and sets PA_DEVERR_BLOCK_ID.
 * num_tokens == 0 is a no-op.
 */
int pa_slot_mapping(const int32_t* block_tables, int32_t table_stride, int32_t num_seqs,
                    const int32_t* token_seq, const int32_t* token_pos, int64_t num_tokens,
                    int32_t block_size, int64_t num_blocks, int64_t* slot_mapping,
                    int32_t* err_word, pa_stream stream);

/*
 * pa_cache_write -- store each new token's K and V rows at its slot.
 * [P1] "How is vLLM's KV cache paged?", bullet "Writing" (the slot mapping);
 * [P1] "What is the essence of vLLM's PagedAttention?" (K_cache[p][r]).
 *   k, v          [num_tokens][num_kv_heads][head_dim], contiguous, dtype
 *   slot_mapping  int64 [num_tokens]; slot s addresses block s / B, row s % B;
 *                 s < 0 marks a padding token that writes nothing;
 *                 s >= num_blocks * B sets PA_DEVERR_SLOT and writes nothing.
 * Bit-exact copy.  Two tokens with the same slot: one of them wins.
 */
int pa_cache_write(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                   void* k_cache, void* v_cache, int64_t num_blocks, int32_t block_size,
                   int32_t num_kv_heads, int32_t head_dim, int32_t dtype, int32_t* err_word,
                   pa_stream stream);

/*
 * pa_cache_write_mapped -- pa_slot_mapping and pa_cache_write in one launch.
 * [P1] "How is vLLM's KV cache paged?", bullet "Writing": each new token at
 * position t of sequence i is stored at slot block_table[i][t / B] * B + t % B.
 * Arguments as in those two calls: block_tables int32 [num_seqs][table_stride],
 * token_seq / token_pos int32 [num_tokens], k, v [num_tokens][num_kv_heads]
 * [head_dim] contiguous in the pool dtype (PA_F16 or PA_BF16).  slot_mapping,
 * int64 [num_tokens], receives the slots when not NULL.  A token with a bad
 * sequence index or position (PA_DEVERR_POSITION) or table entry
 * (PA_DEVERR_BLOCK_ID) gets slot -1 and writes nothing.  The pools and
 * err_word end as after pa_slot_mapping followed by pa_cache_write.
 */
int pa_cache_write_mapped(const void* k, const void* v, const int32_t* block_tables,
                          int32_t table_stride, int32_t num_seqs, const int32_t* token_seq,
                          const int32_t* token_pos, int64_t num_tokens, void* k_cache,
                          void* v_cache, int64_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                          int64_t* slot_mapping, int32_t* err_word, pa_stream stream);

/*
 * pa_copy_blocks -- copy-on-write block copies.
 * [P1] "What operations can cause memory fragmentation, and how does vLLM avoid
 * it?", bullet "Sharing instead of copying": a shared block is copied only when
 * a sequence needs to write into it; [P5] "The part that is easy to miss".
 *   src_dst_pairs int32 [num_pairs][2] (src block, dst block), device memory.
 * Every pair copies all block_size * num_kv_heads * head_dim elements of K and
 * of V from src to dst.  Pairs are independent: dst blocks must be distinct and
 * no dst may also be a src.  A pair out of range, or one that breaks this rule,
 * sets PA_DEVERR_COPY_PAIR and is not copied.  dtype PA_FP8_E4M3 copies pools
 * of 1-byte codes.
 */
int pa_copy_blocks(const int32_t* src_dst_pairs, int32_t num_pairs, void* k_cache, void* v_cache,
                   int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                   int32_t head_dim, int32_t dtype, int32_t* err_word, pa_stream stream);

/*
 * pa_swap_blocks -- move whole blocks between the device pool and a host pool.
 * [P3] "Memory Pressure and Preemption": swapping moves physical blocks from
 * GPU memory to the CPU's system memory and, when GPU memory is free again,
 * back; [P1] notes the V1 engine preempts by recomputation instead.
 *   src_dst_pairs int32 [num_pairs][2] in device memory: (src block, dst
 *                 block); src in the source pool, dst in the destination pool
 *   direction     PA_SWAP_OUT: device -> host; PA_SWAP_IN: host -> device
 *   dev_k, dev_v  device pools [dev_num_blocks][block_size][num_kv_heads][head_dim]
 *   host_k, host_v  host pools of the same block shape that the GPU can
 *                 address: pinned, mapped memory (cudaHostAlloc /
 *                 cudaMallocHost), or, on a node whose GPU reads pageable host
 *                 memory through the host's page tables (a Grace-Blackwell
 *                 node over NVLink-C2C), any host memory; memory that
 *                 cudaHostGetDevicePointer cannot translate returns
 *                 PA_ERR_INVALID_ARG
 *   dtype         PA_F16, PA_BF16 or PA_FP8_E4M3 (1-byte codes)
 * One kernel launch copies every pair (K and V), bit-exact, reading or
 * writing the host pool through its mapped device address.  A pair out of
 * range, or a dst that appears twice, sets PA_DEVERR_COPY_PAIR and is not
 * copied.  Stream-ordered like every call.
 */
int pa_swap_blocks(const int32_t* src_dst_pairs, int32_t num_pairs, int32_t direction,
                   void* dev_k, void* dev_v, int64_t dev_num_blocks, void* host_k, void* host_v,
                   int64_t host_num_blocks, int32_t block_size, int32_t num_kv_heads,
                   int32_t head_dim, int32_t dtype, int32_t* err_word, pa_stream stream);

/*
 * pa_cache_write_fp8 -- pa_cache_write into an E4M3 (FP8) KV cache.
 * [P1] "How can one customize the tokenizer, cache strategy, or scheduler
 * strategy?" (kv_cache_dtype="fp8": half the KV memory of FP16); [P3]
 * "Quantization: Reducing Weight & KV Precision" (--kv-cache-dtype fp8).  The
 * pages name neither the 8-bit format nor a scale; our reading is OCP E4M3
 * with one scale per tensor:
 *   code = e4m3(float32(x) / scale), rounded to nearest even, magnitudes
 *   beyond 448 saturating to +-448; the code stands for e4m3(code) * scale.
 *   k, v          [num_tokens][num_kv_heads][head_dim], contiguous, src_dtype
 *                 (PA_F16 or PA_BF16), finite
 *   k_cache, v_cache  uint8 [num_blocks][block_size][num_kv_heads][head_dim]
 *   k_scale, v_scale  finite and > 0
 * Slots as for pa_cache_write.  The division is IEEE binary32 and the codes
 * are bit-exact.
 */
int pa_cache_write_fp8(const void* k, const void* v, int32_t src_dtype,
                       const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                       void* v_cache, int64_t num_blocks, int32_t block_size,
                       int32_t num_kv_heads, int32_t head_dim, float k_scale, float v_scale,
                       int32_t* err_word, pa_stream stream);

/*
 * pa_cache_write_fp8_mapped -- pa_slot_mapping and pa_cache_write_fp8 in one
 * launch.  [P1] "How is vLLM's KV cache paged?", bullet "Writing" (the slots);
 * the E4M3 reading of pa_cache_write_fp8 (the codes).  Arguments as in those
 * two calls; slot_mapping, int64 [num_tokens], receives the slots when not
 * NULL.  A bad token gets slot -1 and writes nothing, with the error bits of
 * pa_slot_mapping.  The pools and err_word end as after the two calls.
 */
int pa_cache_write_fp8_mapped(const void* k, const void* v, int32_t src_dtype,
                              const int32_t* block_tables, int32_t table_stride, int32_t num_seqs,
                              const int32_t* token_seq, const int32_t* token_pos,
                              int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                              int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                              float k_scale, float v_scale, int64_t* slot_mapping,
                              int32_t* err_word, pa_stream stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs for
 * this shape on the current device: a fixed region of PA_DECODE_MAX_CTAS
 * 32-bit piece counters, then the partial softmax states of contexts split
 * across thread blocks (two per block of the grid).  Because the counters sit
 * at the same place whatever the shape or grid, one workspace sized for the
 * largest call serves calls of any shape and num_ctas.  num_ctas = 0 selects
 * the default grid (a multiple of the SM count); larger than
 * PA_DECODE_MAX_CTAS returns PA_ERR_INVALID_ARG; flags as for pa_decode.
 * dtype PA_FP8_E4M3 sizes the workspace of pa_decode_fp8.
 */
#define PA_DECODE_MAX_CTAS 16384
int pa_decode_workspace_size(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t dtype, int32_t flags, int32_t num_ctas,
                             size_t* bytes);

/*
 * pa_decode -- single-query decode attention over the paged KV pool.
 * [P1] "What is the essence of vLLM's PagedAttention?": the kernel follows the
 * block table (token t -> block block_table[floor(t/B)], row t mod B) instead
 * of reading one contiguous tensor; scores = q.K^T * scale, weights =
 * softmax(scores), output = weights.V.  [P3] "Custom CUDA Kernels for
 * PagedAttention": decode attention is memory-bound; the kernel reads the block
 * table on the GPU and fetches the scattered blocks in parallel.
 *   q          [num_seqs][num_q_heads][head_dim], contiguous, dtype
 *   seq_lens   int32 [num_seqs]: tokens in the cache, including the token
 *              written this step; 0 gives a zero output row
 *   out        [num_seqs][num_q_heads][head_dim], dtype; must not alias q
 *   scale      multiplies q.k (e.g. 1/sqrt(head_dim))
 *   workspace  device buffer of at least pa_decode_workspace_size() bytes,
 *              zero-filled before its first use; every call that runs to its
 *              end (device errors included) leaves it zero-ready for the next
 *              call.  One exception: seq_lens changing while the call reads
 *              it (a caller error) can leave a thread block unable to find
 *              its work; it reports PA_DEVERR_SEQ_LEN without counting its
 *              pieces, and the workspace must be zero-filled again.  Calls
 *              sharing one workspace must not overlap on the GPU.
 * Query head hq reads KV head hq / G (contiguous query groups).  Accumulation
 * is fp32; the output is rounded once to dtype.  The result does not depend on
 * where the blocks sit in the pool.  The work (chunks of one block's worth of
 * tokens of up to 8 KV heads) is split evenly over a persistent grid; each
 * piece of a context split between thread blocks leaves its partial softmax
 * state in the workspace and counts itself, and the block whose piece
 * completes the count merges them (one kernel launch, no block waits for
 * another, any num_ctas).
 * flags: PA_DECODE_AUTO, PA_DECODE_SIMT or PA_DECODE_MMA, optionally OR-ed with
 * PA_DECODE_TABLES_READY; num_ctas: 0 = default.
 */
int pa_decode(const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
              int32_t block_size, int64_t num_blocks, int32_t dtype, float scale, void* out,
              void* workspace, size_t workspace_bytes, int32_t flags, int32_t num_ctas,
              int32_t* err_word, pa_stream stream);

/*
 * pa_decode_window -- pa_decode with sliding-window attention.
 * [P1] "How does it support prompts of arbitrary length? Does it have a
 * sliding window?": in a model trained with sliding-window attention each
 * token attends only to the last W tokens, so only the blocks inside the
 * window are needed and the older ones can be released (at most
 * ceil(W / B) + 1 blocks per sequence).  The query of position T - 1 attends
 * to tokens [max(0, T - window), T) (our reading of "the last W tokens").
 *   window        >= 1 (tokens)
 *   block_tables  logical indexing as for pa_decode; the entries of blocks
 *                 wholly before the block that holds token max(0, T - window)
 *                 are never read and may hold anything (a released block, -1)
 * Every other argument, the errors and the workspace are those of pa_decode.
 */
int pa_decode_window(const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
                     int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t dtype,
                     float scale, int32_t window, void* out, void* workspace,
                     size_t workspace_bytes, int32_t flags, int32_t num_ctas, int32_t* err_word,
                     pa_stream stream);

/*
 * pa_decode_fp8 -- pa_decode over E4M3 pools written by pa_cache_write_fp8.
 * Computes out = softmax(scale * q . K^T) . V with K = e4m3(code_K) * k_scale
 * and V = e4m3(code_V) * v_scale ([P1] "What is the essence of vLLM's
 * PagedAttention?", on the dequantized cache).  The scales are applied outside
 * the products (k_scale joins `scale`, v_scale multiplies the output); the
 * codes convert exactly to binary16, queries in bfloat16 are converted to
 * binary16 (their magnitudes must stay within binary16's range), the softmax
 * weights are binary16 and every sum is fp32.
 *   q, out        [num_seqs][num_q_heads][head_dim] in q_dtype (PA_F16 or PA_BF16)
 *   k_cache, v_cache  uint8 E4M3 pools [num_blocks][block_size][num_kv_heads][head_dim]
 *   workspace     as for pa_decode, sized by pa_decode_workspace_size with
 *                 dtype PA_FP8_E4M3
 * Every other argument, the errors and the workspace rules are those of
 * pa_decode.  pa_gather_kv does not take E4M3 pools.
 */
int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t block_size, int64_t num_blocks, int32_t q_dtype, float scale,
                  float k_scale, float v_scale, void* out, void* workspace,
                  size_t workspace_bytes, int32_t flags, int32_t num_ctas, int32_t* err_word,
                  pa_stream stream);

/*
 * pa_prefill -- multi-query paged attention for chunked prefill, with decode
 * tokens allowed in the same batch.
 * [P1] "How does it support prompts of arbitrary length?": a long prompt is
 * processed in chunks, which run in one batch with other requests' decode
 * tokens; [P4] "Two phases: prefill and decode".  Sequence i brings
 * L_i = query_start[i + 1] - query_start[i] new tokens whose K/V are already in
 * the cache (pa_cache_write) as its last L_i of seq_lens[i] tokens; new token
 * j, at position p = seq_lens[i] - L_i + j, attends causally to tokens [0, p]:
 *   out = softmax(scale * q . K[0..p]^T) . V[0..p]   (fp32 sums, one rounding).
 *   q, out        [total_q][num_q_heads][head_dim], dtype; rows of sequence i
 *                 at [query_start[i], query_start[i + 1]); out must not alias q
 *   query_start   int32 [num_seqs + 1], query_start[0] = 0, non-decreasing,
 *                 query_start[num_seqs] = total_q
 *   workspace     pa_prefill_workspace_size() bytes, zero-filled before its
 *                 first use; every call that runs to its end leaves it zero
 * A sequence with L_i > seq_lens[i] or a length outside its table row sets
 * PA_DEVERR_SEQ_LEN and gets zero rows.  num_seqs <= 4096.  Block sizes of at
 * least 4 (head_dim 128) or 8 (head_dim 64); head_dim 64 or 128; group size
 * at most 16.  Query head hq reads KV head hq / G.
 */
int pa_prefill_workspace_size(size_t* bytes);

/*
 * pa_prefill_kernel -- which kernel pa_prefill runs for this shape on the
 * current device: *kind = PA_PREFILL_TENSOR_CORE (tcgen05.mma with the
 * accumulators in tensor memory; blocks of 8 or more tokens, when its staging
 * fits the device) or PA_PREFILL_WARP_MMA (warp-level m16n8k16 MMAs; the
 * other supported shapes).  Shapes pa_prefill refuses return its error.  The
 * choice is the same as pa_prefill's [P1] "How does it support prompts of
 * arbitrary length?" chunks, at any batch size up to 4096 sequences.
 */
#define PA_PREFILL_WARP_MMA 0
#define PA_PREFILL_TENSOR_CORE 1
int pa_prefill_kernel(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t dtype, int32_t num_seqs, int32_t* kind);
int pa_prefill(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
               const int32_t* query_start, int32_t num_seqs, int64_t total_q,
               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
               int64_t num_blocks, int32_t dtype, float scale, void* out, void* workspace,
               size_t workspace_bytes, int32_t* err_word, pa_stream stream);

/*
 * pa_decode_noalloc -- pa_decode without a caller-provided workspace.
 * The paper has no counterpart to this entry point: it exists for callers that
 * cannot allocate device memory (a runtime whose device memory another
 * allocator already owns, a C program with no device allocator, or a decode
 * loop that cannot afford cudaMalloc's synchronization).  Arguments and result
 * are those of pa_decode.  The workspace is a fixed array of
 * PA_NOALLOC_SCRATCH_BYTES in the library's own device memory, held by every
 * GPU that loads the library until the process exits; this call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).  The
 * first call on a device (and the first after that device's context was reset)
 * looks the array's device address up (cudaGetSymbolAddress) with that device
 * current, so make that first call before any stream capture.  Every call
 * first clears the array's split-context counters on `stream` (one
 * cudaMemsetAsync of 64 KiB), so nothing a previous call left in the array,
 * including one that gave up with PA_DEVERR_TIMEOUT, reaches the next.  A
 * shape whose workspace (pa_decode_workspace_size) exceeds the array returns
 * PA_ERR_WORKSPACE.  All calls share the one array: calls that overlap on the
 * GPU (for instance on two streams) race and must be serialized by the caller.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
int pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
                      int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t dtype,
                      float scale, void* out, int32_t flags, int32_t num_ctas,
                      int32_t* err_word, pa_stream stream);

/*
 * pa_gather_kv -- (test support) gather every sequence's K and V rows into
 * contiguous arrays through the same block-table walk, the same TMA staging
 * into shared memory and the same shared-memory addressing that pa_decode
 * uses (flags: PA_DECODE_SIMT selects the CUDA-core kernel's staging layout,
 * anything else the tensor-core kernel's swizzled layout).
 *   out_offsets  int64 [num_seqs]: first output row of sequence i
 *   k_out, v_out [sum seq_lens][num_kv_heads][head_dim], dtype
 * Bit-exact.
 */
int pa_gather_kv(const void* k_cache, const void* v_cache, const int32_t* block_tables,
                 int32_t table_stride, const int32_t* seq_lens, const int64_t* out_offsets,
                 int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                 int64_t num_blocks, int32_t dtype, int32_t flags, void* k_out, void* v_out,
                 int32_t* err_word, pa_stream stream);

/*
 * pa_get_error -- synchronize `stream`, read *err_word into *flags (if not
 * NULL) and clear it.  Returns PA_ERR_DEVICE_INDEX if any bit was set.
 */
int pa_get_error(int32_t* err_word, pa_stream stream, int32_t* flags);

/* pa_strerror -- a static description of a status code. */
const char* pa_strerror(int status);

/* pa_version -- library version, major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
