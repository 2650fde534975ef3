// Launch plan of the decode / gather kernels, shared between the planner and
// the per-head_dim translation units that instantiate the kernels.
#pragma once

#include "pa_host.h"

namespace pa {

struct DecodeArgs;

struct DecodePlan {
  int mode;          // kModeSimt, kModeMma, kModeGather
  bool bf16;         // queries and output in bfloat16 (else binary16)
  bool f8;           // the KV pools hold E4M3 codes (else the query dtype)
  bool swz;          // 128-byte swizzled staging (tensor-core reads)
  bool hi;           // group size > 8: query heads fill both MMA row halves
  bool split_rows;   // rows of a box stored as two [R][64] planes
  int D, G, B, R, nsb;
  int HG, NGR, TPH, CT;   // heads per group, groups, tiles per head, tokens per chunk
  int stages;
  int kv_bytes, stage_bytes, q_off, q_bytes, q_stride, merge_off, ctrl_off, smem_bytes;
  int smem_optin;    // the device's per-block shared-memory maximum
  int grid;
  size_t ws_count_bytes, ws_rec_bytes;   // workspace: per-CTA piece counters, then records
};

// TMA map over one 16-bit pool (split-row layout) for other kernels.
int encode_pool_map(CUtensorMap* map, const void* cache, const DecodePlan& p, int Hkv,
                    long long num_blocks);
// Per-plane pool map and query-tile map of the tensor-core prefill.
int encode_pool_plane_map(CUtensorMap* map, const void* cache, bool bf16, int D, int B, int R,
                          int Hkv, long long num_blocks, int box_planes);
int encode_q_tile_map(CUtensorMap* map, const void* q, bool bf16, int D, int G, int Hkv,
                      long long total_q, int BM);

// Per-variant occupancy (CTAs per SM) for a given dynamic shared-memory size.
int decode_ctas_per_sm(const DecodePlan& p, int* ctas);

// Launches the decode (or gather) kernel.
int decode_launch(const DecodePlan& p, const CUtensorMap& tk, const CUtensorMap& tv,
                  const DecodeArgs& a, cudaStream_t s);

int decode_ctas_per_sm_d64(const DecodePlan& p, int* ctas);
int decode_ctas_per_sm_d128(const DecodePlan& p, int* ctas);
int decode_launch_d64(const DecodePlan& p, const CUtensorMap& tk, const CUtensorMap& tv,
                      const DecodeArgs& a, cudaStream_t s);
int decode_launch_d128(const DecodePlan& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       const DecodeArgs& a, cudaStream_t s);
int decode_ctas_per_sm_f8_d64(const DecodePlan& p, int* ctas);
int decode_ctas_per_sm_f8_d128(const DecodePlan& p, int* ctas);
int decode_launch_f8_d64(const DecodePlan& p, const CUtensorMap& tk, const CUtensorMap& tv,
                         const DecodeArgs& a, cudaStream_t s);
int decode_launch_f8_d128(const DecodePlan& p, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeArgs& a, cudaStream_t s);

}  // namespace pa
