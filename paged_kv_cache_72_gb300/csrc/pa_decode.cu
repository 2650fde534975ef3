// Host side of pa_decode / pa_gather_kv: shape checks, the launch plan
// (pipeline depth, shared-memory layout, grid), the TMA tensor maps over the
// KV pools, and the C entry points.
#include <string.h>

#include <cmath>

#include <mutex>

#include "pa_decode_kernel.cuh"
#include "pa_decode_launch.h"

namespace pa {

namespace {

constexpr int kMaxStages = 8;

// mbarriers (16 B per stage, 16 B per query buffer), scan scratch, control
// words, merge row scratch
int ctrl_bytes(int stages) {
  return 16 * stages + 16 * kQBufs + kScanBytes + kCtrlBytes + kLenCacheBytes;
}

// kv_dtype: the pools' element type (PA_F16, PA_BF16 or PA_FP8_E4M3);
// q_dtype: queries and output (PA_F16 or PA_BF16; equal to kv_dtype unless
// the pools are E4M3).
int make_plan(int Hq, int Hkv, int D, int B, int kv_dtype, int q_dtype, int flags, int num_ctas,
              bool gather, DecodePlan* p) {
  if (Hq <= 0 || Hkv <= 0 || num_ctas < 0 || num_ctas > PA_DECODE_MAX_CTAS)
    return PA_ERR_INVALID_ARG;
  if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (kv_dtype != q_dtype && kv_dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  const bool f8 = kv_dtype == PA_FP8_E4M3;
  if (f8 && gather) return PA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(B) || B < 2 || B > 256) return PA_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return PA_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (G > 16) return PA_ERR_UNSUPPORTED;
  flags &= ~PA_DECODE_TABLES_READY;   // a launch option, not part of the plan
  if (flags != PA_DECODE_AUTO && flags != PA_DECODE_SIMT && flags != PA_DECODE_MMA)
    return PA_ERR_INVALID_ARG;
  DecodePlan q{};
  q.bf16 = q_dtype == PA_BF16;
  q.f8 = f8;
  const int eb = f8 ? 1 : 2;   // bytes of one KV element
  q.D = D;
  q.G = G;
  q.B = B;
  bool want_swz;
  if (gather) {
    q.mode = kModeGather;
    want_swz = flags != PA_DECODE_SIMT;
  } else if (flags == PA_DECODE_SIMT || (flags == PA_DECODE_AUTO && G == 1)) {
    if (G != 1) return PA_ERR_UNSUPPORTED;
    q.mode = kModeSimt;
    want_swz = false;
  } else {
    q.mode = kModeMma;
    want_swz = true;
  }
  q.hi = q.mode == kModeMma && G > 8;
  // heads per group: the largest power of two (at most 8) dividing H_kv, with
  // at most 64 query rows per group
  q.HG = (Hkv % 8 == 0) ? 8 : (Hkv % 4 == 0) ? 4 : (Hkv % 2 == 0) ? 2 : 1;
  while (q.HG > 1 && q.HG * G > 64) q.HG /= 2;
  q.NGR = Hkv / q.HG;
  q.TPH = kCWarps / q.HG;
  // tokens per warp per chunk: the E4M3 tensor-core consumer takes 32
  q.CT = ((f8 && q.mode == kModeMma) ? kTileF8 : kTile) * q.TPH;
  q.R = B < q.CT ? B : q.CT;
  q.nsb = q.CT / q.R;
  if (q.nsb > 32) return PA_ERR_UNSUPPORTED;   // one producer lane per TMA box
  const int box_bytes = q.R * q.HG * D * eb;
  // the swizzled TMA layout repeats every 1024 bytes (128-byte swizzle) or
  // 512 bytes (the 64-byte swizzle of 64-byte E4M3 rows); boxes land on
  // multiples of box_bytes
  q.swz = want_swz && (box_bytes % ((f8 && D == 64) ? 512 : 1024) == 0);
  q.split_rows = true;
  q.kv_bytes = q.CT * q.HG * D * eb;
  q.stage_bytes = 2 * q.kv_bytes;
  q.q_bytes = gather ? 0 : q.HG * G * D * 2;
  // rows land q_pitch apart (pa_decode_kernel.cuh)
  q.q_stride = gather ? 0 : ((q.HG * G * (D * 2 + 16) + 127) / 128) * 128;
  const int merge_bytes = (gather || q.TPH == 1) ? 0 : kCWarps * (32 + G * D) * 4;

  DeviceInfo di;
  if (int rc = current_device_info(&di)) return rc;
  const int avail = di.smem_per_block - 1024 - kQBufs * q.q_stride - merge_bytes -
                    ctrl_bytes(kMaxStages);
  int st = avail / q.stage_bytes;
  if (st > kMaxStages) st = kMaxStages;
  if (st < 2) return PA_ERR_UNSUPPORTED;
  q.stages = st;
  q.q_off = q.stages * q.stage_bytes;
  q.merge_off = q.q_off + kQBufs * q.q_stride;
  q.ctrl_off = q.merge_off + merge_bytes;
  q.smem_bytes = 1024 + q.ctrl_off + ctrl_bytes(q.stages);
  q.smem_optin = di.smem_per_block;

  // opts the kernel in to its shared memory and reports its occupancy
  int per_sm = 0;
  const int rc = f8 ? (D == 64 ? decode_ctas_per_sm_f8_d64(q, &per_sm)
                               : decode_ctas_per_sm_f8_d128(q, &per_sm))
                    : (D == 64 ? decode_ctas_per_sm_d64(q, &per_sm)
                               : decode_ctas_per_sm_d128(q, &per_sm));
  if (rc != PA_OK) return rc;
  if (per_sm < 1) return PA_ERR_UNSUPPORTED;
  q.grid = num_ctas > 0 ? num_ctas : di.sm_count * per_sm;
  if (q.grid > PA_DECODE_MAX_CTAS) return PA_ERR_INVALID_ARG;
  // the counters' place must not depend on the grid: a call with a small grid
  // would otherwise leave records where a larger grid expects zero counters
  q.ws_count_bytes = gather ? 0 : (size_t)PA_DECODE_MAX_CTAS * sizeof(uint32_t);
  q.ws_rec_bytes = gather ? 0 : (size_t)q.grid * 2 * rec_floats(q.HG * G, D) * sizeof(float);
  *p = q;
  return PA_OK;
}

// Plans depend only on the shape and the device: keep them, so that a call
// does no attribute or occupancy queries after the first one for its shape.
struct PlanKey {
  int dev, Hq, Hkv, D, B, kv_dtype, q_dtype, flags, num_ctas, gather;
  bool operator==(const PlanKey& o) const {
    return dev == o.dev && Hq == o.Hq && Hkv == o.Hkv && D == o.D && B == o.B &&
           kv_dtype == o.kv_dtype && q_dtype == o.q_dtype && flags == o.flags &&
           num_ctas == o.num_ctas && gather == o.gather;
  }
};
constexpr int kPlanCache = 64;
PlanKey g_plan_key[kPlanCache];
DecodePlan g_plan[kPlanCache];
int g_plan_n = 0, g_plan_next = 0;
std::mutex g_plan_mu;

int cached_plan(int Hq, int Hkv, int D, int B, int kv_dtype, int q_dtype, int flags,
                int num_ctas, bool gather, DecodePlan* p) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    // still report shape errors without a device
    return make_plan(Hq, Hkv, D, B, kv_dtype, q_dtype, flags, num_ctas, gather, p);
  }
  const PlanKey k{dev, Hq, Hkv, D, B, kv_dtype, q_dtype, flags, num_ctas, gather ? 1 : 0};
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    for (int i = 0; i < g_plan_n; ++i)
      if (g_plan_key[i] == k) {
        *p = g_plan[i];
        return PA_OK;
      }
  }
  if (int rc = make_plan(Hq, Hkv, D, B, kv_dtype, q_dtype, flags, num_ctas, gather, p)) return rc;
  std::lock_guard<std::mutex> lk(g_plan_mu);
  const int slot = g_plan_n < kPlanCache ? g_plan_n++ : (g_plan_next++ % kPlanCache);
  g_plan_key[slot] = k;
  g_plan[slot] = *p;
  return PA_OK;
}

// TMA map over one pool [num_blocks][B][Hkv][D]: one box = R rows of HG
// heads of one block, all D elements.  With split_rows the box lands as
// [HG][D/64][R][64] (dims: d_lo, row, d_hi, head, block), so that eight
// consecutive rows of one head sit in eight consecutive 128-byte lines;
// otherwise as [R][HG][D/64][64] (dims: d_lo, d_hi, head, row, block).
int encode_kv_map(CUtensorMap* map, const void* cache, const DecodePlan& p, int Hkv,
                  long long num_blocks, bool split_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return PA_ERR_CUDA;
  const int D = p.D, B = p.B;
  cuuint64_t dims[5];
  cuuint64_t strides[4];
  cuuint32_t box[5];
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  if (p.f8) {
    // E4M3 rows of D bytes, one plane: the box lands as [HG][R][D] bytes
    const cuuint64_t row8 = (cuuint64_t)Hkv * D;
    dims[0] = D; dims[1] = B; dims[2] = 1; dims[3] = Hkv; dims[4] = num_blocks;
    strides[0] = row8; strides[1] = D; strides[2] = D; strides[3] = row8 * B;
    box[0] = D; box[1] = p.R; box[2] = 1; box[3] = p.HG; box[4] = 1;
    memset(map, 0, sizeof(*map));
    const CUtensorMapSwizzle sw = !p.swz ? CU_TENSOR_MAP_SWIZZLE_NONE
                                         : (D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                     : CU_TENSOR_MAP_SWIZZLE_64B);
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(cache), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) return PA_OK;
    note_cuda_error(1000 + (int)r, "cuTensorMapEncodeTiled (E4M3 pool)");
    return PA_ERR_CUDA;
  }
  const cuuint64_t row = (cuuint64_t)Hkv * D * 2;
  if (split_rows) {
    dims[0] = 64; dims[1] = B; dims[2] = D / 64; dims[3] = Hkv; dims[4] = num_blocks;
    strides[0] = row; strides[1] = 128; strides[2] = (cuuint64_t)D * 2; strides[3] = row * B;
    box[0] = 64; box[1] = p.R; box[2] = D / 64; box[3] = p.HG; box[4] = 1;
  } else {
    dims[0] = 64; dims[1] = D / 64; dims[2] = Hkv; dims[3] = B; dims[4] = num_blocks;
    strides[0] = 128; strides[1] = (cuuint64_t)D * 2; strides[2] = row; strides[3] = row * B;
    box[0] = 64; box[1] = D / 64; box[2] = p.HG; box[3] = p.R; box[4] = 1;
  }
  memset(map, 0, sizeof(*map));
  CUresult r =
      enc(map, p.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
          const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          p.swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) return PA_OK;
  note_cuda_error(1000 + (int)r, "cuTensorMapEncodeTiled");
  return PA_ERR_CUDA;
}

int encode_maps_uncached(CUtensorMap* tk, CUtensorMap* tv, const void* kc, const void* vc,
                         DecodePlan* p, int Hkv, long long nb) {
  if (p->f8) {
    if (int rc = encode_kv_map(tk, kc, *p, Hkv, nb, true)) return rc;
    return encode_kv_map(tv, vc, *p, Hkv, nb, true);
  }
  if (p->split_rows) {
    if (encode_kv_map(tk, kc, *p, Hkv, nb, true) == PA_OK &&
        encode_kv_map(tv, vc, *p, Hkv, nb, true) == PA_OK)
      return PA_OK;
    p->split_rows = false;  // the driver refused the plane layout: rows stay contiguous
  }
  if (int rc = encode_kv_map(tk, kc, *p, Hkv, nb, false)) return rc;
  return encode_kv_map(tv, vc, *p, Hkv, nb, false);
}

// Tensor maps depend on the pools' addresses and shape: keep the recent ones.
struct alignas(64) MapEntry {
  CUtensorMap tk, tv;
  const void* kc;
  const void* vc;
  long long nb;
  int dev, Hkv, D, B, bf16, f8, swz, split_in, split_out;
};
constexpr int kMapCache = 16;
MapEntry g_maps[kMapCache];
int g_maps_n = 0, g_maps_next = 0;
std::mutex g_maps_mu;

int encode_maps(CUtensorMap* tk, CUtensorMap* tv, const void* kc, const void* vc, DecodePlan* p,
                int Hkv, long long nb) {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return launch_status(e, "cudaGetDevice");
  const int split_in = p->split_rows ? 1 : 0;
  {
    std::lock_guard<std::mutex> lk(g_maps_mu);
    for (int i = 0; i < g_maps_n; ++i) {
      const MapEntry& m = g_maps[i];
      if (m.kc == kc && m.vc == vc && m.nb == nb && m.dev == dev && m.Hkv == Hkv && m.D == p->D &&
          m.B == p->B && m.bf16 == (p->bf16 ? 1 : 0) && m.f8 == (p->f8 ? 1 : 0) &&
          m.swz == (p->swz ? 1 : 0) &&
          m.split_in == split_in) {
        *tk = m.tk;
        *tv = m.tv;
        p->split_rows = m.split_out != 0;
        return PA_OK;
      }
    }
  }
  if (int rc = encode_maps_uncached(tk, tv, kc, vc, p, Hkv, nb)) return rc;
  std::lock_guard<std::mutex> lk(g_maps_mu);
  const int slot = g_maps_n < kMapCache ? g_maps_n++ : (g_maps_next++ % kMapCache);
  MapEntry& m = g_maps[slot];
  m.tk = *tk;
  m.tv = *tv;
  m.kc = kc;
  m.vc = vc;
  m.nb = nb;
  m.dev = dev;
  m.Hkv = Hkv;
  m.D = p->D;
  m.B = p->B;
  m.bf16 = p->bf16 ? 1 : 0;
  m.f8 = p->f8 ? 1 : 0;
  m.swz = p->swz ? 1 : 0;
  m.split_in = split_in;
  m.split_out = p->split_rows ? 1 : 0;
  return PA_OK;
}

void fill_layout(const DecodePlan& p, DecodeArgs* a) {
  a->G = p.G;
  a->B = p.B;
  a->log2B = ilog2(p.B);
  a->HG = p.HG;
  a->NGR = a->Hkv / p.HG;
  a->TPH = p.TPH;
  a->CT = p.CT;
  a->R = p.R;
  a->log2R = ilog2(p.R);
  a->nsb = p.nsb;
  a->stages = p.stages;
  a->kv_bytes = p.kv_bytes;
  a->stage_bytes = p.stage_bytes;
  a->q_off = p.q_off;
  a->q_bytes = p.q_bytes;
  a->q_stride = p.q_stride;
  a->merge_off = p.merge_off;
  a->ctrl_off = p.ctrl_off;
  a->split_rows = p.split_rows ? 1 : 0;
  const int lrow = ilog2((long long)p.D * (p.f8 ? 1 : 2));   // one row of one head
  a->sub_log2 = a->log2R + ilog2(p.HG) + lrow;               // one box
  if (p.f8) {   // [HG][R][D] bytes
    a->head_log2 = a->log2R + lrow;
    a->hi_log2 = 0;
    a->r_log2 = lrow;
  } else if (p.split_rows) {
    a->head_log2 = a->log2R + lrow;
    a->hi_log2 = a->log2R + 7;
    a->r_log2 = 7;
  } else {
    a->head_log2 = lrow;
    a->hi_log2 = 7;
    a->r_log2 = ilog2(p.HG) + lrow;
  }
}

int launch(const DecodePlan& p, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
           cudaStream_t s) {
  if (p.f8)
    return p.D == 64 ? decode_launch_f8_d64(p, tk, tv, a, s) : decode_launch_f8_d128(p, tk, tv, a, s);
  return p.D == 64 ? decode_launch_d64(p, tk, tv, a, s) : decode_launch_d128(p, tk, tv, a, s);
}

// The decode behind pa_decode and pa_decode_fp8.
int decode_call(const void* q, const void* k_cache, const void* v_cache,
                const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
                int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                int32_t block_size, int64_t num_blocks, int32_t kv_dtype, int32_t q_dtype,
                float scale, float k_scale, float v_scale, int32_t window, void* out,
                void* workspace, size_t workspace_bytes, int32_t flags, int32_t num_ctas,
                int32_t* err_word, pa_stream stream) {
  if (num_seqs < 0 || table_stride < 0 || num_blocks < 0 || window < 0) return PA_ERR_INVALID_ARG;
  DecodePlan p;
  const int early = (flags & PA_DECODE_TABLES_READY) ? 1 : 0;
  flags &= ~PA_DECODE_TABLES_READY;
  if (int rc = cached_plan(num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype, q_dtype,
                           flags, num_ctas, false, &p))
    return rc;
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out || !workspace)
    return PA_ERR_INVALID_ARG;
  if (num_blocks == 0 || table_stride == 0 || num_blocks > 0xffffffffLL) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace))
    return PA_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return PA_ERR_INVALID_ARG;
  if (workspace_bytes < p.ws_count_bytes + p.ws_rec_bytes) return PA_ERR_WORKSPACE;
  CUtensorMap tk, tv;
  if (int rc = encode_maps(&tk, &tv, k_cache, v_cache, &p, num_kv_heads, num_blocks)) return rc;
  DecodeArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.bt = block_tables;
  a.seq_lens = seq_lens;
  a.ws_count = static_cast<uint32_t*>(workspace);
  a.ws_rec = reinterpret_cast<float*>(static_cast<char*>(workspace) + p.ws_count_bytes);
  a.err = err_word;
  a.num_blocks = num_blocks;
  a.num_seqs = num_seqs;
  a.stride = table_stride;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.scale_log2 = scale * k_scale * 1.4426950408889634f;
  a.v_scale = v_scale;
  a.window = window;
  a.early_tables = early;
  fill_layout(p, &a);
  return launch(p, tk, tv, a, static_cast<cudaStream_t>(stream));
}

}  // namespace

// A TMA map over one 16-bit pool for other kernels of the library: boxes of
// p.R rows of p.HG heads of one block, split-row layout, swizzled if p.swz.
int encode_pool_map(CUtensorMap* map, const void* cache, const DecodePlan& p, int Hkv,
                    long long num_blocks) {
  return encode_kv_map(map, cache, p, Hkv, num_blocks, true);
}

// One 64-column plane of R rows of one head of one block, 128-byte swizzled:
// copies of the two planes of a box land apart, so that a stage part holds
// [plane][row][128 bytes] (the K-major and MN-major operand layouts of the
// tensor-core prefill).
int encode_pool_plane_map(CUtensorMap* map, const void* cache, bool bf16, int D, int B, int R,
                          int Hkv, long long num_blocks, int box_planes) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return PA_ERR_CUDA;
  const cuuint64_t row = (cuuint64_t)Hkv * D * 2;
  const cuuint64_t dims[5] = {64, (cuuint64_t)B, (cuuint64_t)(D / 64), (cuuint64_t)Hkv,
                              (cuuint64_t)num_blocks};
  const cuuint64_t strides[4] = {row, 128, (cuuint64_t)D * 2, row * B};
  // box_planes 64-column planes of R rows of one head of one block: in shared
  // memory [plane][row][128 bytes]
  if (box_planes < 1 || box_planes > D / 64) return PA_ERR_INVALID_ARG;
  const cuuint32_t box[5] = {64, (cuuint32_t)R, (cuuint32_t)box_planes, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  memset(map, 0, sizeof(*map));
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   5, const_cast<void*>(cache), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) return PA_OK;
  note_cuda_error(1000 + (int)r, "cuTensorMapEncodeTiled (pool plane)");
  return PA_ERR_CUDA;
}

// The query rows of one work item: BM tokens x the G heads of one KV head, one
// 64-column plane per copy, landing as [token][head][128 bytes] with a
// 128-byte swizzle.  Rows past total_q read as zeros.
int encode_q_tile_map(CUtensorMap* map, const void* q, bool bf16, int D, int G, int Hkv,
                      long long total_q, int BM) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return PA_ERR_CUDA;
  const cuuint64_t dims[5] = {64, (cuuint64_t)(D / 64), (cuuint64_t)G, (cuuint64_t)Hkv,
                              (cuuint64_t)total_q};
  const cuuint64_t strides[4] = {128, (cuuint64_t)D * 2, (cuuint64_t)G * D * 2,
                                 (cuuint64_t)Hkv * G * D * 2};
  const cuuint32_t box[5] = {64, 1, (cuuint32_t)G, 1, (cuuint32_t)BM};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  memset(map, 0, sizeof(*map));
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   5, const_cast<void*>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) return PA_OK;
  note_cuda_error(1000 + (int)r, "cuTensorMapEncodeTiled (query tile)");
  return PA_ERR_CUDA;
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_decode_workspace_size(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t dtype, int32_t flags, int32_t num_ctas,
                             size_t* bytes) {
  if (!bytes) return PA_ERR_INVALID_ARG;
  flags &= ~PA_DECODE_TABLES_READY;   // the workspace does not depend on it
  // an E4M3 cache: the workspace does not depend on the query dtype
  const int q_dtype = dtype == PA_FP8_E4M3 ? PA_BF16 : dtype;
  DecodePlan p;
  if (int rc = cached_plan(num_q_heads, num_kv_heads, head_dim, block_size, dtype, q_dtype, flags,
                           num_ctas, false, &p))
    return rc;
  *bytes = p.ws_count_bytes + p.ws_rec_bytes;
  return PA_OK;
}

int pa_decode(const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
              int32_t block_size, int64_t num_blocks, int32_t dtype, float scale, void* out,
              void* workspace, size_t workspace_bytes, int32_t flags, int32_t num_ctas,
              int32_t* err_word, pa_stream stream) {
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  return decode_call(q, k_cache, v_cache, block_tables, table_stride, seq_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, dtype, dtype,
                     scale, 1.f, 1.f, 0, out, workspace, workspace_bytes, flags, num_ctas,
                     err_word, stream);
}

int pa_decode_window(const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
                     int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t block_size, int64_t num_blocks, int32_t dtype,
                     float scale, int32_t window, void* out, void* workspace,
                     size_t workspace_bytes, int32_t flags, int32_t num_ctas, int32_t* err_word,
                     pa_stream stream) {
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (window <= 0) return PA_ERR_INVALID_ARG;
  return decode_call(q, k_cache, v_cache, block_tables, table_stride, seq_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, dtype, dtype,
                     scale, 1.f, 1.f, window, out, workspace, workspace_bytes, flags, num_ctas,
                     err_word, stream);
}

int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t block_size, int64_t num_blocks, int32_t q_dtype, float scale,
                  float k_scale, float v_scale, void* out, void* workspace,
                  size_t workspace_bytes, int32_t flags, int32_t num_ctas, int32_t* err_word,
                  pa_stream stream) {
  return decode_call(q, k_cache, v_cache, block_tables, table_stride, seq_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, PA_FP8_E4M3,
                     q_dtype, scale, k_scale, v_scale, 0, out, workspace, workspace_bytes, flags,
                     num_ctas, err_word, stream);
}

int pa_gather_kv(const void* k_cache, const void* v_cache, const int32_t* block_tables,
                 int32_t table_stride, const int32_t* seq_lens, const int64_t* out_offsets,
                 int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                 int64_t num_blocks, int32_t dtype, int32_t flags, void* k_out, void* v_out,
                 int32_t* err_word, pa_stream stream) {
  if (num_seqs < 0 || table_stride < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  DecodePlan p;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (int rc = cached_plan(num_kv_heads, num_kv_heads, head_dim, block_size, dtype, dtype, flags, 0,
                           true, &p))
    return rc;
  if (num_seqs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_tables || !seq_lens || !out_offsets || !k_out || !v_out)
    return PA_ERR_INVALID_ARG;
  if (num_blocks == 0 || table_stride == 0 || num_blocks > 0xffffffffLL) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_out) || !aligned16(v_out))
    return PA_ERR_INVALID_ARG;
  CUtensorMap tk, tv;
  if (int rc = encode_maps(&tk, &tv, k_cache, v_cache, &p, num_kv_heads, num_blocks)) return rc;
  DecodeArgs a{};
  a.bt = block_tables;
  a.seq_lens = seq_lens;
  a.err = err_word;
  a.out_off = out_offsets;
  a.k_out = static_cast<uint16_t*>(k_out);
  a.v_out = static_cast<uint16_t*>(v_out);
  a.num_blocks = num_blocks;
  a.num_seqs = num_seqs;
  a.stride = table_stride;
  a.Hq = num_kv_heads;
  a.Hkv = num_kv_heads;
  fill_layout(p, &a);
  a.G = 1;
  return launch(p, tk, tv, a, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
