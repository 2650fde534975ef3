// Paged single-query decode attention for sm_103a.
//
// What it computes ("vLLM Framework and Inference Engine Design", section
// "What is the essence of vLLM's PagedAttention?"): for every sequence i and
// query head hq, softmax(scale * q . K^T) . V over the first seq_lens[i] tokens,
// where token t lives in physical block block_table[i][t / B], row t % B, of a
// per-layer pool [num_blocks][B][H_kv][D].  Query head hq reads KV head hq / G.
//
// Design (one GPU, persistent, HBM-bound):
//  * KV heads are taken in groups of HG (the largest of 8, 4, 2, 1 that divides
//    H_kv).  A pipeline stage holds CT = 128 / HG tokens of every head of one
//    group, so that one TMA box carries R = min(B, CT) rows of all HG heads of
//    one physical block: for 16-token blocks and 8 KV heads that is one 32 KB
//    box per block for K and one for V.
//  * The work is the list of chunks (sequence, head group, CT tokens), cut into
//    equal contiguous ranges, one per CTA (grid = the SM count).  Every CTA
//    scans seq_lens once to find its range; a context may be split across
//    CTAs.  Each piece leaves its partial softmax state (m, l, o) in the
//    workspace and counts itself on the context's counter; the piece that
//    completes the count merges them, so no CTA ever waits for another.  The
//    split depends only on seq_lens, so the result does not depend on where the
//    blocks sit.
//  * One producer warp reads the block table one chunk ahead and streams each
//    chunk's K and V boxes with 5-D TMA tensor copies into a ring of shared-
//    memory stages guarded by mbarriers.  When a new (sequence, head group)
//    segment starts it first fetches the group's HG * G query rows with a 1-D
//    bulk copy into a small ring of query buffers.  Each K/V byte is read once
//    and shared by the G query heads of its KV head.
//  * Eight consumer warps: warp w takes 16 tokens (tile w % TPH, TPH = 8 / HG)
//    of head w / TPH of every chunk and keeps its own online-softmax state in
//    fp32.  The tensor-core consumers use m16n8k16 MMAs; for groups of up to
//    8 query heads they compute the transposed products S^T = K.Q^T and
//    O^T += V^T.P^T (tokens / head_dim on M, the heads on N), for larger
//    groups S = Q.K^T and O += P.V (heads on M); P enters as a pair of 16-bit
//    values whose sum carries it to 16 bits.  The CUDA-core consumer (group
//    size 1) uses per-lane head_dim slices and warp shuffles.
//    When a warp owns its head alone (HG = 8) it writes its result directly;
//    otherwise the TPH warps of a head merge through shared memory.
//  * Every wait is bounded; a wait that gives up sets PA_DEVERR_TIMEOUT and the
//    CTA runs to its end without touching the pipeline again.
#pragma once

#include <type_traits>

#include "pa_device.cuh"

namespace pa {

constexpr int kTile = 16;          // tokens per consumer warp per stage
constexpr int kCWarps = 8;         // consumer warps; stage = kCWarps * 16 token-heads
constexpr int kProducerWarp = kCWarps;
enum Mode : int { kModeSimt = 0, kModeMma = 1, kModeGather = 2 };

// A block of nine warps has three on one SM sub-partition, which leaves
// every thread at most 168 registers.  The 16-bit tensor-core consumer for
// groups of more than 8 query heads needs more: its blocks put the producer
// in a warpgroup of its own (three more warps that leave at once), and the
// two warpgroups re-divide the registers the block is launched with
// (setmaxnreg): the producer's group keeps kProducerRegs per thread, the
// consumers take kConsumerRegs.  The other consumers (the transposed one for
// groups of up to 8 among them) fit in 168 and run as nine-warp blocks.
constexpr int kLaunchRegs = 168;     // 65536 / 384, rounded down to a multiple of 8
constexpr int kProducerRegs = 56;
constexpr int kConsumerRegs = 224;
static_assert(kCWarps * 32 * kConsumerRegs + 128 * kProducerRegs <= (kCWarps + 4) * 32 * kLaunchRegs,
              "the register split must fit in what the block is launched with");
__host__ __device__ constexpr bool split_regs(int mode, bool f8, bool hi) {
  return mode == kModeMma && !f8 && hi;
}
__host__ __device__ constexpr int block_threads(int mode, bool f8, bool hi) {
  return (kCWarps + (split_regs(mode, f8, hi) ? 4 : 1)) * 32;
}
constexpr int kQBufs = 2;          // query-row buffers in flight
// Query rows sit in shared memory at a pitch of one row plus 16 bytes, so
// that the fragment loads of rows a full row apart fall in different banks.
template <int D>
__host__ __device__ constexpr int q_pitch() { return D * 2 + 16; }
// Lengths of the first kLenCache sequences, kept in shared memory by the scan
// for the walks of the producer and the consumers.
constexpr int kLenCache = 1024;
// Shared-memory control area after the mbarriers: scan scratch, control words
// (walk start, abort flag, merges this CTA owes), the lengths cache.
constexpr int kScanBytes = 128;
constexpr int kCtrlBytes = 64;
constexpr int kLenCacheBytes = 4 * kLenCache;
constexpr int kCtrlMerges = 5;     // ctrl[5] = pending merges, then 4 ints per merge
constexpr int kCtrlEmpty = 14;     // this CTA owns empty or invalid sequences (early tables)
// counter bit set by a piece whose CTA gave up: the context is left unmerged
constexpr uint32_t kPieceAborted = 0x80000000u;


struct DecodeArgs {
  const uint16_t* q;         // [N][Hq][D]
  uint16_t* out;             // [N][Hq][D]
  const int32_t* bt;         // [N][stride]
  const int32_t* seq_lens;   // [N]
  float* ws_rec;             // [grid][2] records of rec_floats(HG*G, D): o[][D], m[], l[]
  uint32_t* ws_count;        // [PA_DECODE_MAX_CTAS]: pieces of the split context ending in
                             // CTA k that have arrived; zero between calls (the last
                             // arriver resets it)
  int32_t* err;
  const int64_t* out_off;    // gather: first output row of each sequence
  uint16_t* k_out;           // gather outputs [rows][H_kv][D]
  uint16_t* v_out;
  long long num_blocks;
  int num_seqs, stride, Hq, Hkv, G, B, log2B;
  int HG, NGR, TPH, CT, R, log2R, nsb;   // heads per group, groups, tiles per head, tokens per chunk
  int stages;
  float scale_log2;          // scale * log2(e)
  int split_rows;            // box layout: 1 = [HG][D/64][R][64], 0 = [R][HG][D/64][64]
  int sub_log2, head_log2, hi_log2, r_log2;   // byte strides inside a stage part (log2)
  int kv_bytes;              // bytes of one K (or V) stage part: CT * HG * D * 2
  int stage_bytes;           // K part + V part (multiple of 1024)
  int q_off, q_bytes;        // query ring offset and one buffer's bytes (HG * G * D * 2)
  int q_stride;              // bytes between query buffers (multiple of 128)
  int merge_off;             // byte offset of the merge buffer (TPH > 1)
  int ctrl_off;              // byte offset of barriers and control words
  float v_scale;             // E4M3 cache: V value = code * v_scale (1 otherwise)
  int window;                // sliding window: attend to the last `window` tokens (0: all)
  int early_tables;          // seq_lens and block tables are complete before the preceding
                             // kernel starts: read them before waiting for it
};

// Clamped length: invalid lengths count as 0 tokens.
__device__ __forceinline__ int clamp_len(int T, int stride, int B) {
  return (T < 0 || (long long)T > (long long)stride * B) ? 0 : T;
}

// Attended tokens of a sequence of length T: [s0, T), s0 = max(0, T - window)
// with a sliding window ("vLLM Framework and Inference Engine Design", section
// "How does it support prompts of arbitrary length? Does it have a sliding
// window?": each token attends only to the last W tokens), else 0.  Chunks
// start at t0 = s0 rounded down to a multiple of R (so that every TMA box
// stays inside one block); the first lo = s0 - t0 < R tokens of chunk 0 are
// masked.  Table entries of blocks wholly before t0 are never read.
__device__ __forceinline__ int attend_origin(int T, const DecodeArgs& a) {
  const int s0 = (a.window > 0 && T > a.window) ? T - a.window : 0;
  return (s0 >> a.log2R) << a.log2R;
}

__device__ __forceinline__ int seq_chunks(int T, const DecodeArgs& a) {
  return (T - attend_origin(T, a) + a.CT - 1) / a.CT;
}

struct Walk {
  int i, g, c, nc, T;   // sequence, head group, chunk, chunks of the sequence, its length
  int t0, lo;           // first token of chunk 0, leading tokens of chunk 0 outside the window
};

// s_len: the clamped lengths of sequences [0, kLenCache) in shared memory
__device__ __forceinline__ void walk_load_seq(Walk& w, const DecodeArgs& a, const int* s_len) {
  w.T = w.i < kLenCache ? s_len[w.i] : clamp_len(__ldg(a.seq_lens + w.i), a.stride, a.B);
  w.t0 = attend_origin(w.T, a);
  w.lo = (a.window > 0 && w.T > a.window) ? w.T - a.window - w.t0 : 0;
  w.nc = (w.T - w.t0 + a.CT - 1) / a.CT;
}

__device__ __forceinline__ void walk_advance(Walk& w, const DecodeArgs& a, const int* s_len) {
  if (++w.c < w.nc) return;
  w.c = 0;
  if (++w.g < a.NGR) return;
  w.g = 0;
  do {
    ++w.i;
    if (w.i >= a.num_seqs) { w.nc = 0; w.T = 0; return; }
    walk_load_seq(w, a, s_len);
  } while (w.nc == 0);
}

// Block-wide inclusive scan of one value per thread (kThreads threads).
template <int kThreads>
__device__ __forceinline__ long long block_scan_incl(long long v, long long* warp_tot,
                                                     long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  long long off = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    long long t = warp_tot[w];
    if (w < warp) off += t;
    total += t;
  }
  __syncthreads();
  return v + off;
}

// Address of token row `tt` (0..CT-1 within the chunk), half `hi` of head
// part `hpart` (the stage part plus the head's offset).
__device__ __forceinline__ uint32_t row_addr(uint32_t hpart, int tt, int hi, const DecodeArgs& a) {
  const int sub = tt >> a.log2R;
  const int r = tt & ((1 << a.log2R) - 1);
  return hpart + ((uint32_t)sub << a.sub_log2) + ((uint32_t)hi << a.hi_log2) +
         ((uint32_t)r << a.r_log2);
}

template <bool kSwz>
__device__ __forceinline__ uint32_t chunk_addr(uint32_t row, int j) {
  // 128-byte swizzle: the 16-byte chunk index is XOR-ed with address bits 7..9
  const int s = kSwz ? (int)((row >> 7) & 7) : 0;
  return row + ((uint32_t)(j ^ s) << 4);
}

// A partial-state record of `rows` query rows: o[rows][D], then m[rows] and
// l[rows], padded so that every record (and every o row) starts on 16 bytes.
__host__ __device__ __forceinline__ size_t rec_floats(int rows, int D) {
  return (size_t)rows * D + (size_t)((2 * rows + 3) & ~3);
}

// ---------------------------------------------------------------------------
// Consumer state and tile math: tensor-core path
// ---------------------------------------------------------------------------
template <int D, bool kBF16, bool kSwz, bool kHi>
struct MmaConsumer {
  static constexpr int KS = D / 16;   // k-steps of QK
  static constexpr int NT = D / 8;    // n-tiles of PV
  static constexpr int QP = q_pitch<D>();
  uint32_t qa[KS][4];
  float o[NT][4];
  float m[2], l[2];

  // qslot: this head's G query rows, QP bytes apart
  __device__ __forceinline__ void begin(uint32_t qslot, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d0 = ks * 16 + 2 * tig;
      uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
      if (gid < G) {
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a0) : "r"(qslot + gid * QP + d0 * 2));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a2) : "r"(qslot + gid * QP + (d0 + 8) * 2));
      }
      if (kHi && gid + 8 < G) {
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a1) : "r"(qslot + (gid + 8) * QP + d0 * 2));
        asm volatile("ld.shared.b32 %0, [%1];"
                     : "=r"(a3)
                     : "r"(qslot + (gid + 8) * QP + (d0 + 8) * 2));
      }
      qa[ks][0] = a0;
      qa[ks][1] = a1;
      qa[ks][2] = a2;
      qa[ks][3] = a3;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }

  // 16 tokens [tile0, tile0 + 16) of the chunk for this warp's head; tokens
  // [lo, nv) of them are valid (rows before a sliding window or past the
  // sequence's end may hold anything, NaN included: their scores are masked
  // and their V values zeroed in registers).
  __device__ __forceinline__ void tile(uint32_t kpart, uint32_t vpart, int tile0, int lo, int nv,
                                       const DecodeArgs& a, float sl2) {
    const int lane = threadIdx.x & 31, tig = lane & 3;
    // S = Q . K^T : two n-tiles of 8 tokens.  All K fragments are loaded
    // first, then the MMAs run as four independent accumulation chains (two
    // n-tiles x even / odd k-steps), so no MMA waits on a fragment load.
    uint32_t kb[2][D / 32][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int tt = tile0 + nt * 8 + (lane & 7);
#pragma unroll
      for (int kp = 0; kp < D / 32; ++kp) {
        const int cidx = kp * 4 + (lane >> 3);
        const uint32_t ra = row_addr(kpart, tt, cidx >> 3, a);
        ldmatrix_x4(chunk_addr<kSwz>(ra, cidx & 7), kb[nt][kp][0], kb[nt][kp][1], kb[nt][kp][2],
                    kb[nt][kp][3]);
      }
    }
    float s[2][4], s2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = s2[nt][e] = 0.f;
#pragma unroll
    for (int kp = 0; kp < D / 32; ++kp)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        mma_16816<kBF16>(s[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3],
                         kb[nt][kp][0], kb[nt][kp][1]);
        mma_16816<kBF16>(s2[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2],
                         qa[2 * kp + 1][3], kb[nt][kp][2], kb[nt][kp][3]);
      }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
    // V fragments, loaded before the softmax math so that their latency hides
    // behind it
    uint32_t vb[D / 16][4];
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      const int mat = lane >> 3;
      const int tt = tile0 + ((mat & 1) << 3) + (lane & 7);
      const int cidx = 2 * j + (mat >> 1);
      const uint32_t ra = row_addr(vpart, tt, cidx >> 3, a);
      ldmatrix_x4_trans(chunk_addr<kSwz>(ra, cidx & 7), vb[j][0], vb[j][1], vb[j][2], vb[j][3]);
    }
    // online softmax, in the log2 domain, per query-head row.  P goes to the
    // P . V products as a pair of 16-bit values, hi = round(P) and
    // lo = round(P - hi) (P - hi is exact in fp32), so that hi + lo is within
    // 2^-16 (bfloat16) or 2^-22 (binary16) of P; the normaliser l sums the
    // fp32 values.  One 16-bit P would move the output by up to the unit
    // roundoff times the values' spread, many ulps of a small output; the
    // second product costs about 1% of the decode, whose consumers have slack.
    uint32_t pa[4], pl[4];
#pragma unroll
    for (int hr = 0; hr < (kHi ? 2 : 1); ++hr) {
      float v[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = nt * 8 + 2 * tig + e;
          const float x = s[nt][hr * 2 + e] * sl2;
          v[nt * 2 + e] = (t >= lo && t < nv) ? x : -INFINITY;
        }
      float mt = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      const float mn = fmaxf(m[hr], mt);
      const float alpha = exp2f(m[hr] - mn);
      m[hr] = mn;
      const float e0 = exp2f(v[0] - mn), e1 = exp2f(v[1] - mn);
      const float e2 = exp2f(v[2] - mn), e3 = exp2f(v[3] - mn);
      const uint32_t p01 = pack2<kBF16>(e0, e1);
      const uint32_t p23 = pack2<kBF16>(e2, e3);
      const float2 f01 = unpack2<kBF16>(p01), f23 = unpack2<kBF16>(p23);
      pl[hr] = pack2<kBF16>(e0 - f01.x, e1 - f01.y);
      pl[hr + 2] = pack2<kBF16>(e2 - f23.x, e3 - f23.y);
      l[hr] = l[hr] * alpha + ((e0 + e1) + (e2 + e3));
      // once the running maximum settles, alpha is exactly 1 in every lane
      // and the rescale is skipped (multiplying by 1 changes nothing)
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][hr * 2 + 0] *= alpha;
          o[n][hr * 2 + 1] *= alpha;
        }
      }
      pa[hr] = p01;       // row gid (+8): tokens 2tig, 2tig+1
      pa[hr + 2] = p23;   // tokens 8 + 2tig, 9 + 2tig
    }
    if (!kHi) { pa[1] = 0u; pa[3] = 0u; pl[1] = 0u; pl[3] = 0u; }
    if (nv < kTile || lo > 0) {
      // zero the V values of tokens outside [lo, nv) (the low 16 bits of a
      // fragment register hold token 2tig (+8), the high bits token 2tig+1)
      auto in = [&](int t) { return t >= lo && t < nv; };
      const uint32_t mlo = (in(2 * tig) ? 0x0000ffffu : 0u) | (in(2 * tig + 1) ? 0xffff0000u : 0u);
      const uint32_t mhi = (in(8 + 2 * tig) ? 0x0000ffffu : 0u) | (in(9 + 2 * tig) ? 0xffff0000u : 0u);
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        vb[j][0] &= mlo;
        vb[j][2] &= mlo;
        vb[j][1] &= mhi;
        vb[j][3] &= mhi;
      }
    }
    // O += P . V : pairs of n-tiles of 8 head_dim columns
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      mma_16816<kBF16>(o[2 * j], pa[0], pa[1], pa[2], pa[3], vb[j][0], vb[j][1]);
      mma_16816<kBF16>(o[2 * j + 1], pa[0], pa[1], pa[2], pa[3], vb[j][2], vb[j][3]);
      mma_16816<kBF16>(o[2 * j], pl[0], pl[1], pl[2], pl[3], vb[j][0], vb[j][1]);
      mma_16816<kBF16>(o[2 * j + 1], pl[0], pl[1], pl[2], pl[3], vb[j][2], vb[j][3]);
    }
  }

  // Write this warp's (m, l, o) rows into its merge slot: ml[2][16], o[16][D].
  __device__ __forceinline__ void store(float* slot, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int hr = 0; hr < (kHi ? 2 : 1); ++hr) {
      float lt = l[hr];
      lt += __shfl_xor_sync(0xffffffffu, lt, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      const int row = gid + 8 * hr;
      if (row < G) {
        if (tig == 0) {
          slot[row] = m[hr];
          slot[16 + row] = lt;
        }
        float* orow = slot + 32 + row * D;
#pragma unroll
        for (int n = 0; n < NT; ++n)
          *reinterpret_cast<float2*>(orow + n * 8 + 2 * tig) =
              make_float2(o[n][hr * 2], o[n][hr * 2 + 1]);
      }
    }
  }

  // A warp that holds a whole head's segment writes it directly: the output
  // rows (full context) or the partial state record (rows rec_row0 ..).
  __device__ __forceinline__ void write_direct(uint16_t* out_rows, float* rec, int rec_row0,
                                               int rec_rows, bool full, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int hr = 0; hr < (kHi ? 2 : 1); ++hr) {
      float lt = l[hr];
      lt += __shfl_xor_sync(0xffffffffu, lt, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      const int row = gid + 8 * hr;
      if (row < G) {
        if (full) {
          const float inv = 1.f / lt;
          uint16_t* orow = out_rows + (size_t)row * D;
#pragma unroll
          for (int n = 0; n < NT; ++n)
            *reinterpret_cast<uint32_t*>(orow + n * 8 + 2 * tig) =
                pack2<kBF16>(o[n][hr * 2] * inv, o[n][hr * 2 + 1] * inv);
        } else {
          const int r = rec_row0 + row;
          if (tig == 0) {
            rec[(size_t)rec_rows * D + r] = m[hr];
            rec[(size_t)rec_rows * D + rec_rows + r] = lt;
          }
          float* orow = rec + (size_t)r * D;
#pragma unroll
          for (int n = 0; n < NT; ++n)
            *reinterpret_cast<float2*>(orow + n * 8 + 2 * tig) =
                make_float2(o[n][hr * 2], o[n][hr * 2 + 1]);
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// Consumer state and tile math: tensor-core path with transposed products
// (group size at most 8).  S^T = K . Q^T and O^T += V^T . P^T put the 16
// tokens and head_dim on the MMA's 16-wide M side and the (up to 8) query
// heads on its 8-wide N side, so no MMA row is padding: per tile, 8 products
// for the scores and 8 per 16-bit half of P for the output, against 16 and
// 32 with the heads on M.  The K and V fragments are the same ldmatrix loads
// as there, taken as A operands; P^T's B fragments are the score
// accumulators packed to 16 bits and transposed in registers (movmatrix).
// ---------------------------------------------------------------------------
template <int D, bool kBF16, bool kSwz>
struct MmaConsumerT {
  static constexpr int KS = D / 16;   // k-steps of S^T over head_dim
  static constexpr int MT = D / 16;   // m-tiles of O^T over head_dim
  static constexpr int QP = q_pitch<D>();
  uint32_t qb[KS][2];   // Q^T: head gid, head_dim 16 ks + 2 tig (+1) and + 8
  float o[MT][4];       // O^T: head_dim 16 i + gid (+8) x heads 2 tig, 2 tig + 1
  float m[2];           // heads 2 tig + e: running maximum (the same in a tig's 8 lanes)
  float l[2];           // and this lane's share of their running sums

  // qslot: this head group's G query rows, QP bytes apart
  __device__ __forceinline__ void begin(uint32_t qslot, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d0 = ks * 16 + 2 * tig;
      uint32_t b0 = 0, b1 = 0;
      if (gid < G) {
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b0) : "r"(qslot + gid * QP + d0 * 2));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b1) : "r"(qslot + gid * QP + (d0 + 8) * 2));
      }
      qb[ks][0] = b0;
      qb[ks][1] = b1;
    }
#pragma unroll
    for (int i = 0; i < MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }

  // 16 tokens [tile0, tile0 + 16) of the chunk; tokens [lo, nv) of them are
  // valid, lo < nv (the others may hold anything, NaN included: their scores
  // are masked and their V values zeroed in registers).
  __device__ __forceinline__ void tile(uint32_t kpart, uint32_t vpart, int tile0, int lo, int nv,
                                       const DecodeArgs& a, float sl2) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    // K fragments: kb[h][kp][j] holds tokens 8 h + (0..7) x head_dim
    // 32 kp + 8 j + (0..7), so that k-step 2 kp + u takes kb[.][kp][2u], [2u + 1]
    uint32_t kb[2][D / 32][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int tt = tile0 + h * 8 + (lane & 7);
#pragma unroll
      for (int kp = 0; kp < D / 32; ++kp) {
        const int cidx = kp * 4 + (lane >> 3);
        const uint32_t ra = row_addr(kpart, tt, cidx >> 3, a);
        ldmatrix_x4(chunk_addr<kSwz>(ra, cidx & 7), kb[h][kp][0], kb[h][kp][1], kb[h][kp][2],
                    kb[h][kp][3]);
      }
    }
    // S^T: even and odd k-steps in two accumulation chains
    float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kp = 0; kp < D / 32; ++kp) {
      mma_16816<kBF16>(s, kb[0][kp][0], kb[1][kp][0], kb[0][kp][1], kb[1][kp][1], qb[2 * kp][0],
                       qb[2 * kp][1]);
      mma_16816<kBF16>(s2, kb[0][kp][2], kb[1][kp][2], kb[0][kp][3], kb[1][kp][3],
                       qb[2 * kp + 1][0], qb[2 * kp + 1][1]);
    }
    // V fragments (A of O^T): vb[j][.] holds tokens (0..7 | 8..15) x head_dim
    // 16 j + (0..7 | 8..15), loaded before the softmax math so that their
    // latency hides behind it
    uint32_t vb[MT][4];
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      const int mat = lane >> 3;
      const int tt = tile0 + ((mat & 1) << 3) + (lane & 7);
      const int cidx = 2 * j + (mat >> 1);
      const uint32_t ra = row_addr(vpart, tt, cidx >> 3, a);
      ldmatrix_x4_trans(chunk_addr<kSwz>(ra, cidx & 7), vb[j][0], vb[j][1], vb[j][2], vb[j][3]);
    }
    // online softmax per head column (heads 2 tig + e; this lane holds tokens
    // gid and gid + 8): the 8 lanes of a tig reduce the maximum by shuffles
    const bool t0ok = gid >= lo && gid < nv, t1ok = gid + 8 >= lo && gid + 8 < nv;
    const float x0 = t0ok ? (s[0] + s2[0]) * sl2 : -INFINITY;
    const float x1 = t0ok ? (s[1] + s2[1]) * sl2 : -INFINITY;
    const float x2 = t1ok ? (s[2] + s2[2]) * sl2 : -INFINITY;
    const float x3 = t1ok ? (s[3] + s2[3]) * sl2 : -INFINITY;
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
    }
    // token lo is valid, so both maxima are finite
    const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
    const float alpha0 = exp2f(m[0] - mn0), alpha1 = exp2f(m[1] - mn1);
    m[0] = mn0;
    m[1] = mn1;
    const float e0 = exp2f(x0 - mn0), e1 = exp2f(x1 - mn1);
    const float e2 = exp2f(x2 - mn0), e3 = exp2f(x3 - mn1);
    // P enters the products as a pair of 16-bit values, hi = round(P) and
    // lo = round(P - hi) (P - hi is exact in fp32), so that hi + lo is within
    // 2^-16 (bfloat16) or 2^-22 (binary16) of P; the normaliser l sums the
    // fp32 values.  One 16-bit P would move the output by up to the unit
    // roundoff times the spread of the values, many ulps of a small output.
    const uint32_t h01 = pack2<kBF16>(e0, e1), h23 = pack2<kBF16>(e2, e3);
    const float2 f01 = unpack2<kBF16>(h01), f23 = unpack2<kBF16>(h23);
    const uint32_t l01 = pack2<kBF16>(e0 - f01.x, e1 - f01.y);
    const uint32_t l23 = pack2<kBF16>(e2 - f23.x, e3 - f23.y);
    l[0] = l[0] * alpha0 + (e0 + e2);
    l[1] = l[1] * alpha1 + (e1 + e3);
    // once the running maxima settle, alpha is exactly 1 in every lane and
    // the rescale is skipped (multiplying by 1 changes nothing)
    if (__any_sync(0xffffffffu, alpha0 != 1.f || alpha1 != 1.f)) {
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        o[i][0] *= alpha0;
        o[i][1] *= alpha1;
        o[i][2] *= alpha0;
        o[i][3] *= alpha1;
      }
    }
    // P^T's B fragments: head gid x tokens 2 tig (+1) and 2 tig + 8 (+9)
    const uint32_t ph0 = movmatrix_trans(h01), ph1 = movmatrix_trans(h23);
    const uint32_t pl0 = movmatrix_trans(l01), pl1 = movmatrix_trans(l23);
    if (nv < kTile || lo > 0) {
      // zero the V values of tokens outside [lo, nv) (the low 16 bits of a
      // fragment register hold token 2tig (+8), the high bits token 2tig+1)
      auto in = [&](int t) { return t >= lo && t < nv; };
      const uint32_t mlo = (in(2 * tig) ? 0x0000ffffu : 0u) | (in(2 * tig + 1) ? 0xffff0000u : 0u);
      const uint32_t mhi = (in(8 + 2 * tig) ? 0x0000ffffu : 0u) | (in(9 + 2 * tig) ? 0xffff0000u : 0u);
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        vb[j][0] &= mlo;
        vb[j][2] &= mlo;
        vb[j][1] &= mhi;
        vb[j][3] &= mhi;
      }
    }
    // O^T += V^T . P^T, m-tile j = head_dim 16 j .. 16 j + 15
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      mma_16816<kBF16>(o[j], vb[j][0], vb[j][2], vb[j][1], vb[j][3], ph0, ph1);
      mma_16816<kBF16>(o[j], vb[j][0], vb[j][2], vb[j][1], vb[j][3], pl0, pl1);
    }
  }

  // the full sum of head 2 tig + e over the 8 lanes that share it
  __device__ __forceinline__ float total_l(int e) const {
    float lt = l[e];
    lt += __shfl_xor_sync(0xffffffffu, lt, 4);
    lt += __shfl_xor_sync(0xffffffffu, lt, 8);
    lt += __shfl_xor_sync(0xffffffffu, lt, 16);
    return lt;
  }

  // this lane's fp32 values of head 2 tig + e into row `orow` (D floats)
  __device__ __forceinline__ void store_row_f32(float* orow, int e) const {
    const int gid = (threadIdx.x & 31) >> 2;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      orow[16 * i + gid] = o[i][e];
      orow[16 * i + 8 + gid] = o[i][2 + e];
    }
  }

  // Write this warp's (m, l, o) rows into its merge slot: ml[2][16], o[16][D].
  __device__ __forceinline__ void store(float* slot, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float lt = total_l(e);
      const int row = 2 * tig + e;
      if (row < G) {
        if (gid == 0) {
          slot[row] = m[e];
          slot[16 + row] = lt;
        }
        store_row_f32(slot + 32 + row * D, e);
      }
    }
  }

  // A warp that holds a whole head group's segment writes it directly: the
  // output rows (full context, each normalised and rounded once, then
  // transposed in registers so that a lane writes pairs of columns) or the
  // partial state record (rows rec_row0 ..).
  __device__ __forceinline__ void write_direct(uint16_t* out_rows, float* rec, int rec_row0,
                                               int rec_rows, bool full, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const float lt0 = total_l(0), lt1 = total_l(1);
    if (full) {
      const float inv0 = 1.f / lt0, inv1 = 1.f / lt1;
      uint16_t* dst = out_rows + (size_t)gid * D + 2 * tig;
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const uint32_t t0 = movmatrix_trans(pack2<kBF16>(o[i][0] * inv0, o[i][1] * inv1));
        const uint32_t t1 = movmatrix_trans(pack2<kBF16>(o[i][2] * inv0, o[i][3] * inv1));
        if (gid < G) {
          *reinterpret_cast<uint32_t*>(dst + 16 * i) = t0;
          *reinterpret_cast<uint32_t*>(dst + 16 * i + 8) = t1;
        }
      }
      return;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int row = 2 * tig + e;
      if (row >= G) continue;
      const int r = rec_row0 + row;
      if (gid == 0) {
        rec[(size_t)rec_rows * D + r] = m[e];
        rec[(size_t)rec_rows * D + rec_rows + r] = e ? lt1 : lt0;
      }
      store_row_f32(rec + (size_t)r * D, e);
    }
  }
};

// ---------------------------------------------------------------------------
// Consumer state and tile math: CUDA-core path (group size 1)
// ---------------------------------------------------------------------------
template <int D, bool kBF16, bool kF8 = false>
struct SimtConsumer {
  static constexpr int VEC = D / 32;   // head_dim elements per lane
  float qf[VEC];
  float o[VEC];
  float m, l;
  float vscale = 1.f;                  // E4M3 cache: the V scale, applied to the output

  __device__ __forceinline__ int col() const { return (threadIdx.x & 31) * VEC; }

  __device__ __forceinline__ void load_row(uint32_t part, int tt, const DecodeArgs& a,
                                           float* x) const {
    const int c = col();
    if constexpr (kF8) {
      // E4M3 rows of D bytes, unswizzled: this lane's VEC codes, exact in f16
      const uint32_t ra = row_addr(part, tt, 0, a) + (uint32_t)c;
      if constexpr (VEC == 4) {
        uint32_t w;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(ra));
        const float2 p = unpack2<false>(e4m3x2_to_f16x2(w & 0xffffu));
        const float2 q = unpack2<false>(e4m3x2_to_f16x2(w >> 16));
        x[0] = p.x; x[1] = p.y; x[2] = q.x; x[3] = q.y;
      } else {
        uint16_t h;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(ra));
        const float2 p = unpack2<false>(e4m3x2_to_f16x2(h));
        x[0] = p.x; x[1] = p.y;
      }
      return;
    }
    const uint32_t ra = row_addr(part, tt, c >> 6, a) + (uint32_t)((c & 63) * 2);
    if constexpr (VEC == 4) {
      uint32_t w0, w1;
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(ra));
      const float2 p = unpack2<kBF16>(w0), q = unpack2<kBF16>(w1);
      x[0] = p.x; x[1] = p.y; x[2] = q.x; x[3] = q.y;
    } else {
      uint32_t w0;
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w0) : "r"(ra));
      const float2 p = unpack2<kBF16>(w0);
      x[0] = p.x; x[1] = p.y;
    }
  }

  __device__ __forceinline__ void begin(uint32_t qslot, int /*G*/) {
    const int c = col();
#pragma unroll
    for (int v = 0; v < VEC; v += 2) {
      uint32_t w;
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(qslot + (c + v) * 2));
      const float2 f = unpack2<kBF16>(w);
      qf[v] = f.x;
      qf[v + 1] = f.y;
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) o[v] = 0.f;
    m = -INFINITY;
    l = 0.f;
  }

  // tokens [lo, nv) of [tile0, tile0 + 16) are valid
  __device__ __forceinline__ void tile(uint32_t kpart, uint32_t vpart, int tile0, int lo, int nv,
                                       const DecodeArgs& a, float sl2) {
    const int lane = threadIdx.x & 31;
    // partial dot products of the 16 tokens over this lane's head_dim slice
    float part[kTile];
#pragma unroll
    for (int t = 0; t < kTile; ++t) {
      float x[VEC];
      load_row(kpart, tile0 + t, a, x);
      float acc = 0.f;
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc = fmaf(qf[v], x[v], acc);
      part[t] = acc;
    }
    // transpose-reduce across the warp: halve the token set at offsets
    // 16, 8, 4, 2, then add at offset 1; lanes 2t and 2t+1 end with token t
    int n = kTile;
#pragma unroll
    for (int off = 16; off >= 2; off >>= 1) {
      n >>= 1;
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int t = 0; t < kTile / 2; ++t) {
        if (t < n) {
          const float send = upper ? part[t] : part[t + n];
          const float keep = upper ? part[t + n] : part[t];
          part[t] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
    }
    float sc = part[0] + __shfl_xor_sync(0xffffffffu, part[0], 1);
    const int my_t = lane >> 1;
    sc = (my_t >= lo && my_t < nv) ? sc * sl2 : -INFINITY;
    float mt = sc;
#pragma unroll
    for (int off = 2; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
    const float mn = fmaxf(m, mt);
    const float alpha = exp2f(m - mn);
    m = mn;
    const float p = exp2f(sc - mn);
    l = l * alpha + ((lane & 1) ? 0.f : p);
#pragma unroll
    for (int v = 0; v < VEC; ++v) o[v] *= alpha;
    if (nv == kTile && lo == 0) {
#pragma unroll
      for (int t = 0; t < kTile; ++t) {
        const float pt = __shfl_sync(0xffffffffu, p, 2 * t);
        float x[VEC];
        load_row(vpart, tile0 + t, a, x);
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = fmaf(pt, x[v], o[v]);
      }
    } else {
      for (int t = lo; t < nv; ++t) {
        const float pt = __shfl_sync(0xffffffffu, p, 2 * t);
        float x[VEC];
        load_row(vpart, tile0 + t, a, x);
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = fmaf(pt, x[v], o[v]);
      }
    }
  }

  __device__ __forceinline__ float total_l() const {
    float lt = l;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
    return lt;
  }

  __device__ __forceinline__ void store(float* slot, int /*G*/) {
    const float lt = total_l();
    if ((threadIdx.x & 31) == 0) {
      slot[0] = m;
      slot[16] = lt;
    }
    float* orow = slot + 32;
#pragma unroll
    for (int v = 0; v < VEC; ++v) orow[col() + v] = o[v] * vscale;
  }

  __device__ __forceinline__ void write_direct(uint16_t* out_rows, float* rec, int rec_row0,
                                               int rec_rows, bool full, int /*G*/) {
    const float lt = total_l();
    const int c = col();
    if (full) {
      const float inv = vscale / lt;
#pragma unroll
      for (int v = 0; v < VEC; v += 2)
        *reinterpret_cast<uint32_t*>(out_rows + c + v) = pack2<kBF16>(o[v] * inv, o[v + 1] * inv);
    } else {
      if ((threadIdx.x & 31) == 0) {
        rec[(size_t)rec_rows * D + rec_row0] = m;
        rec[(size_t)rec_rows * D + rec_rows + rec_row0] = lt;
      }
      float* orow = rec + (size_t)rec_row0 * D;
#pragma unroll
      for (int v = 0; v < VEC; ++v) orow[c + v] = o[v] * vscale;
    }
  }
};

}  // namespace pa

#include "pa_decode_fp8.cuh"

namespace pa {

// ---------------------------------------------------------------------------
// Segment merge across the TPH warps of each head and the output / partial
// write (used when a head is split over several warps, TPH > 1).
// ---------------------------------------------------------------------------
template <int D, bool kBF16>
__device__ __forceinline__ void merge_and_write(const DecodeArgs& a, const float* mbuf, int i,
                                                int grp, bool full, int slot_idx) {
  const int G = a.G, HG = a.HG, TPH = a.TPH;
  const int rows = HG * G;
  const int slot_floats = 32 + G * D;
  float* rec = a.ws_rec + ((size_t)blockIdx.x * 2 + slot_idx) * rec_floats(rows, D);
  for (int e = threadIdx.x; e < rows * (D / 2); e += kCWarps * 32) {
    const int r = e / (D / 2);             // row = head_local * G + g
    const int d = 2 * (e % (D / 2));
    const int hl = r / G, g = r - hl * G;
    float mx = -INFINITY;
    for (int t = 0; t < TPH; ++t) mx = fmaxf(mx, mbuf[(hl * TPH + t) * slot_floats + g]);
    float L = 0.f, o0 = 0.f, o1 = 0.f;
    for (int t = 0; t < TPH; ++t) {
      const float* sw = mbuf + (hl * TPH + t) * slot_floats;
      const float mw = sw[g];
      const float wt = (mw == -INFINITY) ? 0.f : exp2f(mw - mx);
      const float2 ov = *reinterpret_cast<const float2*>(sw + 32 + g * D + d);
      L = fmaf(wt, sw[16 + g], L);
      o0 = fmaf(wt, ov.x, o0);
      o1 = fmaf(wt, ov.y, o1);
    }
    if (full) {
      const float inv = 1.f / L;
      uint16_t* dst = a.out + ((size_t)i * a.Hq + (size_t)grp * rows + r) * D + d;
      *reinterpret_cast<uint32_t*>(dst) = pack2<kBF16>(o0 * inv, o1 * inv);
    } else {
      *reinterpret_cast<float2*>(rec + (size_t)r * D + d) = make_float2(o0, o1);
      if (d == 0) {
        rec[(size_t)rows * D + r] = mx;
        rec[(size_t)rows * D + rows + r] = L;
      }
    }
  }
}

// Gather mode: copy the valid rows of this warp's 16-token tile of its head to
// the contiguous outputs, undoing the shared-memory layout.
template <int D, bool kSwz>
__device__ __forceinline__ void gather_tile(const DecodeArgs& a, uint32_t kpart, uint32_t vpart,
                                            int tile0, int nv, int i, int head, int c) {
  const int lane = threadIdx.x & 31;
  const long long row0 = __ldg(a.out_off + i) + (long long)c * a.CT + tile0;
  for (int e = lane; e < nv * (D / 8); e += 32) {
    const int r = e / (D / 8);
    const int cj = e % (D / 8);
    const uint32_t ka = chunk_addr<kSwz>(row_addr(kpart, tile0 + r, cj >> 3, a), cj & 7);
    const uint32_t va = chunk_addr<kSwz>(row_addr(vpart, tile0 + r, cj >> 3, a), cj & 7);
    uint4 kv, vv;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(kv.x), "=r"(kv.y), "=r"(kv.z), "=r"(kv.w)
                 : "r"(ka));
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(vv.x), "=r"(vv.y), "=r"(vv.z), "=r"(vv.w)
                 : "r"(va));
    const size_t off = (((size_t)(row0 + r) * a.Hkv + head) * D) + cj * 8;
    *reinterpret_cast<uint4*>(a.k_out + off) = kv;
    *reinterpret_cast<uint4*>(a.v_out + off) = vv;
  }
}

// ---------------------------------------------------------------------------
// Merge of a context split across CTAs, run by the CTA whose piece arrived
// last.  The context's chunks start at global chunk index g0 and number nc,
// so its pieces sit in CTAs first = g0 / cpc .. last = (g0 + nc - 1) / cpc,
// each in record slot 0 except the first CTA's when the context began after
// that CTA's own first chunk (then it is that CTA's second segment, slot 1):
//   out = sum_k 2^(m_k - m*) o_k / sum_k 2^(m_k - m*) l_k.
// D / 16 threads share a row, each owning 16 of its head_dim columns, and
// fold pieces in with the online rescaling, a piece's (m, l) and 16 o values
// loaded together.  When one set of rows x D / 16 threads leaves room, up to
// 256 / set sets take every set-th piece in parallel and their partial
// states are combined through shared memory (scratch: the stage buffers,
// idle once the loop is done).  Consumer threads only; the records come
// from other CTAs, so they are read from L2 (ld.global.cg).
// ---------------------------------------------------------------------------
template <int D>
struct MergeState {
  float m = -INFINITY, l = 0.f;
  float4 acc[4];
  __device__ __forceinline__ MergeState() {
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // fold in a partial state (mk, lk, ok) with weight 2^(mk - m*)
  __device__ __forceinline__ void fold(float mk, float lk, const float4* ok) {
    if (mk == -INFINITY) return;
    const float mn = fmaxf(m, mk);
    const float so = exp2f(m - mn), sn = exp2f(mk - mn);   // so = 0 while m = -inf
    l = l * so + lk * sn;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      acc[c].x = acc[c].x * so + ok[c].x * sn;
      acc[c].y = acc[c].y * so + ok[c].y * sn;
      acc[c].z = acc[c].z * so + ok[c].z * sn;
      acc[c].w = acc[c].w * so + ok[c].w * sn;
    }
    m = mn;
  }
};

// Not inlined, with scalar arguments: its registers stay out of the
// allocation of the kernel's main loop.
template <int D, bool kBF16, int kBatch>
__device__ __forceinline__ void merge_split(uint16_t* out, const float* ws_rec, int Hq, int rows,
                                         int i, int grp, long long g0, int nc, long long cpc,
                                         float* scratch) {
  const int tid = threadIdx.x;   // consumer threads 0 .. kCWarps * 32 - 1
  constexpr int kThr = kCWarps * 32;
  constexpr int kTPR = D / 16;   // threads per row
  const int first = (int)(g0 / cpc);
  const int last = (int)((g0 + nc - 1) / cpc);
  const size_t rf = rec_floats(rows, D);
  const size_t ml = (size_t)rows * D;   // m[] then l[] follow o[][]
  const int set = rows * kTPR;
  int nsets = set <= kThr ? kThr / set : 1;
  if (nsets > last - first + 1) nsets = last - first + 1;
  const int d = (tid % kTPR) * 16;
  // Pieces are read kBatch at a time, every load of a batch issued before its
  // first fold, so that a batch costs one L2 round trip.  Only the 16-bit
  // tensor-core kernels batch, where two pieces fit in their registers: in
  // the others the extra registers raise spills in the main loop (measured:
  // +0.4 us on the E4M3 decode with two, +3.9 us with four).
  auto fold_pieces = [&](MergeState<D>& st, int r, int k0, int step) {
    for (int kb = k0; kb <= last; kb += kBatch * step) {
      float mk[kBatch], lk[kBatch];
      float4 ok[kBatch][4];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int k = kb + u * step;
        mk[u] = -INFINITY;
        lk[u] = 0.f;
        if (k <= last) {
          const int slot = (k == first && g0 != (long long)first * cpc) ? 1 : 0;
          const float* rec = ws_rec + ((size_t)k * 2 + slot) * rf;
          mk[u] = __ldcg(rec + ml + r);
          lk[u] = __ldcg(rec + ml + rows + r);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            ok[u][c] = __ldcg(reinterpret_cast<const float4*>(rec + (size_t)r * D + d + 4 * c));
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (kb + u * step <= last) st.fold(mk[u], lk[u], ok[u]);
    }
  };
  auto write_row = [&](const MergeState<D>& st, int r) {
    const float inv = 1.f / st.l;
    uint4 pk[2];
    uint32_t* w = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      w[2 * c] = pack2<kBF16>(st.acc[c].x * inv, st.acc[c].y * inv);
      w[2 * c + 1] = pack2<kBF16>(st.acc[c].z * inv, st.acc[c].w * inv);
    }
    uint4* dst =
        reinterpret_cast<uint4*>(out + ((size_t)i * Hq + (size_t)grp * rows + r) * D + d);
    dst[0] = pk[0];
    dst[1] = pk[1];
  };
  if (nsets <= 1) {
    for (int r = tid / kTPR; r < rows; r += kThr / kTPR) {
      MergeState<D> st;
      fold_pieces(st, r, first, 1);
      write_row(st, r);
    }
    return;
  }
  // several sets: set q folds pieces first + q, first + q + nsets, ...; its
  // state for row r goes to scratch[(q * rows + r) * (D + 4)]: o[D], m, l
  const int q = tid / set, r = (tid % set) / kTPR;
  if (q < nsets) {
    MergeState<D> st;
    fold_pieces(st, r, first + q, nsets);
    float* sp = scratch + (size_t)(q * rows + r) * (D + 4);
#pragma unroll
    for (int c = 0; c < 4; ++c) *reinterpret_cast<float4*>(sp + d + 4 * c) = st.acc[c];
    if (d == 0) {
      sp[D] = st.m;
      sp[D + 1] = st.l;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kThr) : "memory");
  if (tid < set) {
    MergeState<D> st;
    for (int p = 0; p < nsets; ++p) {
      const float* sp = scratch + (size_t)(p * rows + r) * (D + 4);
      st.fold(sp[D], sp[D + 1], reinterpret_cast<const float4*>(sp + d));
    }
    write_row(st, r);
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kThr) : "memory");   // scratch is reused by the next merge
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int D, bool kBF16, int kMode, bool kSwz, bool kHi, bool kF8>
__global__ void __launch_bounds__(block_threads(kMode, kF8, kHi), 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (128-byte swizzled TMA boxes need it)
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  constexpr int kThreads = block_threads(kMode, kF8, kHi);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.stages;
  const uint32_t bar_full = base + a.ctrl_off;      // S x 8 bytes
  const uint32_t bar_empty = bar_full + 8 * S;      // S x 8 bytes
  const uint32_t bar_qfull = bar_empty + 8 * S;     // kQBufs x 8 bytes
  const uint32_t bar_qempty = bar_qfull + 8 * kQBufs;
  const int ctrl_words = a.ctrl_off + 16 * S + 16 * kQBufs;
  long long* const scan_tmp = reinterpret_cast<long long*>(gbase + ctrl_words);
  int* const ctrl = reinterpret_cast<int*>(gbase + ctrl_words + kScanBytes);
  volatile int* const abort_flag = ctrl + 4;
  int* const s_len = reinterpret_cast<int*>(gbase + ctrl_words + kScanBytes + kCtrlBytes);

  if (tid == 0) {
    ctrl[0] = -1;
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kCWarps);
    }
    for (int s = 0; s < kQBufs; ++s) {
      mbar_init(bar_qfull + 8 * s, 32);   // one arrival per producer lane
      mbar_init(bar_qempty + 8 * s, kCWarps);
    }
    *abort_flag = 0;
    ctrl[kCtrlMerges] = 0;
    ctrl[kCtrlEmpty] = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  // Warm L2 with the small inputs (lengths, block tables, queries) while the
  // previous kernel in the stream drains: a prefetch returns no data, so it
  // is harmless even if that kernel is still writing them.
  {
    const size_t step = (size_t)gridDim.x * blockDim.x * 128;
    const size_t t0 = ((size_t)blockIdx.x * blockDim.x + tid) * 128;
    const char* sl = reinterpret_cast<const char*>(a.seq_lens);
    const char* bt = reinterpret_cast<const char*>(a.bt);
    const size_t sl_bytes = (size_t)a.num_seqs * 4, bt_bytes = sl_bytes * a.stride;
    for (size_t o = t0; o < sl_bytes; o += step) prefetch_l2(sl + o);
    for (size_t o = t0; o < bt_bytes; o += step) prefetch_l2(bt + o);
    if (kMode != kModeGather) {
      // the split-context counters: a piece's count waits on its line
      const char* wc = reinterpret_cast<const char*>(a.ws_count);
      for (size_t o = t0; o < (size_t)gridDim.x * 4; o += step) prefetch_l2(wc + o);
      const char* qp = reinterpret_cast<const char*>(a.q);
      const size_t q_bytes = (size_t)a.num_seqs * a.Hq * D * 2;
      for (size_t o = t0; o < q_bytes; o += step) prefetch_l2(qp + o);
    }
  }
  // inputs may come from the previous kernel in the stream; with early
  // tables only q, the pools, out and the workspace may, and the lengths and
  // tables are read first, while that kernel drains
  if (!a.early_tables) grid_dep_wait();

  // ---- find this CTA's range of chunks -------------------------------------
  // The work is the list of chunks over (sequence, head group, CT tokens), in
  // that order, cut into equal contiguous ranges of cpc chunks.  One pass:
  // each thread sums the chunks of a contiguous run of sequences, one
  // block-wide scan gives every run's offset, and the thread whose run holds
  // this CTA's first chunk locates it.
  const int per = (a.num_seqs + kThreads - 1) / kThreads;
  const int run0 = min(a.num_seqs, tid * per), run1 = min(a.num_seqs, run0 + per);
  long long my_nc = 0;
  for (int i = run0; i < run1; ++i) {
    const int T0 = __ldg(a.seq_lens + i);
    const int T = clamp_len(T0, a.stride, a.B);
    my_nc += seq_chunks(T, a);
    if (i < kLenCache) s_len[i] = T;
    if ((i % gridDim.x) == blockIdx.x && (T != T0 || (kMode != kModeGather && T == 0))) {
      if (a.early_tables) {
        ctrl[kCtrlEmpty] = 1;   // reported and zeroed below, once err and out may be written
      } else {
        if (T != T0) set_error(a.err, PA_DEVERR_SEQ_LEN);
        if (kMode != kModeGather && T == 0) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + (size_t)i * a.Hq * D);
          for (int e = 0; e < a.Hq * D / 2; ++e) dst[e] = 0u;
        }
      }
    }
  }
  long long total_nc;
  const long long my_excl = block_scan_incl<kThreads>(my_nc, scan_tmp, total_nc) - my_nc;
  const long long U = total_nc * a.NGR;
  const long long cpc = (U + gridDim.x - 1) / gridDim.x;
  const long long start = (long long)blockIdx.x * cpc;
  const long long end = min(U, start + cpc);
  const int n_chunks = (start < end) ? (int)(end - start) : 0;
  if (n_chunks > 0 && my_nc > 0 && start >= my_excl * a.NGR && start < (my_excl + my_nc) * a.NGR) {
    long long off = my_excl * a.NGR;
    for (int i = run0; i < run1; ++i) {
      const int nc = seq_chunks(clamp_len(__ldg(a.seq_lens + i), a.stride, a.B), a);
      const long long span = (long long)nc * a.NGR;
      if (nc > 0 && start < off + span) {
        const long long rem = start - off;
        ctrl[0] = i;
        ctrl[1] = (int)(rem / nc);
        ctrl[2] = (int)(rem % nc);
        break;
      }
      off += span;
    }
  }
  __syncthreads();
  // let the next kernel get scheduled; it still waits for this whole grid
  // before reading anything
  if (tid == 0) grid_dep_launch();
  if (a.early_tables && ctrl[kCtrlEmpty]) {
    grid_dep_wait();
    for (int i = run0; i < run1; ++i) {
      if ((i % gridDim.x) != blockIdx.x) continue;
      const int T0 = __ldg(a.seq_lens + i);
      const int T = clamp_len(T0, a.stride, a.B);
      if (T != T0) set_error(a.err, PA_DEVERR_SEQ_LEN);
      if (kMode != kModeGather && T == 0) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + (size_t)i * a.Hq * D);
        for (int e = 0; e < a.Hq * D / 2; ++e) dst[e] = 0u;
      }
    }
  }
  if (n_chunks == 0) return;
  // Cannot happen for a consistent scan (seq_lens changing during the call
  // could cause it); never walk blind.  This CTA's pieces go uncounted, so
  // the caller must zero the workspace again (the no-allocation entry point
  // clears its counters at every call).
  if (ctrl[0] < 0) {
    if (a.early_tables) grid_dep_wait();
    if (tid == 0) set_error(a.err, PA_DEVERR_SEQ_LEN);
    return;
  }

  Walk w0;
  w0.i = ctrl[0];
  w0.g = ctrl[1];
  w0.c = ctrl[2];
  walk_load_seq(w0, a, s_len);

  const uint32_t box_bytes = 1u << a.sub_log2;

  if (warp >= kCWarps) {
    if constexpr (split_regs(kMode, kF8, kHi)) {
      setmaxnreg_dec<kProducerRegs>();
      if (warp != kProducerWarp) return;
    }
    // ======================= producer =======================
    const uint64_t pol = policy_evict_first();
    Walk w = w0;
    auto load_entry = [&](const Walk& ww) -> int {
      int ent = -1;
      if (lane < a.nsb) {
        const int tok0 = ww.t0 + ww.c * a.CT + lane * a.R;
        if (tok0 < ww.T) ent = __ldg(a.bt + (size_t)ww.i * a.stride + (tok0 >> a.log2B));
      }
      return ent;
    };
    int ent = load_entry(w);
    // the pools and q may come from the preceding kernel
    if (a.early_tables) grid_dep_wait();
    int issued = 0;
    uint32_t seg = 0;
    int st = 0;          // stage of chunk n (n % S), kept incrementally
    uint32_t ph = 0;     // phase parity of that stage ((n / S) & 1)
    for (int n = 0; n < n_chunks; ++n) {
      const bool seg_start = (n == 0) || (w.c == 0);
      if (kMode != kModeGather && seg_start) {
        // this segment's query rows, into query buffer seg % kQBufs once the
        // consumers have taken the rows of segment seg - kQBufs out of it
        const int qb = (int)(seg % kQBufs);
        bool waited = true;
        if (seg >= kQBufs)
          waited = mbar_wait_bounded(bar_qempty + 8 * qb, ((seg / kQBufs) - 1) & 1u, abort_flag);
        const bool timed_out = __any_sync(0xffffffffu, !waited);
        if (__any_sync(0xffffffffu, timed_out || *abort_flag != 0)) {
          if (lane == 0) {
            if (timed_out) set_error(a.err, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
          break;
        }
        {
          // the rows by 16-byte asynchronous copies into rows q_pitch apart
          // (one TMA bulk copy per row would queue dozens of small copies in
          // front of the next chunk's); every lane arrives once its own
          // copies have landed
          constexpr int kPR = D * 2 / 16;   // 16-byte pieces per row
          const uint32_t qdst = base + a.q_off + (uint32_t)qb * a.q_stride;
          const char* qsrc = reinterpret_cast<const char*>(
              a.q + ((size_t)w.i * a.Hq + (size_t)w.g * a.HG * a.G) * D);
          for (int e = lane; e < a.HG * a.G * kPR; e += 32) {
            const int r = e / kPR, c = e % kPR;
            cp_async16(qdst + (uint32_t)(r * q_pitch<D>() + c * 16), qsrc + (size_t)e * 16);
          }
          cp_async_arrive_noinc(bar_qfull + 8 * qb);
        }
        __syncwarp();
        ++seg;
      }
      const bool waited = mbar_wait_bounded(bar_empty + 8 * st, ph ^ 1u, abort_flag);
      const bool timed_out = __any_sync(0xffffffffu, !waited);
      if (__any_sync(0xffffffffu, timed_out || *abort_flag != 0)) {
        if (lane == 0) {
          if (timed_out) set_error(a.err, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      const int valid_tok = min(a.CT, w.T - w.t0 - w.c * a.CT);
      const int nvsub = (valid_tok + a.R - 1) >> a.log2R;
      const bool in_sub = lane < nvsub;
      const bool ok = in_sub && ent >= 0 && (long long)ent < a.num_blocks;
      if (in_sub && !ok) set_error(a.err, PA_DEVERR_BLOCK_ID);
      const unsigned okmask = __ballot_sync(0xffffffffu, ok);
      const uint32_t sbase = base + (uint32_t)st * a.stage_bytes;
      if (lane == 0) {
        const uint32_t tx = (uint32_t)__popc(okmask) * box_bytes * 2u;
        mbar_arrive_expect_tx(bar_full + 8 * st, tx);
      }
      __syncwarp();
      if (ok) {
        const int row_off = (w.t0 + w.c * a.CT + lane * a.R) & (a.B - 1);
        const uint32_t dk = sbase + (uint32_t)lane * box_bytes;
        const int h0 = w.g * a.HG;
        if (a.split_rows) {
          tma_load_5d(dk, &tmk, bar_full + 8 * st, 0, row_off, 0, h0, ent, pol);
          tma_load_5d(dk + a.kv_bytes, &tmv, bar_full + 8 * st, 0, row_off, 0, h0, ent, pol);
        } else {
          tma_load_5d(dk, &tmk, bar_full + 8 * st, 0, 0, h0, row_off, ent, pol);
          tma_load_5d(dk + a.kv_bytes, &tmv, bar_full + 8 * st, 0, 0, h0, row_off, ent, pol);
        }
      }
      // at a sequence's first chunk, pull the next sequence's block-table row
      // towards L1 so that its first entries do not stall the next segment
      if (w.c == 0 && w.g == 0 && lane < 2 && w.i + 1 < a.num_seqs && lane * 32 < a.stride)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(a.bt + (size_t)(w.i + 1) * a.stride + lane * 32));
      ++issued;
      if (++st == S) {
        st = 0;
        ph ^= 1u;
      }
      walk_advance(w, a, s_len);
      if (n + 1 < n_chunks) ent = load_entry(w);
    }
    // drain: make sure no TMA write is still in flight into this CTA's shared
    // memory when it exits (only matters after an abort)
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      for (int k = max(0, issued - S); k < issued; ++k)
        mbar_wait_bounded(bar_full + 8 * (k % S), (uint32_t)(k / S) & 1u, nullptr);
      for (uint32_t k = (seg > kQBufs ? seg - kQBufs : 0); k < seg; ++k)
        mbar_wait_bounded(bar_qfull + 8 * (k % kQBufs), (k / kQBufs) & 1u, nullptr);
    }
    return;
  }

  // ======================= consumers =======================
  if constexpr (split_regs(kMode, kF8, kHi)) setmaxnreg_inc<kConsumerRegs>();
  // out and the workspace may be touched by the preceding kernel
  if (a.early_tables) grid_dep_wait();
  using Mma16 = typename std::conditional<kHi, MmaConsumer<D, kBF16, kSwz, kHi>,
                                          MmaConsumerT<D, kBF16, kSwz>>::type;
  using Mma = typename std::conditional<kF8, MmaConsumerF8<D, kBF16, kSwz, kHi>, Mma16>::type;
  using Consumer =
      typename std::conditional<kMode == kModeSimt, SimtConsumer<D, kBF16, kF8>, Mma>::type;
  Consumer cs;
  if constexpr (kF8) cs.vscale = a.v_scale;
  float* const mbuf = reinterpret_cast<float*>(gbase + a.merge_off);
  const int slot_floats = 32 + a.G * D;
  const int hl = warp / a.TPH;                 // this warp's head within the group
  // tokens per warp per chunk: 32 for the E4M3 tensor-core consumer, else 16
  constexpr int kWarpTile = (kF8 && kMode == kModeMma) ? kTileF8 : kTile;
  const int tile0 = (warp % a.TPH) * kWarpTile;   // and its tokens of every chunk
  const uint32_t head_off = (uint32_t)hl << a.head_log2;
  const int rows = a.HG * a.G;
  Walk w = w0;
  int seg_c0 = w.c;
  bool first_seg = true;
  uint32_t seg = 0;
  const float sl2 = a.scale_log2;
  int st = 0;          // stage of chunk n (n % S), kept incrementally
  uint32_t ph = 0;     // phase parity of that stage ((n / S) & 1)
  for (int n = 0; n < n_chunks; ++n) {
    const bool seg_start = (n == 0) || (w.c == 0);
    if (seg_start) {
      seg_c0 = w.c;
      if constexpr (kMode != kModeGather) {
        const int qb = (int)(seg % kQBufs);
        if (!*abort_flag) {
          if (!mbar_wait_bounded(bar_qfull + 8 * qb, (seg / kQBufs) & 1u, abort_flag) &&
              lane == 0) {
            set_error(a.err, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
        }
        if (!__any_sync(0xffffffffu, *abort_flag != 0))
          cs.begin(base + a.q_off + (uint32_t)qb * a.q_stride +
                       (uint32_t)(hl * a.G * q_pitch<D>()), a.G);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_qempty + 8 * qb);
        ++seg;
      }
    }
    if (!*abort_flag) {
      if (!mbar_wait_bounded(bar_full + 8 * st, ph, abort_flag)) {
        if (lane == 0) {
          set_error(a.err, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
      }
    }
    const bool live = !__any_sync(0xffffffffu, *abort_flag != 0);
    const uint32_t sbase = base + (uint32_t)st * a.stage_bytes;
    const uint32_t kpart = sbase + head_off, vpart = sbase + a.kv_bytes + head_off;
    const int valid_tok = min(a.CT, w.T - w.t0 - w.c * a.CT);
    const int nv = max(0, min(kWarpTile, valid_tok - tile0));
    // tokens of this warp's tile before the window (chunk 0 only)
    const int lo = w.c == 0 ? max(0, w.lo - tile0) : 0;
    if (live && nv > lo) {
      if constexpr (kMode == kModeGather) {
        gather_tile<D, kSwz>(a, kpart, vpart, tile0, nv, w.i, w.g * a.HG + hl, w.c);
      } else {
        cs.tile(kpart, vpart, tile0, lo, nv, a, sl2);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * st);

    const bool seg_end = (n == n_chunks - 1) || (w.c == w.nc - 1);
    if constexpr (kMode != kModeGather) {
      if (seg_end) {
        const bool full = (seg_c0 == 0) && (w.c == w.nc - 1);
        const int slot_idx = first_seg ? 0 : 1;
        if (a.TPH == 1) {
          // this warp holds the whole head: write it out directly
          uint16_t* out_rows =
              a.out + ((size_t)w.i * a.Hq + (size_t)(w.g * a.HG + hl) * a.G) * D;
          float* rec = a.ws_rec + ((size_t)blockIdx.x * 2 + slot_idx) * rec_floats(rows, D);
          cs.write_direct(out_rows, rec, hl * a.G, rows, full, a.G);
        } else {
          cs.store(mbuf + warp * slot_floats, a.G);
          asm volatile("bar.sync 1, %0;" ::"r"(kCWarps * 32) : "memory");
          merge_and_write<D, kBF16>(a, mbuf, w.i, w.g, full, slot_idx);
          asm volatile("bar.sync 1, %0;" ::"r"(kCWarps * 32) : "memory");
        }
        if (!full) {
          // a piece of a context split across CTAs: once its record is
          // complete, count it on the counter of the context's last CTA; the
          // piece that completes the count owes the merge
          asm volatile("bar.sync 1, %0;" ::"r"(kCWarps * 32) : "memory");
          if (tid == 0) {
            const long long g0 = start + n - w.c;   // global index of the context's chunk 0
            const int first = (int)(g0 / cpc), last = (int)((g0 + w.nc - 1) / cpc);
            uint32_t* cnt = a.ws_count + last;
            if (*abort_flag) atomicOr(cnt, kPieceAborted);
            // releases this CTA's record (ordered before by the barrier) and
            // acquires those of the pieces counted before it
            const uint32_t now = atom_add_acq_rel_gpu(cnt, 1u) + 1u;
            if ((now & ~kPieceAborted) == (uint32_t)(last - first + 1)) {
              *cnt = 0u;         // every piece is in: ready for the next call
              if (!(now & kPieceAborted)) {
                int* pm = ctrl + kCtrlMerges;
                const int k = pm[0]++;
                pm[1 + 4 * k] = w.i;
                pm[2 + 4 * k] = w.g;
                pm[3 + 4 * k] = (int)(g0 - start);
                pm[4 + 4 * k] = w.nc;
              }
            }
          }
        }
        first_seg = false;
      }
    }
    if (++st == S) {
      st = 0;
      ph ^= 1u;
    }
    walk_advance(w, a, s_len);
  }
  if constexpr (kMode != kModeGather) {
    // the merges this CTA owes (at most two: its first and its last segment
    // are the only ones that can be pieces); a CTA that gave up merges nothing.
    // Thread 0 decides for all, so that every thread takes the same barriers.
    if (tid == 0 && *abort_flag) ctrl[kCtrlMerges] = 0;
    asm volatile("bar.sync 1, %0;" ::"r"(kCWarps * 32) : "memory");
    const int* pm = ctrl + kCtrlMerges;
    const int owed = pm[0];
    for (int k = 0; k < owed; ++k)
      merge_split<D, kBF16, (kMode == kModeMma && !kF8) ? 2 : 1>(
          a.out, a.ws_rec, a.Hq, a.HG * a.G, pm[1 + 4 * k], pm[2 + 4 * k], start + pm[3 + 4 * k],
          pm[4 + 4 * k], cpc, reinterpret_cast<float*>(gbase));
  }
}

}  // namespace pa
