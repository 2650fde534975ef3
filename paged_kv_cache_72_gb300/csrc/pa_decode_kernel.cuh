// Paged single-query decode attention for sm_103a.
//
// What it computes ("vLLM Framework and Inference Engine Design", section
// "What is the essence of vLLM's PagedAttention?"): for every sequence i and
// query head hq, softmax(scale * q . K^T) . V over the first seq_lens[i] tokens,
// where token t lives in physical block block_table[i][t / B], row t % B, of a
// per-layer pool [num_blocks][B][H_kv][D].  Query head hq reads KV head hq / G.
//
// Design (one GPU, persistent, HBM-bound):
//  * Work is the flattened list of 64-token chunks over (sequence, KV head),
//    split into equal contiguous ranges, one per CTA (grid = a multiple of the
//    SM count).  Every CTA scans seq_lens once to find its range; a sequence's
//    context may therefore be split across CTAs, whose partial softmax states
//    (m, l, o) a second kernel merges.  The split depends only on seq_lens, so
//    the result does not depend on block placement.
//  * One producer warp streams each chunk's K and V rows with 5-D TMA tensor
//    copies (one box per physical block or per 64 rows of it) into a ring of
//    shared-memory stages guarded by mbarriers, reading the block table one
//    chunk ahead.  The G query rows of the chunk's KV head come along by a 1-D
//    bulk copy whenever a new (sequence, head) segment starts, so the query
//    group shares every K/V byte it loads.
//  * Four consumer warps each take 16 tokens of every chunk and keep their own
//    online-softmax state in fp32; at a segment end they merge through shared
//    memory.  The tensor-core consumer computes S = Q.K^T and O += P.V with
//    m16n8k16 MMAs (query heads on M, tokens / head_dim on N); the CUDA-core
//    consumer (group size 1) uses per-lane head_dim slices and warp shuffles.
//  * Every wait is bounded; a wait that gives up sets PA_DEVERR_TIMEOUT and the
//    CTA runs to its end without touching the pipeline again.
#pragma once

#include <type_traits>

#include "pa_device.cuh"

namespace pa {

constexpr int kChunk = 64;     // tokens per pipeline stage
constexpr int kTile = 16;      // tokens per consumer warp per stage
constexpr int kCWarps = kChunk / kTile;
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr int kProducerWarp = kCWarps;

enum Mode : int { kModeSimt = 0, kModeMma = 1, kModeGather = 2 };

struct DecodeArgs {
  const uint16_t* q;         // [N][Hq][D]
  uint16_t* out;             // [N][Hq][D]
  const int32_t* bt;         // [N][stride]
  const int32_t* seq_lens;   // [N]
  float* ws_rec;             // [grid][2][G][D + 2]: m[G], l[G], o[G][D]
  int* ws_meta;              // [grid][8]: needs, i, h, seg_start, cpc
  int32_t* err;
  const int64_t* out_off;    // gather: first output row of each sequence
  uint16_t* k_out;           // gather outputs [rows][H_kv][D]
  uint16_t* v_out;
  long long num_blocks;
  int num_seqs, stride, Hq, Hkv, G, B, log2B, R, log2R, nsb;
  int stages;
  float scale_log2;          // scale * log2(e)
  int split_rows;            // 1: box rows stored as [D/64][R][64]; 0: as [R][D]
  int hi_log2;               // log2 byte stride between the two 64-element halves of a row
  int r_log2;                // log2 byte stride between rows of a box
  int kv_bytes;              // bytes of one K (or V) stage part: 64 * D * 2
  int stage_bytes;           // K part + V part + Q part (multiple of 1024)
  int merge_off;             // byte offset of the merge buffer
  int ctrl_off;              // byte offset of barriers and control words
};

// Clamped length: invalid lengths count as 0 tokens.
__device__ __forceinline__ int clamp_len(int T, int stride, int B) {
  return (T < 0 || (long long)T > (long long)stride * B) ? 0 : T;
}

struct Walk {
  int i, h, c, nc, T;
};

__device__ __forceinline__ void walk_load_seq(Walk& w, const DecodeArgs& a) {
  w.T = clamp_len(__ldg(a.seq_lens + w.i), a.stride, a.B);
  w.nc = (w.T + kChunk - 1) / kChunk;
}

__device__ __forceinline__ void walk_advance(Walk& w, const DecodeArgs& a) {
  if (++w.c < w.nc) return;
  w.c = 0;
  if (++w.h < a.Hkv) return;
  w.h = 0;
  do {
    ++w.i;
    if (w.i >= a.num_seqs) { w.nc = 0; w.T = 0; return; }
    walk_load_seq(w, a);
  } while (w.nc == 0);
}

// Block-wide inclusive scan of one int per thread (kThreads threads).
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

// Address of row `tt` (0..63 within the chunk), half `hi` of a stage part.
// One TMA box holds R rows of D elements; boxes follow each other.  Inside a
// box a row's two 64-element halves are either adjacent (r stride D*2, half
// stride 128) or split into two [R][64] planes (r stride 128, half stride
// R*128), which makes 8 consecutive rows hit 8 distinct swizzle phases.
template <int D>
__device__ __forceinline__ uint32_t row_addr(uint32_t part, int tt, int hi, int log2R, int hi_log2,
                                             int r_log2) {
  const int sub = tt >> log2R;
  const int r = tt & ((1 << log2R) - 1);
  return part + ((uint32_t)sub << (log2R + (D == 128 ? 8 : 7))) + ((uint32_t)hi << hi_log2) +
         ((uint32_t)r << r_log2);
}

template <bool kSwz>
__device__ __forceinline__ uint32_t chunk_addr(uint32_t row, int j) {
  // 128-byte swizzle: the 16-byte chunk index is XOR-ed with address bits 7..9
  const int s = kSwz ? (int)((row >> 7) & 7) : 0;
  return row + ((uint32_t)(j ^ s) << 4);
}

// ---------------------------------------------------------------------------
// Consumer state and tile math: tensor-core path
// ---------------------------------------------------------------------------
template <int D, bool kBF16, bool kSwz, bool kHi>
struct MmaConsumer {
  static constexpr int KS = D / 16;   // k-steps of QK
  static constexpr int NT = D / 8;    // n-tiles of PV
  uint32_t qa[KS][4];
  float o[NT][4];
  float m[2], l[2];

  __device__ __forceinline__ void begin(uint32_t qslot, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int d0 = ks * 16 + 2 * tig;
      uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
      if (gid < G) {
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a0) : "r"(qslot + (gid * D + d0) * 2));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a2) : "r"(qslot + (gid * D + d0 + 8) * 2));
      }
      if (kHi && gid + 8 < G) {
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a1) : "r"(qslot + ((gid + 8) * D + d0) * 2));
        asm volatile("ld.shared.b32 %0, [%1];"
                     : "=r"(a3)
                     : "r"(qslot + ((gid + 8) * D + d0 + 8) * 2));
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

  // 16 tokens [tile0, tile0 + 16) of the stage; `nv` of them are valid.
  __device__ __forceinline__ void tile(uint32_t kpart, uint32_t vpart, int tile0, int nv,
                                       int log2R, int hil, int rl, float sl2) {
    const int lane = threadIdx.x & 31, tig = lane & 3;
    if (nv < kTile) {
      // rows past the end of the sequence may hold anything (NaN included):
      // zero them in V so that 0 * garbage cannot reach the accumulator
      const int nbad = kTile - nv;
      for (int e = lane; e < nbad * (D / 8); e += 32) {
        const int rr = tile0 + nv + e / (D / 8);
        const int cj = e % (D / 8);
        const uint32_t ra = row_addr<D>(vpart, rr, cj >> 3, log2R, hil, rl);
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(ra + ((cj & 7) << 4)),
                     "r"(0)
                     : "memory");
      }
      __syncwarp();
    }
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
        const uint32_t ra = row_addr<D>(kpart, tt, cidx >> 3, log2R, hil, rl);
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
    // online softmax, in the log2 domain, per query-head row
    uint32_t pa[4];
#pragma unroll
    for (int hr = 0; hr < (kHi ? 2 : 1); ++hr) {
      float v[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = nt * 8 + 2 * tig + e;
          const float x = s[nt][hr * 2 + e] * sl2;
          v[nt * 2 + e] = (t < nv) ? x : -INFINITY;
        }
      float mt = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      const float mn = fmaxf(m[hr], mt);
      const float alpha = exp2f(m[hr] - mn);
      m[hr] = mn;
      const uint32_t p01 = pack2<kBF16>(exp2f(v[0] - mn), exp2f(v[1] - mn));
      const uint32_t p23 = pack2<kBF16>(exp2f(v[2] - mn), exp2f(v[3] - mn));
      const float2 f01 = unpack2<kBF16>(p01), f23 = unpack2<kBF16>(p23);
      l[hr] = l[hr] * alpha + ((f01.x + f01.y) + (f23.x + f23.y));
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][hr * 2 + 0] *= alpha;
        o[n][hr * 2 + 1] *= alpha;
      }
      pa[hr] = p01;       // row gid (+8): tokens 2tig, 2tig+1
      pa[hr + 2] = p23;   // tokens 8 + 2tig, 9 + 2tig
    }
    if (!kHi) { pa[1] = 0u; pa[3] = 0u; }
    // O += P . V : pairs of n-tiles of 8 head_dim columns; fragments first
    uint32_t vb[D / 16][4];
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      const int mat = lane >> 3;
      const int tt = tile0 + ((mat & 1) << 3) + (lane & 7);
      const int cidx = 2 * j + (mat >> 1);
      const uint32_t ra = row_addr<D>(vpart, tt, cidx >> 3, log2R, hil, rl);
      ldmatrix_x4_trans(chunk_addr<kSwz>(ra, cidx & 7), vb[j][0], vb[j][1], vb[j][2], vb[j][3]);
    }
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      mma_16816<kBF16>(o[2 * j], pa[0], pa[1], pa[2], pa[3], vb[j][0], vb[j][1]);
      mma_16816<kBF16>(o[2 * j + 1], pa[0], pa[1], pa[2], pa[3], vb[j][2], vb[j][3]);
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
};

// ---------------------------------------------------------------------------
// Consumer state and tile math: CUDA-core path (group size 1)
// ---------------------------------------------------------------------------
template <int D, bool kBF16>
struct SimtConsumer {
  static constexpr int VEC = D / 32;   // head_dim elements per lane
  float qf[VEC];
  float o[VEC];
  float m, l;

  __device__ __forceinline__ int col() const { return (threadIdx.x & 31) * VEC; }

  __device__ __forceinline__ void load_row(uint32_t part, int tt, int log2R, int hil, int rl,
                                           float* x) const {
    const int c = col();
    const uint32_t ra = row_addr<D>(part, tt, c >> 6, log2R, hil, rl) + (uint32_t)((c & 63) * 2);
    if constexpr (VEC == 4) {
      uint32_t w0, w1;
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(ra));
      const float2 a = unpack2<kBF16>(w0), b = unpack2<kBF16>(w1);
      x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    } else {
      uint32_t w0;
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w0) : "r"(ra));
      const float2 a = unpack2<kBF16>(w0);
      x[0] = a.x; x[1] = a.y;
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

  __device__ __forceinline__ void tile(uint32_t kpart, uint32_t vpart, int tile0, int nv,
                                       int log2R, int hil, int rl, float sl2) {
    const int lane = threadIdx.x & 31;
    // partial dot products of the 16 tokens over this lane's head_dim slice
    float part[kTile];
#pragma unroll
    for (int t = 0; t < kTile; ++t) {
      float x[VEC];
      load_row(kpart, tile0 + t, log2R, hil, rl, x);
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
    sc = (my_t < nv) ? sc * sl2 : -INFINITY;
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
    if (nv == kTile) {
#pragma unroll
      for (int t = 0; t < kTile; ++t) {
        const float pt = __shfl_sync(0xffffffffu, p, 2 * t);
        float x[VEC];
        load_row(vpart, tile0 + t, log2R, hil, rl, x);
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = fmaf(pt, x[v], o[v]);
      }
    } else {
      for (int t = 0; t < nv; ++t) {
        const float pt = __shfl_sync(0xffffffffu, p, 2 * t);
        float x[VEC];
        load_row(vpart, tile0 + t, log2R, hil, rl, x);
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = fmaf(pt, x[v], o[v]);
      }
    }
  }

  __device__ __forceinline__ void store(float* slot, int /*G*/) {
    const int lane = threadIdx.x & 31;
    float lt = l;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
    if (lane == 0) {
      slot[0] = m;
      slot[16] = lt;
    }
    float* orow = slot + 32;
#pragma unroll
    for (int v = 0; v < VEC; ++v) orow[col() + v] = o[v];
  }
};

// ---------------------------------------------------------------------------
// Segment merge across the consumer warps and the output / partial write.
// ---------------------------------------------------------------------------
template <int D, bool kBF16>
__device__ __forceinline__ void merge_and_write(const DecodeArgs& a, const float* mbuf, int i,
                                                int h, bool full, int slot_idx) {
  const int G = a.G;
  const int slot_floats = 32 + G * D;
  const int tid = threadIdx.x;  // 0..127 (consumer warps)
  float* rec = a.ws_rec + ((size_t)blockIdx.x * 2 + slot_idx) * (size_t)G * (D + 2);
  for (int e = tid; e < G * (D / 2); e += kCWarps * 32) {
    const int g = e / (D / 2);
    const int d = 2 * (e % (D / 2));
    float mw[kCWarps];
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCWarps; ++w) {
      mw[w] = mbuf[w * slot_floats + g];
      mx = fmaxf(mx, mw[w]);
    }
    float L = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < kCWarps; ++w) {
      const float wt = (mw[w] == -INFINITY) ? 0.f : exp2f(mw[w] - mx);
      const float* sw = mbuf + w * slot_floats;
      const float2 ov = *reinterpret_cast<const float2*>(sw + 32 + g * D + d);
      L = fmaf(wt, sw[16 + g], L);
      o0 = fmaf(wt, ov.x, o0);
      o1 = fmaf(wt, ov.y, o1);
    }
    if (full) {
      const float inv = 1.f / L;
      const uint32_t packed = pack2<kBF16>(o0 * inv, o1 * inv);
      uint16_t* dst = a.out + ((size_t)i * a.Hq + (size_t)h * G + g) * D + d;
      *reinterpret_cast<uint32_t*>(dst) = packed;
    } else {
      *reinterpret_cast<float2*>(rec + 2 * G + g * D + d) = make_float2(o0, o1);
      if (d == 0) {
        rec[g] = mx;
        rec[G + g] = L;
      }
    }
  }
}

// Gather mode: copy the valid rows of this warp's 16-token tile to the
// contiguous outputs, undoing the shared-memory layout.
template <int D, bool kSwz>
__device__ __forceinline__ void gather_tile(const DecodeArgs& a, uint32_t kpart, uint32_t vpart,
                                            int tile0, int nv, int i, int h, int c) {
  const int lane = threadIdx.x & 31;
  const long long row0 = __ldg(a.out_off + i) + (long long)c * kChunk + tile0;
  for (int e = lane; e < nv * (D / 8); e += 32) {
    const int r = e / (D / 8);
    const int cj = e % (D / 8);
    const uint32_t ka = chunk_addr<kSwz>(
        row_addr<D>(kpart, tile0 + r, cj >> 3, a.log2R, a.hi_log2, a.r_log2), cj & 7);
    const uint32_t va = chunk_addr<kSwz>(
        row_addr<D>(vpart, tile0 + r, cj >> 3, a.log2R, a.hi_log2, a.r_log2), cj & 7);
    uint4 kv, vv;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(kv.x), "=r"(kv.y), "=r"(kv.z), "=r"(kv.w)
                 : "r"(ka));
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(vv.x), "=r"(vv.y), "=r"(vv.z), "=r"(vv.w)
                 : "r"(va));
    const size_t off = (((size_t)(row0 + r) * a.Hkv + h) * D) + cj * 8;
    *reinterpret_cast<uint4*>(a.k_out + off) = kv;
    *reinterpret_cast<uint4*>(a.v_out + off) = vv;
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int D, bool kBF16, int kMode, bool kSwz, bool kHi>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (128-byte swizzled TMA boxes need it)
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.stages;
  const uint32_t bar_full = base + a.ctrl_off;      // S x 8 bytes
  const uint32_t bar_empty = bar_full + 8 * S;      // S x 8 bytes
  long long* const scan_tmp = reinterpret_cast<long long*>(gbase + a.ctrl_off + 16 * S);
  int* const ctrl = reinterpret_cast<int*>(gbase + a.ctrl_off + 16 * S + 8 * 8);
  volatile int* const abort_flag = ctrl + 4;

  if (tid == 0) {
    ctrl[0] = -1;
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kCWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }

  // ---- find this CTA's range of chunks -------------------------------------
  // The work is the list of 64-token chunks over (sequence, KV head), in
  // sequence-major, then head, then chunk order, cut into equal contiguous
  // ranges of cpc chunks.  One pass: each thread sums the chunks of a
  // contiguous run of sequences, one block-wide scan gives every run's offset,
  // and the thread whose run holds this CTA's first chunk locates it.
  const int per = (a.num_seqs + kThreads - 1) / kThreads;
  const int run0 = min(a.num_seqs, tid * per), run1 = min(a.num_seqs, run0 + per);
  long long my_nc = 0;
  for (int i = run0; i < run1; ++i) {
    const int T0 = __ldg(a.seq_lens + i);
    const int T = clamp_len(T0, a.stride, a.B);
    my_nc += (T + kChunk - 1) / kChunk;
    if ((i % gridDim.x) == blockIdx.x) {
      if (T != T0) set_error(a.err, PA_DEVERR_SEQ_LEN);
      if (kMode != kModeGather && T == 0) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + (size_t)i * a.Hq * D);
        for (int e = 0; e < a.Hq * D / 2; ++e) dst[e] = 0u;
      }
    }
  }
  long long total_nc;
  const long long my_excl = block_scan_incl(my_nc, scan_tmp, total_nc) - my_nc;
  const long long U = total_nc * a.Hkv;
  const long long cpc = (U + gridDim.x - 1) / gridDim.x;
  const long long start = (long long)blockIdx.x * cpc;
  const long long end = min(U, start + cpc);
  const int n_chunks = (start < end) ? (int)(end - start) : 0;
  if (n_chunks > 0 && my_nc > 0 && start >= my_excl * a.Hkv && start < (my_excl + my_nc) * a.Hkv) {
    long long off = my_excl * a.Hkv;
    for (int i = run0; i < run1; ++i) {
      const int nc = (clamp_len(__ldg(a.seq_lens + i), a.stride, a.B) + kChunk - 1) / kChunk;
      const long long span = (long long)nc * a.Hkv;
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
  if (kMode != kModeGather && tid == 0) {
    int* meta = a.ws_meta + (size_t)blockIdx.x * 8;
    meta[0] = 0;
    meta[4] = (int)cpc;
  }
  __syncthreads();
  // let the merge kernel (a programmatic dependent launch) get scheduled; it
  // still waits for this whole grid before reading anything
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (n_chunks == 0) return;
  if (ctrl[0] < 0) {   // cannot happen for a consistent scan; never walk blind
    if (tid == 0) set_error(a.err, PA_DEVERR_SEQ_LEN);
    return;
  }

  Walk w0;
  w0.i = ctrl[0];
  w0.h = ctrl[1];
  w0.c = ctrl[2];
  walk_load_seq(w0, a);

  const int qbytes = (kMode == kModeGather) ? 0 : a.G * D * 2;
  const uint32_t box_bytes = (uint32_t)(a.R * D * 2);

  if (warp == kProducerWarp) {
    // ======================= producer =======================
    const uint64_t pol = policy_evict_first();
    Walk w = w0;
    auto load_entry = [&](const Walk& ww) -> int {
      int ent = -1;
      if (lane < a.nsb) {
        const int tok0 = ww.c * kChunk + lane * a.R;
        if (tok0 < ww.T) ent = __ldg(a.bt + (size_t)ww.i * a.stride + (tok0 >> a.log2B));
      }
      return ent;
    };
    int ent = load_entry(w);
    int issued = 0;
    for (int n = 0; n < n_chunks; ++n) {
      const int st = n % S;
      const uint32_t round = (uint32_t)(n / S);
      const bool waited = mbar_wait_bounded(bar_empty + 8 * st, (round & 1u) ^ 1u, abort_flag);
      const bool timed_out = __any_sync(0xffffffffu, !waited);
      if (__any_sync(0xffffffffu, timed_out || *abort_flag != 0)) {
        if (lane == 0) {
          if (timed_out) set_error(a.err, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      const int valid_tok = min(kChunk, w.T - w.c * kChunk);
      const int nvsub = (valid_tok + a.R - 1) >> a.log2R;
      const bool in_sub = lane < nvsub;
      const bool ok = in_sub && ent >= 0 && (long long)ent < a.num_blocks;
      if (in_sub && !ok) set_error(a.err, PA_DEVERR_BLOCK_ID);
      const unsigned okmask = __ballot_sync(0xffffffffu, ok);
      const bool seg_start = (n == 0) || (w.c == 0);
      const uint32_t sbase = base + (uint32_t)st * a.stage_bytes;
      if (lane == 0) {
        const uint32_t tx =
            (uint32_t)__popc(okmask) * box_bytes * 2u + (seg_start ? (uint32_t)qbytes : 0u);
        mbar_arrive_expect_tx(bar_full + 8 * st, tx);
      }
      __syncwarp();
      if (ok) {
        const int row_off = (w.c * kChunk + lane * a.R) & (a.B - 1);
        const uint32_t dk = sbase + (uint32_t)lane * box_bytes;
        if (a.split_rows) {
          tma_load_5d(dk, &tmk, bar_full + 8 * st, 0, row_off, 0, w.h, ent, pol);
          tma_load_5d(dk + a.kv_bytes, &tmv, bar_full + 8 * st, 0, row_off, 0, w.h, ent, pol);
        } else {
          tma_load_5d(dk, &tmk, bar_full + 8 * st, 0, 0, w.h, row_off, ent, pol);
          tma_load_5d(dk + a.kv_bytes, &tmv, bar_full + 8 * st, 0, 0, w.h, row_off, ent, pol);
        }
      }
      if (kMode != kModeGather && lane == 0 && seg_start) {
        const uint16_t* qsrc = a.q + ((size_t)w.i * a.Hq + (size_t)w.h * a.G) * D;
        bulk_load(sbase + 2 * a.kv_bytes, qsrc, (uint32_t)qbytes, bar_full + 8 * st);
      }
      ++issued;
      walk_advance(w, a);
      if (n + 1 < n_chunks) ent = load_entry(w);
    }
    // drain: make sure no TMA write is still in flight into this CTA's shared
    // memory when it exits (only matters after an abort)
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      for (int k = max(0, issued - S); k < issued; ++k) {
        mbar_wait_bounded(bar_full + 8 * (k % S), (uint32_t)(k / S) & 1u, nullptr);
      }
    }
    return;
  }

  // ======================= consumers =======================
  using Consumer = typename std::conditional<kMode == kModeSimt, SimtConsumer<D, kBF16>,
                                             MmaConsumer<D, kBF16, kSwz, kHi>>::type;
  Consumer cs;
  float* const mbuf = reinterpret_cast<float*>(gbase + a.merge_off);
  const int slot_floats = 32 + a.G * D;
  Walk w = w0;
  int seg_c0 = w.c;
  bool first_seg = true;
  const float sl2 = a.scale_log2;
  for (int n = 0; n < n_chunks; ++n) {
    const int st = n % S;
    const uint32_t round = (uint32_t)(n / S);
    if (!*abort_flag) {
      if (!mbar_wait_bounded(bar_full + 8 * st, round & 1u, abort_flag)) {
        if (lane == 0) {
          set_error(a.err, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
      }
    }
    const bool live = !__any_sync(0xffffffffu, *abort_flag != 0);
    const uint32_t sbase = base + (uint32_t)st * a.stage_bytes;
    const uint32_t kpart = sbase, vpart = sbase + a.kv_bytes, qslot = sbase + 2 * a.kv_bytes;
    const bool seg_start = (n == 0) || (w.c == 0);
    if (seg_start) {
      seg_c0 = w.c;
      if constexpr (kMode != kModeGather) {
        if (live) cs.begin(qslot, a.G);
      }
    }
    const int valid_tok = min(kChunk, w.T - w.c * kChunk);
    const int tile0 = warp * kTile;
    const int nv = max(0, min(kTile, valid_tok - tile0));
    if (live && nv > 0) {
      if constexpr (kMode == kModeGather) {
        gather_tile<D, kSwz>(a, kpart, vpart, tile0, nv, w.i, w.h, w.c);
      } else {
        cs.tile(kpart, vpart, tile0, nv, a.log2R, a.hi_log2, a.r_log2, sl2);
      }
    }
    // this stage may be refilled by TMA once every consumer warp is done; the
    // rows a warp zeroed must be ordered before that async-proxy write
    if (kMode == kModeMma && nv > 0 && nv < kTile) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * st);

    const bool seg_end = (n == n_chunks - 1) || (w.c == w.nc - 1);
    if constexpr (kMode != kModeGather) {
      if (seg_end) {
        const bool full = (seg_c0 == 0) && (w.c == w.nc - 1);
        cs.store(mbuf + warp * slot_floats, a.G);
        asm volatile("bar.sync 1, %0;" ::"r"(kCWarps * 32) : "memory");
        merge_and_write<D, kBF16>(a, mbuf, w.i, w.h, full, first_seg ? 0 : 1);
        if (first_seg && seg_c0 > 0 && w.c == w.nc - 1 && tid == 0) {
          // this CTA finishes a (sequence, head) begun by earlier CTAs: the
          // reduce kernel merges its pieces
          int* meta = a.ws_meta + (size_t)blockIdx.x * 8;
          meta[1] = w.i;
          meta[2] = w.h;
          meta[3] = (int)(start - seg_c0);
          meta[0] = 1;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kCWarps * 32) : "memory");
        first_seg = false;
      }
    }
    walk_advance(w, a);
  }
}

// ---------------------------------------------------------------------------
// Merge of split contexts: one block per decode CTA; the CTA that finished a
// split (sequence, head) merges the partial states of every CTA that held a
// piece of it.  out = sum_k 2^(m_k - m*) o_k / sum_k 2^(m_k - m*) l_k.
// ---------------------------------------------------------------------------
template <int D, bool kBF16>
__global__ void __launch_bounds__(128) split_reduce_kernel(const DecodeArgs a) {
  // wait until the decode grid has finished and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int* meta = a.ws_meta + (size_t)blockIdx.x * 8;
  if (meta[0] == 0) return;
  const int i = meta[1], h = meta[2];
  const long long gstart = meta[3];
  const long long cpc = meta[4];
  const int G = a.G;
  const int last = blockIdx.x;
  const int first = (int)(gstart / cpc);
  const size_t rec_floats = (size_t)G * (D + 2);
  for (int e = threadIdx.x; e < G * (D / 2); e += blockDim.x) {
    const int g = e / (D / 2);
    const int d = 2 * (e % (D / 2));
    float mx = -INFINITY;
    for (int k = first; k <= last; ++k) {
      const int slot = (k == first && gstart != (long long)first * cpc) ? 1 : 0;
      const float* rec = a.ws_rec + ((size_t)k * 2 + slot) * rec_floats;
      mx = fmaxf(mx, rec[g]);
    }
    float L = 0.f, o0 = 0.f, o1 = 0.f;
    for (int k = first; k <= last; ++k) {
      const int slot = (k == first && gstart != (long long)first * cpc) ? 1 : 0;
      const float* rec = a.ws_rec + ((size_t)k * 2 + slot) * rec_floats;
      const float wt = exp2f(rec[g] - mx);
      L = fmaf(wt, rec[G + g], L);
      const float2 ov = *reinterpret_cast<const float2*>(rec + 2 * G + g * D + d);
      o0 = fmaf(wt, ov.x, o0);
      o1 = fmaf(wt, ov.y, o1);
    }
    const float inv = 1.f / L;
    uint16_t* dst = a.out + ((size_t)i * a.Hq + (size_t)h * G + g) * D + d;
    *reinterpret_cast<uint32_t*>(dst) = pack2<kBF16>(o0 * inv, o1 * inv);
  }
}

}  // namespace pa
