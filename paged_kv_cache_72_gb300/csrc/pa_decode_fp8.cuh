// Tensor-core consumer of the decode kernel for an E4M3 (FP8) KV cache.
//
// What it computes is the decode of the 16-bit consumers with K and V stored
// as E4M3 codes and one scale per tensor (our reading of the pages' "fp8" KV
// cache, "vLLM Framework and Inference Engine Design", section "How can one
// customize the tokenizer, cache strategy, or scheduler strategy?"):
//   s_t = scale * k_scale * (q . code_K[t]),   o = v_scale * sum_t p_t code_V[t].
// The scales stay outside the products: the host folds k_scale into the
// softmax scale, and v_scale multiplies the output.  K and V bytes are
// converted to binary16 in registers (exact: every E4M3 value is a binary16
// value); queries are converted to binary16 too when the model dtype is
// bfloat16, and the softmax weights are binary16, so every MMA is f16 x f16
// with fp32 accumulation.
//
// Fragment index maps.  A contraction does not depend on the order of its
// summation index, and the output columns may be held in any order that the
// write-out undoes, so each lane reads contiguous bytes and no byte transpose
// is needed:
//  * S = Q K^T, k-step s: the MMA's k index 2 tig + e (e = 0, 1) stands for
//    head_dim d = (D/4) tig + 4 s + e, and 2 tig + 8 + e for
//    d = (D/4) tig + 4 s + 2 + e.  Lane (gid, tig) reads bytes
//    [(D/4) tig, (D/4)(tig + 1)) of K rows gid and gid + 8, and the query
//    fragments take the same d.
//  * O += P V, n-tile j: the MMA's column n stands for d = n (D/8) + j.  Lane
//    (gid, tig) reads bytes [(D/8) gid, (D/8)(gid + 1)) of V rows 2 tig,
//    2 tig + 1, 2 tig + 8, 2 tig + 9, pairs byte j of two rows with one byte
//    select, and holds output columns [(D/4) tig, (D/4)(tig + 1)) of its rows.
#pragma once

#include "pa_device.cuh"

namespace pa {

template <int D, bool kBF16, bool kSwz, bool kHi>
struct MmaConsumerF8 {
  static constexpr int KS = D / 16;   // k-steps of QK
  static constexpr int NT = D / 8;    // n-tiles of PV
  static constexpr int KB = D / 4;    // K bytes per lane per row
  static constexpr int VB = D / 8;    // V bytes per lane per row (== NT)
  static constexpr int kMask = kSwz ? (D == 128 ? 7 : 3) : 0;   // 128- or 64-byte swizzle
  uint32_t qa[KS][4];
  float o[NT][4];
  float m[2], l[2];
  float vscale = 1.f;

  // query elements (d, d + 1) of row `row` of the query slot, as f16x2
  __device__ __forceinline__ static uint32_t q_pair(uint32_t qslot, int row, int d) {
    uint32_t w;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(qslot + (uint32_t)(row * D + d) * 2));
    if constexpr (kBF16) {
      const float2 f = unpack2<true>(w);
      return pack2<false>(f.x, f.y);
    } else {
      return w;
    }
  }

  __device__ __forceinline__ void begin(uint32_t qslot, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      const int d0 = KB * tig + 4 * s;
      uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
      if (gid < G) {
        a0 = q_pair(qslot, gid, d0);
        a2 = q_pair(qslot, gid, d0 + 2);
      }
      if (kHi && gid + 8 < G) {
        a1 = q_pair(qslot, gid + 8, d0);
        a3 = q_pair(qslot, gid + 8, d0 + 2);
      }
      qa[s][0] = a0;
      qa[s][1] = a1;
      qa[s][2] = a2;
      qa[s][3] = a3;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }

  // 16 tokens [tile0, tile0 + 16) of the chunk; `nv` of them are valid (the
  // codes of the others may be anything, NaN codes included: their scores are
  // masked and their V bytes cleared before conversion).
  __device__ __forceinline__ void tile(uint32_t kpart, uint32_t vpart, int tile0, int nv,
                                       const DecodeArgs& a, float sl2) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    // K bytes of tokens gid (n-tile 0) and 8 + gid (n-tile 1)
    uint32_t kw[2][KB / 4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t row = row_addr(kpart, tile0 + nt * 8 + gid, 0, a) + (uint32_t)(KB * tig);
#pragma unroll
      for (int c = 0; c < KB / 16; ++c) {
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(kw[nt][4 * c]), "=r"(kw[nt][4 * c + 1]), "=r"(kw[nt][4 * c + 2]),
                       "=r"(kw[nt][4 * c + 3])
                     : "r"(swz16<kMask>(row + 16u * c)));
      }
    }
    // V bytes of tokens 2tig, 2tig + 1, 2tig + 8, 2tig + 9
    uint32_t vw[4][VB / 4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = 2 * tig + (r & 1) + ((r >> 1) << 3);
      const uint32_t la = row_addr(vpart, tile0 + t, 0, a) + (uint32_t)(VB * gid);
      const uint32_t pa16 = swz16<kMask>(la & ~15u) + (la & 15u);
      if constexpr (VB == 16) {
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(vw[r][0]), "=r"(vw[r][1]), "=r"(vw[r][2]), "=r"(vw[r][3])
                     : "r"(pa16));
      } else {
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                     : "=r"(vw[r][0]), "=r"(vw[r][1])
                     : "r"(pa16));
      }
      if (t >= nv) {
#pragma unroll
        for (int w = 0; w < VB / 4; ++w) vw[r][w] = 0u;
      }
    }
    // S = Q . K^T: four independent accumulation chains (n-tile x k-step parity)
    float s[2][4], s2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = s2[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint32_t w = kw[nt][ks];
        const uint32_t b0 = e4m3x2_to_f16x2(w & 0xffffu);
        const uint32_t b1 = e4m3x2_to_f16x2(w >> 16);
        mma_16816<false>((ks & 1) ? s2[nt] : s[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3],
                         b0, b1);
      }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
    // online softmax in the log2 domain, per query-head row; weights in f16
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
      const uint32_t p01 = pack2<false>(exp2f(v[0] - mn), exp2f(v[1] - mn));
      const uint32_t p23 = pack2<false>(exp2f(v[2] - mn), exp2f(v[3] - mn));
      const float2 f01 = unpack2<false>(p01), f23 = unpack2<false>(p23);
      l[hr] = l[hr] * alpha + ((f01.x + f01.y) + (f23.x + f23.y));
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][hr * 2 + 0] *= alpha;
        o[n][hr * 2 + 1] *= alpha;
      }
      pa[hr] = p01;       // row gid (+8): tokens 2tig, 2tig + 1
      pa[hr + 2] = p23;   // tokens 8 + 2tig, 9 + 2tig
    }
    if (!kHi) {
      pa[1] = 0u;
      pa[3] = 0u;
    }
    // O += P . V: byte j of rows (2tig, 2tig + 1) and of rows (2tig + 8,
    // 2tig + 9) make the two B registers of n-tile j
#pragma unroll
    for (int w = 0; w < VB / 4; ++w) {
#pragma unroll
      for (int q = 0; q < 4; q += 2) {
        const uint32_t sel = (uint32_t)(q | ((4 + q) << 4) | ((q + 1) << 8) | ((5 + q) << 12));
        const uint32_t lo = prmt(vw[0][w], vw[1][w], sel);
        const uint32_t hi = prmt(vw[2][w], vw[3][w], sel);
        const int j = 4 * w + q;
        mma_16816<false>(o[j], pa[0], pa[1], pa[2], pa[3], e4m3x2_to_f16x2(lo & 0xffffu),
                         e4m3x2_to_f16x2(hi & 0xffffu));
        mma_16816<false>(o[j + 1], pa[0], pa[1], pa[2], pa[3], e4m3x2_to_f16x2(lo >> 16),
                         e4m3x2_to_f16x2(hi >> 16));
      }
    }
  }

  // this lane's output columns of row `hr`: [(D/4) tig, (D/4) tig + D/8) from
  // accumulator element 2 hr, the next D/8 from element 2 hr + 1
  __device__ __forceinline__ void store_row_f32(float* orow, int hr, float mul) const {
    const int tig = (threadIdx.x & 31) & 3;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float* dst = orow + (2 * tig + half) * VB;
#pragma unroll
      for (int j = 0; j < NT; j += 4)
        *reinterpret_cast<float4*>(dst + j) =
            make_float4(o[j][2 * hr + half] * mul, o[j + 1][2 * hr + half] * mul,
                        o[j + 2][2 * hr + half] * mul, o[j + 3][2 * hr + half] * mul);
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
        store_row_f32(slot + 32 + row * D, hr, vscale);
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
          const float mul = vscale / lt;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint16_t* dst = out_rows + (size_t)row * D + (2 * tig + half) * VB;
            const int e = 2 * hr + half;
#pragma unroll
            for (int j = 0; j < NT; j += 8) {
              uint4 pk;
              pk.x = pack2<kBF16>(o[j][e] * mul, o[j + 1][e] * mul);
              pk.y = pack2<kBF16>(o[j + 2][e] * mul, o[j + 3][e] * mul);
              pk.z = pack2<kBF16>(o[j + 4][e] * mul, o[j + 5][e] * mul);
              pk.w = pack2<kBF16>(o[j + 6][e] * mul, o[j + 7][e] * mul);
              *reinterpret_cast<uint4*>(dst + j) = pk;
            }
          }
        } else {
          const int r = rec_row0 + row;
          if (tig == 0) {
            rec[(size_t)rec_rows * D + r] = m[hr];
            rec[(size_t)rec_rows * D + rec_rows + r] = lt;
          }
          store_row_f32(rec + (size_t)r * D, hr, vscale);
        }
      }
    }
  }
};

}  // namespace pa
