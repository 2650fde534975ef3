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
// Transposed products.  With only G query heads per KV head, the m16n8k16
// MMA's 16-row M dimension goes to the tokens and to head_dim, and the query
// heads take its 8-wide N dimension:
//   S^T = K Q^T     (M = 16 tokens, N = 8 heads, K = head_dim)
//   O^T += V^T P^T  (M = 16 head_dim rows, N = 8 heads, K = 16 tokens),
// half the MMAs of putting the query heads on M.  P^T's fragment comes from
// S^T's accumulator by an in-register 8x8 transpose (movmatrix).
//
// Index maps.  A contraction does not depend on the order of its summation
// index, and an output row may be held in any order that the write-out
// undoes, so each lane reads contiguous bytes and no byte transpose is needed:
//  * S^T, k-step s: the MMA's k index 2 tig + e (e = 0, 1) stands for
//    head_dim d = (D/4) tig + 4 s + e, and 2 tig + 8 + e for
//    d = (D/4) tig + 4 s + 2 + e.  Lane (gid, tig) reads bytes
//    [(D/4) tig, (D/4)(tig + 1)) of its K rows; the query fragments take the
//    same d.
//  * O^T, m-tile i: row gid stands for d = (D/8) gid + 2 i and row gid + 8 for
//    d = (D/8) gid + 2 i + 1.  Lane (gid, tig) reads bytes
//    [(D/8) gid, (D/8)(gid + 1)) of V rows 2 tig, 2 tig + 1, 2 tig + 8,
//    2 tig + 9, pairs bytes 2i, 2i + 1 of two rows with one byte select, and
//    ends up holding head_dim [(D/8) gid, (D/8)(gid + 1)) of heads 2 tig and
//    2 tig + 1.
#pragma once

#include "pa_device.cuh"

namespace pa {

// Tokens per warp per chunk of this consumer (the 16-bit consumers take 16).
constexpr int kTileF8 = 32;

template <int D, bool kBF16, bool kSwz, bool kHi>
struct MmaConsumerF8 {
  static constexpr int KS = D / 16;        // k-steps of S^T over head_dim
  static constexpr int MT = D / 16;        // m-tiles of O^T over head_dim
  static constexpr int KB = D / 4;         // K bytes per lane per row
  static constexpr int VB = D / 8;         // V bytes per lane per row
  static constexpr int NH = kHi ? 2 : 1;   // 8-head tiles of N
  static constexpr int kMask = kSwz ? (D == 128 ? 7 : 3) : 0;   // 128- or 64-byte swizzle
  uint32_t qb[NH][KS][2];   // Q^T fragments (the B operand of S^T)
  float o[NH][MT][4];       // O^T accumulators
  float m[NH][2];           // running maximum of heads 8 nh + 2 tig + e (same in a tig's 8 lanes)
  float l[NH][2];           // this lane's share of their running sums
  float vscale = 1.f;

  // query elements (d, d + 1) of row `row` of the query slot (rows q_pitch
  // bytes apart), as f16x2
  __device__ __forceinline__ static uint32_t q_pair(uint32_t qslot, int row, int d) {
    uint32_t w;
    asm volatile("ld.shared.b32 %0, [%1];"
                 : "=r"(w)
                 : "r"(qslot + (uint32_t)(row * q_pitch<D>() + d * 2)));
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
    for (int nh = 0; nh < NH; ++nh) {
      const int h = 8 * nh + gid;
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int d0 = KB * tig + 4 * s;
        qb[nh][s][0] = h < G ? q_pair(qslot, h, d0) : 0u;
        qb[nh][s][1] = h < G ? q_pair(qslot, h, d0 + 2) : 0u;
      }
#pragma unroll
      for (int i = 0; i < MT; ++i) o[nh][i][0] = o[nh][i][1] = o[nh][i][2] = o[nh][i][3] = 0.f;
      m[nh][0] = m[nh][1] = -INFINITY;
      l[nh][0] = l[nh][1] = 0.f;
    }
  }

  // 32 tokens [tile0, tile0 + 32) of the chunk; tokens [lo, nv) of them are
  // valid, lo < nv (the codes of the others may be anything, NaN codes
  // included: their scores are masked and their V bytes cleared before
  // conversion).
  __device__ __forceinline__ void tile(uint32_t kpart, uint32_t vpart, int tile0, int lo, int nv,
                                       const DecodeArgs& a, float sl2) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    // ---- S^T = K Q^T: m-tile mt holds tokens 16 mt + gid (rows gid) and
    // 16 mt + 8 + gid (rows gid + 8)
    float s[2][NH][4];
    {
      uint32_t kw[4][KB / 4];   // K bytes of tokens 8 r + gid
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t row = row_addr(kpart, tile0 + 8 * r + gid, 0, a) + (uint32_t)(KB * tig);
#pragma unroll
        for (int c = 0; c < KB / 16; ++c) {
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(kw[r][4 * c]), "=r"(kw[r][4 * c + 1]), "=r"(kw[r][4 * c + 2]),
                         "=r"(kw[r][4 * c + 3])
                       : "r"(swz16<kMask>(row + 16u * c)));
        }
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[mt][nh][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(kw[2 * mt][ks], a0, a2);
          e4m3x4_to_f16x2x2(kw[2 * mt + 1][ks], a1, a3);
#pragma unroll
          for (int nh = 0; nh < NH; ++nh)
            mma_16816<false>(s[mt][nh], a0, a1, a2, a3, qb[nh][ks][0], qb[nh][ks][1]);
        }
    }
    // ---- online softmax per head column (heads 8 nh + 2 tig + e): the 8
    // lanes of a tig share a head and reduce its maximum by shuffles.  The B
    // fragment of P^T for PV k-step kk is the transpose of m-tile kk's packed
    // weights.  Token lo of the tile is valid, so every maximum is finite.
    uint32_t pb[2][NH][2];
#pragma unroll
    for (int nh = 0; nh < NH; ++nh) {
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 16 * mt + gid + ((e >> 1) << 3);
          const float x = s[mt][nh][e] * sl2;
          s[mt][nh][e] = (t >= lo && t < nv) ? x : -INFINITY;
          mx[e & 1] = fmaxf(mx[e & 1], s[mt][nh][e]);
        }
      float alpha[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 4));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
        const float mn = fmaxf(m[nh][e], mx[e]);
        alpha[e] = exp2f(m[nh][e] - mn);
        m[nh][e] = mn;
      }
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        uint32_t pk[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {   // rows gid (hh = 0) and gid + 8 (hh = 1)
          pk[hh] = pack2<false>(exp2f(s[mt][nh][2 * hh] - m[nh][0]),
                                exp2f(s[mt][nh][2 * hh + 1] - m[nh][1]));
          const float2 f = unpack2<false>(pk[hh]);
          sum0 += f.x;
          sum1 += f.y;
        }
        pb[mt][nh][0] = movmatrix_trans(pk[0]);   // tokens 2 tig, 2 tig + 1 of head gid
        pb[mt][nh][1] = movmatrix_trans(pk[1]);   // tokens 2 tig + 8, 2 tig + 9
      }
      l[nh][0] = l[nh][0] * alpha[0] + sum0;
      l[nh][1] = l[nh][1] * alpha[1] + sum1;
      // once the running maximum settles, alpha is exactly 1 in every lane
      // and the rescale is skipped (multiplying by 1 changes nothing)
      if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          o[nh][i][0] *= alpha[0];
          o[nh][i][1] *= alpha[1];
          o[nh][i][2] *= alpha[0];
          o[nh][i][3] *= alpha[1];
        }
      }
    }
    // ---- O^T += V^T P^T, two k-steps of 16 tokens; m-tile i takes bytes 2i
    // and 2i + 1 of V rows (2 tig, 2 tig + 1) and of rows (2 tig + 8,
    // 2 tig + 9)
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t vw[4][VB / 4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int t = 16 * kk + 2 * tig + (r & 1) + ((r >> 1) << 3);
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
        if (t < lo || t >= nv) {
#pragma unroll
          for (int w = 0; w < VB / 4; ++w) vw[r][w] = 0u;
        }
      }
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const int w = i >> 1, q = (i & 1) * 2;
        const uint32_t sel = (uint32_t)(q | ((4 + q) << 4) | ((q + 1) << 8) | ((5 + q) << 12));
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(prmt(vw[0][w], vw[1][w], sel), a0, a1);
        e4m3x4_to_f16x2x2(prmt(vw[2][w], vw[3][w], sel), a2, a3);
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
          mma_16816<false>(o[nh][i], a0, a1, a2, a3, pb[kk][nh][0], pb[kk][nh][1]);
      }
    }
  }

  // the full sum of head (8 nh + 2 tig + e) over the 8 lanes that share it
  __device__ __forceinline__ float total_l(int nh, int e) const {
    float lt = l[nh][e];
    lt += __shfl_xor_sync(0xffffffffu, lt, 4);
    lt += __shfl_xor_sync(0xffffffffu, lt, 8);
    lt += __shfl_xor_sync(0xffffffffu, lt, 16);
    return lt;
  }

  // this lane's head_dim slice [VB gid, VB gid + VB) of head column e of head
  // tile nh, times mul, as fp32
  __device__ __forceinline__ void store_slice_f32(float* dst, int nh, int e, float mul) const {
#pragma unroll
    for (int i = 0; i < MT; i += 2)
      *reinterpret_cast<float4*>(dst + 2 * i) =
          make_float4(o[nh][i][e] * mul, o[nh][i][2 + e] * mul, o[nh][i + 1][e] * mul,
                      o[nh][i + 1][2 + e] * mul);
  }

  // Write this warp's (m, l, o) rows into its merge slot: ml[2][16], o[16][D].
  __device__ __forceinline__ void store(float* slot, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float lt = total_l(nh, e);
        const int row = 8 * nh + 2 * tig + e;
        if (row < G) {
          if (gid == 0) {
            slot[row] = m[nh][e];
            slot[16 + row] = lt;
          }
          store_slice_f32(slot + 32 + row * D + VB * gid, nh, e, vscale);
        }
      }
  }

  // A warp that holds a whole head's segment writes it directly: the output
  // rows (full context) or the partial state record (rows rec_row0 ..).
  __device__ __forceinline__ void write_direct(uint16_t* out_rows, float* rec, int rec_row0,
                                               int rec_rows, bool full, int G) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float lt = total_l(nh, e);
        const int row = 8 * nh + 2 * tig + e;
        if (row >= G) continue;
        if (full) {
          const float mul = vscale / lt;
          uint16_t* dst = out_rows + (size_t)row * D + VB * gid;
#pragma unroll
          for (int i = 0; i < MT; i += 4) {
            uint4 pk;
            pk.x = pack2<kBF16>(o[nh][i][e] * mul, o[nh][i][2 + e] * mul);
            pk.y = pack2<kBF16>(o[nh][i + 1][e] * mul, o[nh][i + 1][2 + e] * mul);
            pk.z = pack2<kBF16>(o[nh][i + 2][e] * mul, o[nh][i + 2][2 + e] * mul);
            pk.w = pack2<kBF16>(o[nh][i + 3][e] * mul, o[nh][i + 3][2 + e] * mul);
            *reinterpret_cast<uint4*>(dst + 2 * i) = pk;
          }
        } else {
          const int r = rec_row0 + row;
          if (gid == 0) {
            rec[(size_t)rec_rows * D + r] = m[nh][e];
            rec[(size_t)rec_rows * D + rec_rows + r] = lt;
          }
          store_slice_f32(rec + (size_t)r * D + VB * gid, nh, e, vscale);
        }
      }
  }
};

}  // namespace pa
