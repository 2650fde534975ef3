// Multi-query paged attention for chunked prefill (and decode tokens in the
// same batch) on sm_103a.
//
// What it computes ("vLLM Framework and Inference Engine Design", section "How
// does it support prompts of arbitrary length?": a long prompt is processed in
// chunks, run in one batch with other requests' decode tokens; "vLLM
// self-hosted", section "Two phases: prefill and decode"): sequence i brings
// L_i new tokens, already written to the cache at the end of its T_i tokens;
// new token j, at position p = T_i - L_i + j, attends causally to cached tokens
// [0, p] through the block table:
//   out = softmax(scale * q . K[0..p]^T) . V[0..p].
//
// Design (one GPU, persistent, tensor cores):
//  * A work item is (sequence, KV head, tile of BM = 128 / G new tokens): 128
//    query rows (token, head of the KV head's group), so that every K/V byte
//    staged in shared memory serves 128 rows.  Items are handed out by an
//    atomic counter, the later tiles of each sequence (more keys) first.
//  * One producer warp walks an item's keys [0, p_last] in stages of 64 tokens:
//    for each it reads the block table and issues 5-D TMA copies of the K and
//    V boxes of that KV head (a box is R = min(B, 64) rows of one block), and
//    tags the stage with its item, so that the consumers need no other
//    handshake.  Stages are guarded by mbarriers.
//  * Eight consumer warps each own 16 query rows: S = Q . K^T and O += P . V
//    with m16n8k16 MMAs (rows on M), online softmax in fp32, a causal mask per
//    row; a 64-token stage is taken as two halves of 32 tokens, and a half that
//    lies wholly past every row's position is skipped.
//  * Every wait is bounded; a wait that gives up sets PA_DEVERR_TIMEOUT.
#include <string.h>

#include <type_traits>

#include "pa_decode_launch.h"
#include "pa_device.cuh"

namespace pa {
namespace {

constexpr int kPW = 8;                   // consumer warps
constexpr int kPProducer = kPW;
constexpr int kPThreads = (kPW + 1) * 32;
constexpr int kPRows = 16 * kPW;         // query rows per work item
constexpr int kPBN = 64;                 // key tokens per stage
constexpr int kPMaxSeqs = 4096;          // per-sequence item offsets kept in shared memory
constexpr int kPMaxStages = 8;
// Up to this many sequences, the tensor-core kernel numbers its work items
// longest sequence first (a rank per sequence, one thread each).  At 192, the
// ranks' two bytes per sequence still leave room for five 32 KB stages at
// head_dim 128 in 227 KB of shared memory.
constexpr int kTcSortSeqs = 192;

struct PrefillArgs {
  const uint16_t* q;            // [total_q][Hq][D]
  uint16_t* out;                // [total_q][Hq][D]
  const int32_t* bt;            // [N][stride]
  const int32_t* seq_lens;      // [N]: tokens in the cache, the new ones included
  const int32_t* query_start;   // [N + 1]: new tokens of sequence i are q rows [qs[i], qs[i+1])
  uint32_t* ws;                 // [0] next work item, [1] CTAs finished; zero between calls
  int32_t* err;
  long long num_blocks;
  int num_seqs, stride, Hq, Hkv, G, B, log2B, BM, R, log2R, nsb, stages;
  float scale_log2;             // scale * log2(e)
  int sub_log2, hi_log2;        // in a stage part: box j at j << sub_log2, 64-column plane at
                                // hi << hi_log2, row r at r << 7
  int kv_bytes, stage_bytes, ctrl_off;
  int q_off, q_tx;              // tensor-core kernel: query tiles, bytes of one query tile
};

struct Item {
  int i, h, q0, ntok, p0, T, n_kt;   // sequence, KV head, first q row, tokens, first position,
                                     // cached tokens, key stages
};

__device__ __forceinline__ int clamp_seq(int T, int stride, int B) {
  return (T < 0 || (long long)T > (long long)stride * B) ? -1 : T;
}

// Item number -> (sequence, KV head, token tile).  toff[i] = Hkv * (tiles of
// sequences < i); within a sequence the items run over KV heads, then over
// token tiles from the last (most keys) to the first.
__device__ __forceinline__ void decode_item(int item, const int* toff, const PrefillArgs& a,
                                            Item& it) {
  int lo = 0, hi = a.num_seqs;   // the largest i with toff[i] <= item
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (toff[mid] <= item) lo = mid;
    else hi = mid;
  }
  const int i = lo;
  const int tiles = (toff[i + 1] - toff[i]) / a.Hkv;
  const int r = item - toff[i];
  const int qt = tiles - 1 - r % tiles;
  const int L = __ldg(a.query_start + i + 1) - __ldg(a.query_start + i);
  const int T = __ldg(a.seq_lens + i);
  it.i = i;
  it.h = r / tiles;
  it.q0 = __ldg(a.query_start + i) + qt * a.BM;
  it.ntok = min(a.BM, L - qt * a.BM);
  it.p0 = T - L + qt * a.BM;
  it.T = T;
  it.n_kt = (it.p0 + it.ntok - 1) / kPBN + 1;
}

// A work item of the tensor-core kernel: two consecutive token tiles A and B of
// one sequence and KV head, which share the stream of keys (B's keys; A's are a
// prefix of them).  Pair number -> (sequence, KV head, pair).  Sequences are
// numbered in rank order: rank s is sequence perm[s] (longest first), or s
// itself without perm; toff[s] = Hkv * (pairs of ranks < s).  Within a sequence
// the pairs run from the last (most keys) to the first, each over the KV
// heads, so the counter hands out the costliest items first and the short ones
// fill the end of the launch.  Tile B is absent (no tokens) when the sequence
// has an odd number of tiles and this is its first pair.
struct Pair {
  int i, h, q0, ntok_a, ntok_b, p0, T, nkt_a, nkt;   // q0, p0: tile A's first q row and
                                                     // position; stages of A and of the pair
};

__device__ __forceinline__ void decode_pair(int item, const int* toff, const uint16_t* perm,
                                            const PrefillArgs& a, Pair& it) {
  int lo = 0, hi = a.num_seqs;   // the largest rank s with toff[s] <= item
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (toff[mid] <= item) lo = mid;
    else hi = mid;
  }
  const int i = perm ? (int)perm[lo] : lo;
  const int pairs = (toff[lo + 1] - toff[lo]) / a.Hkv;
  const int r = item - toff[lo];
  const int pr = pairs - 1 - r / a.Hkv;
  const int L = __ldg(a.query_start + i + 1) - __ldg(a.query_start + i);
  const int T = __ldg(a.seq_lens + i);
  const int ta = 2 * pr * a.BM;   // tile A's first new token
  it.i = i;
  it.h = r % a.Hkv;
  it.q0 = __ldg(a.query_start + i) + ta;
  it.ntok_a = min(a.BM, L - ta);
  it.ntok_b = max(0, min(a.BM, L - ta - a.BM));
  it.p0 = T - L + ta;
  it.T = T;
  it.nkt_a = (it.p0 + it.ntok_a - 1) / kPBN + 1;
  it.nkt = it.ntok_b > 0 ? (it.p0 + a.BM + it.ntok_b - 1) / kPBN + 1 : it.nkt_a;
}

__device__ __forceinline__ uint32_t stage_row(uint32_t part, int tt, int hi, const PrefillArgs& a) {
  return part + ((uint32_t)(tt >> a.log2R) << a.sub_log2) + ((uint32_t)hi << a.hi_log2) +
         ((uint32_t)(tt & (a.R - 1)) << 7);
}

__device__ __forceinline__ uint32_t swz_chunk(uint32_t row, int j) {
  // 128-byte swizzle: the 16-byte chunk index is XOR-ed with address bits 7..9
  return row + ((uint32_t)(j ^ (int)((row >> 7) & 7)) << 4);
}

// Block-wide exclusive scan of one value per thread (NT threads).
template <int NT>
__device__ __forceinline__ long long scan_excl(long long v, long long* tmp, long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  long long off = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) off += tmp[w];
    total += tmp[w];
  }
  __syncthreads();
  return off + x - v;
}

// Item offsets: each thread sums the items (kTPI token tiles each) of a run of
// sequence ranks, one block scan gives toff[] and the item count.  With perm
// (at most NT sequences), the ranks first order the sequences by length,
// longest first, ties by index: perm[rank] = sequence.  Without it, rank s is
// sequence s.  A sequence whose length lies outside its table, or with more
// new tokens than tokens, ranks last; it is reported and its rows get zeros.
// Ends with a block barrier.
template <int NT, int D, int kTPI>
__device__ __forceinline__ void item_offsets(const PrefillArgs& a, int* toff, long long* scan_tmp,
                                             int* total_items_s, uint16_t* perm = nullptr) {
  const int tid = threadIdx.x;
  if (perm) {
    // one sequence per thread; toff holds the lengths until the ranks are known
    int key = -1;
    if (tid < a.num_seqs) {
      const int L = __ldg(a.query_start + tid + 1) - __ldg(a.query_start + tid);
      const int T = clamp_seq(__ldg(a.seq_lens + tid), a.stride, a.B);
      key = (L >= 0 && T >= 0 && L <= T) ? T : -1;
      toff[tid] = key;
    }
    __syncthreads();
    int rank = 0;
    if (tid < a.num_seqs)
      for (int j = 0; j < a.num_seqs; ++j) {
        const int kj = toff[j];
        rank += (kj > key || (kj == key && j < tid)) ? 1 : 0;
      }
    __syncthreads();
    if (tid < a.num_seqs) perm[rank] = (uint16_t)tid;
    __syncthreads();
  }
  const int per = (a.num_seqs + NT - 1) / NT;
  const int run0 = min(a.num_seqs, tid * per), run1 = min(a.num_seqs, run0 + per);
  long long mine = 0;
  for (int s = run0; s < run1; ++s) {
    const int i = perm ? (int)perm[s] : s;
    const int L = __ldg(a.query_start + i + 1) - __ldg(a.query_start + i);
    const int T = clamp_seq(__ldg(a.seq_lens + i), a.stride, a.B);
    const bool ok = L >= 0 && T >= 0 && L <= T;
    if (ok) mine += (long long)(((L + a.BM - 1) / a.BM + kTPI - 1) / kTPI) * a.Hkv;
    if ((i % gridDim.x) == blockIdx.x && !ok) {
      // a length outside its table, or more new tokens than tokens: reported,
      // and its rows get zeros
      set_error(a.err, PA_DEVERR_SEQ_LEN);
      if (L > 0) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(
            a.out + (size_t)__ldg(a.query_start + i) * a.Hq * D);
        for (long long e = 0; e < (long long)L * a.Hq * D / 2; ++e) dst[e] = 0u;
      }
    }
  }
  long long total;
  long long off = scan_excl<NT>(mine, scan_tmp, total);
  for (int s = run0; s < run1; ++s) {
    const int i = perm ? (int)perm[s] : s;
    toff[s] = (int)off;
    const int L = __ldg(a.query_start + i + 1) - __ldg(a.query_start + i);
    const int T = clamp_seq(__ldg(a.seq_lens + i), a.stride, a.B);
    if (L >= 0 && T >= 0 && L <= T)
      off += (long long)(((L + a.BM - 1) / a.BM + kTPI - 1) / kTPI) * a.Hkv;
  }
  if (tid == 0) {
    toff[a.num_seqs] = (int)total;
    *total_items_s = (int)total;
  }
  __syncthreads();
}

template <int D, bool kBF16>
__global__ void __launch_bounds__(kPThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.stages;
  const uint32_t bar_full = base + a.ctrl_off;
  const uint32_t bar_empty = bar_full + 8 * S;
  int4* const meta = reinterpret_cast<int4*>(gbase + a.ctrl_off + 16 * S);   // per stage
  int* const toff = reinterpret_cast<int*>(gbase + a.ctrl_off + 32 * S);    // [N + 1]
  long long* const scan_tmp = reinterpret_cast<long long*>(gbase + a.ctrl_off + 32 * S +
                                                           4 * (kPMaxSeqs + 1) + 12);
  volatile int* const abort_flag = reinterpret_cast<int*>(scan_tmp + 16);
  int* const total_items_s = reinterpret_cast<int*>(scan_tmp + 16) + 1;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kPW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kPProducer && lane == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  grid_dep_wait();

  item_offsets<kPThreads, D, 1>(a, toff, scan_tmp, total_items_s);
  if (tid == 0) grid_dep_launch();
  const int total_items = *total_items_s;

  if (warp == kPProducer) {
    // ======================= producer =======================
    const uint64_t pol = policy_evict_first();
    const uint32_t box_bytes = 1u << a.sub_log2;
    int n = 0;   // stages issued so far
    bool stop = false;
    while (!stop) {
      int item = 0;
      if (lane == 0) item = (int)atomicAdd(a.ws, 1u);
      item = __shfl_sync(0xffffffffu, item, 0);
      Item it;
      if (item < total_items) decode_item(item, toff, a, it);
      else stop = true;
      const int n_kt = stop ? 1 : it.n_kt;
      for (int kt = 0; kt < n_kt; ++kt) {
        const int st = n % S;
        const bool waited =
            mbar_wait_bounded(bar_empty + 8 * st, ((uint32_t)(n / S) & 1u) ^ 1u, abort_flag);
        if (__any_sync(0xffffffffu, !waited)) {
          if (lane == 0) {
            set_error(a.err, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
          }
        }
        if (*abort_flag) {   // the consumers leave on the flag
          stop = true;
          break;
        }
        if (stop) {
          // tell the consumers to finish: a stage that carries no item
          if (lane == 0) {
            meta[st] = make_int4(-1, 0, 0, 0);
            mbar_arrive(bar_full + 8 * st);
          }
          break;
        }
        const int tok0 = kt * kPBN + lane * a.R;
        int ent = -1;
        bool ok = false;
        if (lane < a.nsb && tok0 < it.T) {
          ent = __ldg(a.bt + (size_t)it.i * a.stride + (tok0 >> a.log2B));
          ok = ent >= 0 && (long long)ent < a.num_blocks;
          if (!ok) set_error(a.err, PA_DEVERR_BLOCK_ID);
        }
        const unsigned okmask = __ballot_sync(0xffffffffu, ok);
        const uint32_t sbase = base + (uint32_t)st * a.stage_bytes;
        if (lane == 0) {
          meta[st] = make_int4(item, kt, it.n_kt, 0);
          mbar_arrive_expect_tx(bar_full + 8 * st, (uint32_t)__popc(okmask) * box_bytes * 2u);
        }
        __syncwarp();
        if (ok) {
          const uint32_t dk = sbase + (uint32_t)lane * box_bytes;
          const int row_off = tok0 & (a.B - 1);
          tma_load_5d(dk, &tmk, bar_full + 8 * st, 0, row_off, 0, it.h, ent, pol);
          tma_load_5d(dk + a.kv_bytes, &tmv, bar_full + 8 * st, 0, row_off, 0, it.h, ent, pol);
        }
        ++n;
      }
    }
    // after an abort, drain: no TMA write may land in shared memory after the
    // CTA exits (otherwise the consumers waited for every stage issued)
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      for (int k = max(0, n - S); k < n; ++k)
        mbar_wait_bounded(bar_full + 8 * (k % S), (uint32_t)(k / S) & 1u, nullptr);
    }
  } else {
    // ======================= consumers =======================
    constexpr int KS = D / 16, NT = D / 8;
    const int gid = lane >> 2, tig = lane & 3;
    uint32_t qa[KS][4];
    float o[NT][4];
    float m[2], l[2];
    int prow[2];      // positions of this lane's two rows (-1: padding row)
    int pmax = -1;    // the warp's largest row position
    Item it;
    const float sl2 = a.scale_log2;
    int n = 0;
    while (true) {
      const int st = n % S;
      if (!*abort_flag) {
        if (!mbar_wait_bounded(bar_full + 8 * st, (uint32_t)(n / S) & 1u, abort_flag) &&
            lane == 0) {
          set_error(a.err, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int4 md = meta[st];
      if (md.x < 0) break;
      const int kt = md.y;
      if (kt == 0) {
        // a new item: its query rows, as A fragments, straight from global memory
        decode_item(md.x, toff, a, it);
        pmax = -1;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int rr = 16 * warp + gid + 8 * hr;
          const int tok = rr / a.G, g = rr - tok * a.G;
          const bool valid = tok < it.ntok && rr < a.BM * a.G;
          prow[hr] = valid ? it.p0 + tok : -1;
          const uint16_t* qrow =
              a.q + ((size_t)(it.q0 + (valid ? tok : 0)) * a.Hq + (size_t)it.h * a.G + g) * D;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const int d = ks * 16 + 2 * tig;
            qa[ks][hr] = valid ? __ldg(reinterpret_cast<const uint32_t*>(qrow + d)) : 0u;
            qa[ks][hr + 2] = valid ? __ldg(reinterpret_cast<const uint32_t*>(qrow + d + 8)) : 0u;
          }
          m[hr] = -INFINITY;
          l[hr] = 0.f;
        }
        if (16 * warp < min(it.ntok * a.G, a.BM * a.G)) {
          const int last = min(16 * warp + 15, a.BM * a.G - 1) / a.G;   // the warp's last token
          pmax = it.p0 + min(last, it.ntok - 1);
        }   // else every row of the warp is padding: it idles through the item
#pragma unroll
        for (int nn = 0; nn < NT; ++nn) o[nn][0] = o[nn][1] = o[nn][2] = o[nn][3] = 0.f;
      }
      const uint32_t sbase = base + (uint32_t)st * a.stage_bytes;
      const uint32_t kpart = sbase, vpart = sbase + a.kv_bytes;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int tb = kt * kPBN + 32 * hh;   // first key position of this half
        if (tb > pmax) break;                 // wholly past every row of the warp
        // ---- S = Q K^T over 32 keys: four n-tiles of 8
        float s[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int tt = 32 * hh + 8 * nt + (lane & 7);   // key row within the stage
#pragma unroll
          for (int kp = 0; kp < D / 32; ++kp) {
            const int cidx = kp * 4 + (lane >> 3);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(swz_chunk(stage_row(kpart, tt, cidx >> 3, a), cidx & 7), b0, b1, b2, b3);
            mma_16816<kBF16>(s[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3],
                             b0, b1);
            mma_16816<kBF16>(s[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2],
                             qa[2 * kp + 1][3], b2, b3);
          }
        }
        // ---- causal mask and online softmax, rows gid (hr = 0) and gid + 8
        uint32_t pa[2][4];   // A fragments of the two 16-key steps
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int p = prow[hr];
          float v[8];
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int t = tb + 8 * nt + 2 * tig + e;
              // a padding row keeps finite scores against cached keys
              const bool in = p >= 0 ? t <= p : t < it.T;
              v[2 * nt + e] = in ? s[nt][2 * hr + e] * sl2 : -INFINITY;
            }
          float mt = v[0];
#pragma unroll
          for (int k = 1; k < 8; ++k) mt = fmaxf(mt, v[k]);
          mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
          mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
          const float mn = fmaxf(m[hr], mt);
          const float alpha = mn == -INFINITY ? 1.f : exp2f(m[hr] - mn);
          float sum = 0.f;
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            const float p0 = mn == -INFINITY ? 0.f : exp2f(v[2 * nt] - mn);
            const float p1 = mn == -INFINITY ? 0.f : exp2f(v[2 * nt + 1] - mn);
            const uint32_t pk = pack2<kBF16>(p0, p1);
            const float2 f = unpack2<kBF16>(pk);
            sum += f.x + f.y;
            pa[nt >> 1][hr + 2 * (nt & 1)] = pk;
          }
          m[hr] = mn;
          l[hr] = l[hr] * alpha + sum;
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int nn = 0; nn < NT; ++nn) {
              o[nn][2 * hr] *= alpha;
              o[nn][2 * hr + 1] *= alpha;
            }
          }
        }
        // ---- O += P V: two steps of 16 keys; keys at or past T hold no data
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int t0 = tb + 16 * kk;
          const int nv = it.T - t0;   // valid keys in this step (may be <= 0 or >= 16)
          if (nv <= 0) break;
          const uint32_t mlo = (2 * tig < nv ? 0x0000ffffu : 0u) | (2 * tig + 1 < nv ? 0xffff0000u : 0u);
          const uint32_t mhi =
              (8 + 2 * tig < nv ? 0x0000ffffu : 0u) | (9 + 2 * tig < nv ? 0xffff0000u : 0u);
#pragma unroll
          for (int j = 0; j < D / 16; ++j) {
            const int mat = lane >> 3;
            const int tt = 32 * hh + 16 * kk + ((mat & 1) << 3) + (lane & 7);
            const int cidx = 2 * j + (mat >> 1);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(swz_chunk(stage_row(vpart, tt, cidx >> 3, a), cidx & 7), b0, b1,
                              b2, b3);
            if (nv < 16) {
              b0 &= mlo;
              b2 &= mlo;
              b1 &= mhi;
              b3 &= mhi;
            }
            mma_16816<kBF16>(o[2 * j], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
            mma_16816<kBF16>(o[2 * j + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
      if (kt == md.z - 1) {
        // the item's last stage: normalize and write its rows
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          float lt = l[hr];
          lt += __shfl_xor_sync(0xffffffffu, lt, 1);
          lt += __shfl_xor_sync(0xffffffffu, lt, 2);
          if (prow[hr] < 0) continue;
          const int rr = 16 * warp + gid + 8 * hr;
          const int tok = rr / a.G, g = rr - tok * a.G;
          const float inv = 1.f / lt;
          uint16_t* orow = a.out + ((size_t)(it.q0 + tok) * a.Hq + (size_t)it.h * a.G + g) * D;
#pragma unroll
          for (int nn = 0; nn < NT; ++nn)
            *reinterpret_cast<uint32_t*>(orow + nn * 8 + 2 * tig) =
                pack2<kBF16>(o[nn][2 * hr] * inv, o[nn][2 * hr + 1] * inv);
        }
      }
      ++n;
    }
  }
  // ---- the last CTA to finish resets the work counters for the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.ws + 1, 1u) == gridDim.x - 1) {
      a.ws[0] = 0u;
      a.ws[1] = 0u;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Tensor-core (tcgen05) variant.  A work item is a pair of consecutive token
// tiles (A, then B: 128 query rows each) of one sequence and KV head; both
// read the same stream of keys, so every staged K/V byte serves 256 query
// rows, and the tensor core works on one tile while the other's softmax runs.
// Items are numbered longest sequence first (batches of up to kTcSortSeqs
// sequences; see decode_pair), so the short ones fill the end of the launch.
// The contraction runs on the fifth-generation tensor cores with the
// accumulators in tensor memory:
//  * warps 0-3 (softmax of tile A) and 4-7 (tile B): thread r of a warpgroup
//    owns query row r of its tile, which is TMEM lane r.  Per 64-key stage it
//    reads its row of S, masks it, updates the running maximum and sum, and
//    writes its row of P (16-bit) into one of its tile's two P regions of
//    tensor memory.  The maximum used for the exponentials moves only when a
//    row's maximum passes it by more than kTcTau (log2 units): then the row
//    of O is rescaled in TMEM;
//    otherwise P stays below 2^kTcTau and O, l and the stale maximum stay
//    consistent (the result is their quotient).  At the tile's last stage it
//    reads O, divides by l and writes the rows.  Tile A needs at most the
//    pair's stages; its warpgroup skips the others.
//  * warp 8 (producer): items from the atomic counter; per item the two query
//    tiles by TMA (one copy per 64-column plane, [row][128 bytes], 128-byte
//    swizzle); per stage, tagged with the item, the K planes of the item's KV
//    head (one copy per 64-column plane of a block: [plane][key][128 bytes])
//    and its V rows (one copy per block, every plane: [block][plane][row][128
//    bytes]).
//  * warps 9 and 10 (score products, one thread each, one per tile): per
//    stage S = Q . K^T (M 128, N 64, K = head_dim) into the tile's S buffer,
//    once the P region that the stage's P will go to is free again, so that
//    the softmax never waits for it;
//  * warp 11 (one thread, both tiles): per stage and tile O += P . V (M 128,
//    N head_dim, K 64; P from tensor memory, V from shared memory as an
//    MN-major operand) once its P is written.  A tcgen05.mma holds its
//    issuing thread for tens of cycles, and that issue time was the bound on
//    the stage rate with one thread issuing all of a tile's products.
// Tensor memory: tile t's S buffer at columns 256 t .. +63, its P regions
// (64 keys of 16 bits, two to a column) at 256 t + 64 and 256 t + 96, its O at
// 256 t + 128.  Every wait is bounded; a wait that gives up sets
// PA_DEVERR_TIMEOUT and the roles leave.
// ---------------------------------------------------------------------------
// D[tmem] (+)= A . B with A in tensor memory: M rows in lanes 0..M-1, K along
// the columns, two 16-bit elements per 32-bit column (the even one in the low
// half); B from shared memory by its descriptor
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

constexpr int kTcWarps = 12;
constexpr int kTcThreads = kTcWarps * 32;
static_assert(kTcSortSeqs <= kTcThreads, "one thread ranks one sequence");
constexpr int kTcProducer = 8;
constexpr int kTcMma = 9;           // warps 9 and 10: the score-product issuers of tiles A and B
constexpr int kTcPv = 11;           // the P . V issuer of both tiles
// per tile, the queue of P . V records from its score issuer to the P . V
// issuer: a ring of four records, then tail (records pushed), head (records
// issued), and fin (the score issuer has stopped); eight words a tile
constexpr int kTcPvqWords = 16;
constexpr uint32_t kTcTmemCols = 512;
constexpr float kTcTau = 8.f;
constexpr float kTcTauPow = 256.f;   // 2^kTcTau
// barriers (8 bytes each): q full, q empty; per tile 8 slots (s full, s free,
// p full[2], p empty[2], o free, one unused); done[3] (one per issuing thread)
constexpr int kTcBars = 2 + 2 * 8 + 3;

__host__ __device__ constexpr int tc_toff_bytes(int num_seqs) {
  return ((4 * (num_seqs + 1) + 15) / 16) * 16;
}
__host__ __device__ constexpr int tc_perm_bytes(int num_seqs) {
  return num_seqs <= kTcSortSeqs ? ((2 * num_seqs + 15) / 16) * 16 : 0;
}

// shared-memory control area of the tensor-core kernel (after the query tiles):
// full/empty/seen barriers, the other barriers, stage tags (two int4 per
// stage, from a 16-byte boundary), the P . V record queues, TMEM address and
// flags, item offsets, scan scratch, the sequences in rank order
__host__ __device__ constexpr int tc_tags_off(int S) { return (24 * S + 8 * kTcBars + 15) & ~15; }
__host__ __device__ constexpr int tc_ctrl_bytes(int S, int num_seqs) {
  return tc_tags_off(S) + 32 * S + 4 * kTcPvqWords + 16 + tc_toff_bytes(num_seqs) +
         8 * (kTcThreads / 32) + tc_perm_bytes(num_seqs);
}

template <int D, bool kBF16>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv,
                            const __grid_constant__ CUtensorMap tmq, const PrefillArgs a) {
  constexpr int NP = D / 64;          // 64-column planes of a row
  constexpr uint32_t kQPlane = 16384; // 128 rows x 128 bytes
  constexpr uint32_t kKPlane = 8192;  // 64 keys x 128 bytes
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.stages;
  const uint32_t bar_full = base + a.ctrl_off;      // S
  const uint32_t bar_empty = bar_full + 8 * S;      // S
  // S: every softmax warp has read the stage's tag.  A warpgroup skips the
  // stages its tile does not read, so the MMA thread can release them without
  // it; the producer refills a stage only once it is also seen, so that no
  // warpgroup waits on a stage that has already been refilled.
  const uint32_t bar_seen = bar_empty + 8 * S;
  const uint32_t bar_qfull = bar_seen + 8 * S;
  const uint32_t bar_qempty = bar_qfull + 8;
  // tile t's barriers: s full at +0, s free at +16, p full of P region 0 at
  // +32 and of region 1 at +24, p empty of region 0 at +40 and of region 1 at
  // +56, o free at +48.  P full is one barrier per region: a warp may reach
  // stage k + 1 while another of its warpgroup still writes stage k's P (the
  // next scores need only every warp to have read stage k's), so with one
  // barrier its arrival for k + 1 could complete stage k's phase early.  It
  // cannot reach stage k + 2, which waits for the P . V of stage k.
  const uint32_t bar_tile0 = bar_qfull + 16;
  const uint32_t bar_done = bar_tile0 + 128;
  uint8_t* const cgen = gbase + a.ctrl_off + tc_tags_off(S);
  int4* const meta = reinterpret_cast<int4*>(cgen);                         // [S]
  int4* const meta2 = reinterpret_cast<int4*>(cgen + 16 * S);               // [S]
  volatile uint32_t* const pvq = reinterpret_cast<volatile uint32_t*>(cgen + 32 * S);
  uint8_t* const cgen2 = cgen + 32 * S + 4 * kTcPvqWords;
  uint32_t* const tslot = reinterpret_cast<uint32_t*>(cgen2);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  int* const total_items_s = reinterpret_cast<int*>(tslot + 2);
  int* const toff = reinterpret_cast<int*>(cgen2 + 16);                     // [N + 1]
  long long* const scan_tmp =
      reinterpret_cast<long long*>(cgen2 + 16 + tc_toff_bytes(a.num_seqs));
  uint16_t* const perm = a.num_seqs <= kTcSortSeqs
                             ? reinterpret_cast<uint16_t*>(scan_tmp + kTcThreads / 32)
                             : nullptr;   // [N]

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 4);       // per tile: its score issuer's K share, its P . V share
      mbar_init(bar_seen + 8 * s, 8);        // one arrival per softmax warp
    }
    mbar_init(bar_qfull, 1);                 // the producer's expect-tx
    mbar_init(bar_qempty, 2);                // a commit of each MMA issuer
    for (int t = 0; t < 2; ++t) {
      const uint32_t bt = bar_tile0 + 64 * t;
      mbar_init(bt, 1);                      // s full: a commit
      mbar_init(bt + 16, 128);               // s free: the warpgroup's threads
      mbar_init(bt + 32, 128);               // p full, region 0: the warpgroup's threads
      mbar_init(bt + 24, 128);               // p full, region 1
      mbar_init(bt + 40, 1);                 // p empty, region 0: a commit
      mbar_init(bt + 56, 1);                 // p empty, region 1: a commit
      mbar_init(bt + 48, 128);               // o free: the warpgroup's threads
    }
    mbar_init(bar_done, 1);
    mbar_init(bar_done + 8, 1);
    mbar_init(bar_done + 16, 1);
    for (int w = 0; w < kTcPvqWords; ++w) pvq[w] = 0u;
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kTcProducer && lane == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    prefetch_tensormap(&tmq);
  }
  if (warp == kTcMma) {
    tmem_alloc(smem_u32(tslot), kTcTmemCols);
    tc_fence_before();
  }
  grid_dep_wait();
  item_offsets<kTcThreads, D, 2>(a, toff, scan_tmp, total_items_s, perm);   // ends with a barrier
  tc_fence_after();
  if (tid == 0) grid_dep_launch();
  const int total_items = *total_items_s;
  const uint32_t tmem = *tslot;

  // a wait whose outcome is the same in every lane of the warp
  auto wait_warp = [&](uint32_t bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort_flag)) != 0;
  };

  if (warp == kTcProducer) {
    // ======================= producer =======================
    // K and V are read again by the sequence's other token tiles: keep them
    // in L2; a query tile is read once
    const uint64_t pol_kv = policy_evict_last();
    const uint64_t pol_q = policy_evict_first();
    const uint32_t box_bytes = (uint32_t)a.R * 128u;
    int j = 0, n = 0, nq = 0;   // stages issued, items started, query tiles issued
    int jst = 0;                // j % S and the parity of j / S, kept as j advances
    uint32_t jph = 0u;
    bool stop = false;
    while (!stop) {
      int item = 0;
      if (lane == 0) item = (int)atomicAdd(a.ws, 1u);
      item = __shfl_sync(0xffffffffu, item, 0);
      Pair it;
      if (item < total_items) decode_pair(item, toff, perm, a, it);
      else stop = true;
      const int n_kt = stop ? 1 : it.nkt;
      // block-table entries two stages ahead of their copies (lane l < nsb:
      // the block of the stage's l-th box), so that the producer does not
      // wait on each entry's load
      auto load_ent = [&](int kt) -> int {
        const int tok0 = kt * kPBN + lane * a.R;
        return (lane < a.nsb && tok0 < it.T)
                   ? __ldg(a.bt + (size_t)it.i * a.stride + (tok0 >> a.log2B))
                   : -1;
      };
      int e0 = stop ? -1 : load_ent(0);
      int e1 = (stop || n_kt < 2) ? -1 : load_ent(1);
      for (int kt = 0; kt < n_kt; ++kt) {
        const int ent = e0;
        e0 = e1;
        e1 = kt + 2 < n_kt ? load_ent(kt + 2) : -1;
        const int st = jst;
        bool ok_wait = wait_warp(bar_empty + 8 * st, jph ^ 1u) &&
                       wait_warp(bar_seen + 8 * st, jph ^ 1u);
        if (ok_wait && !stop && kt == 0)   // the query tiles' buffers are free
          ok_wait = wait_warp(bar_qempty, ((uint32_t)n & 1u) ^ 1u);
        if (!ok_wait) {
          if (lane == 0 && !*abort_flag) set_error(a.err, PA_DEVERR_TIMEOUT);
          if (lane == 0) *abort_flag = 1;
        }
        __syncwarp();
        if (*abort_flag) {   // the other roles leave on the flag
          stop = true;
          break;
        }
        if (stop) {
          // tell the others to finish: a stage that carries no item
          if (lane == 0) {
            meta[st] = make_int4(-1, 0, 0, 0);
            mbar_arrive(bar_full + 8 * st);
          }
          break;
        }
        if (kt == 0) {
          // tile A's rows into buffer 0, tile B's (if it has tokens) into 1
          const int ntiles = it.ntok_b > 0 ? 2 : 1;
          if (lane == 0) mbar_arrive_expect_tx(bar_qfull, (uint32_t)(a.q_tx * ntiles));
          __syncwarp();
          if (lane < NP * ntiles) {
            const int t = lane / NP, pl = lane % NP;
            tma_load_5d(base + (uint32_t)a.q_off + (uint32_t)(t * NP + pl) * kQPlane, &tmq,
                        bar_qfull, 0, pl, 0, it.h, it.q0 + t * a.BM, pol_q);
          }
          ++nq;
        }
        const int tok0 = kt * kPBN + lane * a.R;
        bool ok = false;
        if (lane < a.nsb && tok0 < it.T) {
          ok = ent >= 0 && (long long)ent < a.num_blocks;
          if (!ok) set_error(a.err, PA_DEVERR_BLOCK_ID);
        }
        const unsigned okmask = __ballot_sync(0xffffffffu, ok);
        if (lane == 0) {
          meta[st] = make_int4(item, kt, it.nkt, n);
          meta2[st] = make_int4(it.nkt_a, it.ntok_b > 0 ? 1 : 0, 0, 0);
          mbar_arrive_expect_tx(bar_full + 8 * st,
                                (uint32_t)__popc(okmask) * box_bytes * (uint32_t)(2 * NP));
        }
        __syncwarp();
        if (ok) {
          const uint32_t kdst = base + (uint32_t)st * a.stage_bytes + (uint32_t)lane * box_bytes;
          const int row_off = tok0 & (a.B - 1);
#pragma unroll
          for (int p = 0; p < NP; ++p)
            tma_load_5d(kdst + (uint32_t)p * kKPlane, &tmk, bar_full + 8 * st, 0, row_off, p, it.h,
                        ent, pol_kv);
          // the block's V rows, every plane, in one box: [plane][row][128 bytes]
          tma_load_5d(base + (uint32_t)st * a.stage_bytes + (uint32_t)a.kv_bytes +
                          (uint32_t)lane * box_bytes * (uint32_t)NP,
                      &tmv, bar_full + 8 * st, 0, row_off, 0, it.h, ent, pol_kv);
        }
        ++j;
        if (++jst == S) {
          jst = 0;
          jph ^= 1u;
        }
      }
      if (!stop) ++n;
    }
    // after an abort, drain: no TMA write may land in shared memory after the
    // CTA exits
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      for (int k = max(0, j - S); k < j; ++k)
        mbar_wait_bounded(bar_full + 8 * (k % S), (uint32_t)(k / S) & 1u, nullptr);
      if (nq > 0) mbar_wait_bounded(bar_qfull, (uint32_t)(nq - 1) & 1u, nullptr);
    }
  } else if (warp == kTcMma || warp == kTcMma + 1) {
    // ======================= score products (one thread per tile) ============
    // Warp 9 issues tile A's score products, warp 10 tile B's; each walks
    // every stage.  An event loop: the next stage's S = Q . K^T as soon as
    // its K/V have landed, the query tile has, and the S buffer's previous
    // scores have been read -- once at most one of the tile's P . V products
    // is pending, so that a P . V is never queued behind score products two
    // stages ahead (the tensor pipe executes in issue order).  Each score
    // product pushes a record for its P . V onto the tile's queue.  A stage
    // takes four arrivals to be released, per tile a K share and a V share:
    // the score issuer commits the K share after its product (at once, with
    // the V share too, where its tile does not read the stage); the query
    // tiles are released by a commit of each score issuer after its last
    // product that reads them.
    const int t = warp - kTcMma;
    if (lane == 0) {
      constexpr uint32_t id_s = umma_idesc_f16(kBF16, 128, kPBN, false);
      // a record of 6 bits: stage slot (bits 0-2), first stage of an item
      // (3), O must be free first (4), the parity of that wait (5)
      static_assert(kPMaxStages <= 8, "stage slots take 3 bits");
      volatile uint32_t* const q = pvq + 8 * t;   // ring[4], tail, head, fin
      int rt = 0;              // records pushed
      int ns = 0;              // score products issued
      int ni = 0;              // items started
      int js = 0;              // next stage to walk
      int sst = 0;             // js % S and the parity of js / S
      uint32_t sph = 0u;
      auto next_stage = [&]() {
        ++js;
        if (++sst == S) {
          sst = 0;
          sph ^= 1u;
        }
      };
      bool ok = true;
      const uint32_t bt = bar_tile0 + 64 * t;
      const uint32_t tcol = tmem + (uint32_t)(256 * t);
      const uint64_t da = umma_desc_sw128(base + (uint32_t)a.q_off + (uint32_t)(t * NP) * kQPlane,
                                          16, 1024);
      long long t_last = clock64();
      while (true) {
        bool progressed = false;
        bool done = false;
        if (rt - (int)q[5] < 2) {
          const int st = sst;
          if (mbar_test(bar_full + 8 * st, sph)) {
            const int4 md = meta[st];
            if (md.x < 0) {
              done = true;
            } else {
              const int4 m2 = meta2[st];
              const int kt = md.y, nkt = md.z, n = md.w;
              const bool act = t == 0 ? kt < m2.x : (m2.y != 0 && kt < nkt);
              if (!act) {
                // keys past this tile's last position: nothing to compute
                umma_commit(bar_empty + 8 * st);
                mbar_arrive(bar_empty + 8 * st);
                if (kt == nkt - 1) umma_commit(bar_qempty);
                next_stage();
                progressed = true;
              } else {
                // the query tile has landed, and the S buffer's previous
                // scores have been read
                bool ready = kt != 0 || mbar_test(bar_qfull, (uint32_t)n & 1u);
                if (ready && ns >= 1) ready = mbar_test(bt + 16, (uint32_t)(ns - 1) & 1u);
                // and the P region these scores' P will go to is free (the
                // P . V two products back has completed), so that the softmax,
                // once it sees the scores, writes P without a wait of its own
                if (ready && ns >= 2)
                  ready = mbar_test(bt + ((ns & 1) ? 56 : 40), (uint32_t)((ns >> 1) - 1) & 1u);
                if (ready) {
                  tc_fence_after();
                  const uint64_t db =
                      umma_desc_sw128(base + (uint32_t)st * a.stage_bytes, 16, 1024);
                  // K steps of 16 columns; within a 64-column plane a step
                  // moves the start 32 bytes (the swizzle is applied to the
                  // address; the descriptors' address field is in 16-byte
                  // units: a step adds its offset / 16 to the base descriptor)
#pragma unroll
                  for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (uint32_t)(ks & 3) * 32u;
                    umma_f16(tcol, da + (((uint32_t)(ks >> 2) * kQPlane + off) >> 4),
                             db + (((uint32_t)(ks >> 2) * kKPlane + off) >> 4), id_s, ks > 0);
                  }
                  umma_commit(bt);
                  umma_commit(bar_empty + 8 * st);   // this tile no longer reads K
                  if (kt == nkt - 1) umma_commit(bar_qempty);   // the query tile is free
                  uint32_t rc = (uint32_t)st;
                  if (kt == 0) {
                    rc |= 8u;
                    if (ni > 0) rc |= 16u | ((uint32_t)((ni - 1) & 1) << 5);
                    ++ni;
                  }
                  q[rt & 3] = rc;
                  __threadfence_block();   // the record before the tail that publishes it
                  q[4] = (uint32_t)(rt + 1);
                  ++rt;
                  ++ns;
                  next_stage();
                  progressed = true;
                }
              }
            }
          }
        }
        if (done) break;
        if (progressed) {
          t_last = clock64();
        } else {
          if (*abort_flag) {
            ok = false;
            break;
          }
          if (clock64() - t_last > kWaitLimitCycles) {
            ok = false;
            break;
          }
          __nanosleep(20);   // leave the issue slots to the softmax warps beside it
        }
      }
      if (!ok) {
        if (!*abort_flag) set_error(a.err, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      __threadfence_block();
      q[6] = 1u;   // no more records
      // every MMA issued has completed before the tensor memory is released
      umma_commit(bar_done + 8 * t);
      mbar_wait_bounded(bar_done + 8 * t, 0u, nullptr);
    }
    __syncwarp();
  } else if (warp == kTcPv) {
    // ======================= P . V products (one thread, both tiles) =========
    // Per tile, the oldest record on its queue: O += P . V once its P is
    // written (and, at an item's first stage, once O has been read out for
    // the tile's item before).  The commits free the P region (the softmax
    // waits on it to reuse the region and to rescale O) and give the stage
    // the tile's V share.
    if (lane == 0) {
      constexpr uint32_t id_o = umma_idesc_f16(kBF16, 128, D, true);
      int rh0 = 0, rh1 = 0;    // records issued, per tile (P . V products)
      bool ok = true;
      long long t_last = clock64();
      // one tile's oldest record, if it can go; returns whether it went
      auto try_pv = [&](int t, int& rh) -> bool {
        volatile uint32_t* const q = pvq + 8 * t;
        if ((int)q[4] == rh) return false;
        __threadfence_block();   // the record after the tail that published it
        const uint32_t rc = q[rh & 3];
        const uint32_t bt = bar_tile0 + 64 * t;
        const int np = rh;
        if (!mbar_test(bt + ((np & 1) ? 24 : 32), (uint32_t)(np >> 1) & 1u)) return false;
        if ((rc & 16u) && !mbar_test(bt + 48, (rc >> 5) & 1u)) return false;
        // P (128 x 64) from the tile's P region np % 2 in tensor memory (16
        // keys = 8 columns per K step), V (64 keys x D, MN-major) from the
        // stage's V part: block b's box at b * vblk, [plane][row][128 bytes],
        // so the 64-column planes are vrow bytes apart (the leading offset)
        // and 8-key groups 1024 bytes apart within a block of 16 or more
        // rows, one block apart at 8 rows (the stride offset).  A K step's
        // 16 keys are rows (16k) % R.. of block (16k) / R.  The tile's first
        // stage of an item overwrites O.
        tc_fence_after();
        const int pst = (int)(rc & 7u);
        const bool first = (rc & 8u) != 0u;
        const uint32_t tcol = tmem + (uint32_t)(256 * t);
        const uint32_t vrow = (uint32_t)a.R * 128u, vblk = vrow * (uint32_t)NP;
        const uint32_t vpart = base + (uint32_t)pst * a.stage_bytes + (uint32_t)a.kv_bytes;
        const uint64_t dv = umma_desc_sw128(vpart, vrow, a.R >= 16 ? 1024u : vblk);
        const uint32_t preg = tcol + 64u + 32u * (uint32_t)(np & 1);
#pragma unroll
        for (int k = 0; k < kPBN / 16; ++k) {
          const uint32_t off = (uint32_t)((16 * k) >> a.log2R) * vblk +
                               (uint32_t)((16 * k) & (a.R - 1)) * 128u;
          umma_f16_tmem_a(tcol + 128u, preg + 8u * k, dv + (off >> 4), id_o, !first || k > 0);
        }
        umma_commit(bt + ((np & 1) ? 56 : 40));  // the P region is free, O updated
        umma_commit(bar_empty + 8 * pst);        // this tile no longer reads V
        ++rh;
        q[5] = (uint32_t)rh;
        return true;
      };
      while (true) {
        bool progressed = try_pv(0, rh0);
        progressed = try_pv(1, rh1) || progressed;
        if (!progressed) {
          // both score issuers have stopped and every record is issued
          if (pvq[6] && pvq[8 + 6]) {
            __threadfence_block();
            if ((int)pvq[4] == rh0 && (int)pvq[8 + 4] == rh1) break;
          }
          if (*abort_flag) {
            ok = false;
            break;
          }
          if (clock64() - t_last > kWaitLimitCycles) {
            ok = false;
            break;
          }
          __nanosleep(20);
        } else {
          t_last = clock64();
        }
      }
      if (!ok) {
        if (!*abort_flag) set_error(a.err, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(bar_done + 16);
      mbar_wait_bounded(bar_done + 16, 0u, nullptr);
    }
    __syncwarp();
  } else {
    // ======================= softmax (warps 0-7) =======================
    const int tile = warp >> 2;          // 0: tile A, 1: tile B
    const int r = tid & 127;             // this thread's query row of the tile, TMEM lane r
    const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(256 * tile);
    const uint32_t bt = bar_tile0 + 64 * tile;
    const float sl2 = a.scale_log2;
    Pair it{};
    int q0 = 0, p0 = 0, nkt_t = 0;   // this tile's first q row, first position, stages
    int prow = -1;         // the row's position (-1: a padding row)
    bool valid = false;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    int jst = 0;           // the ring slot of the next stage to see
    uint32_t jph = 0u;     // the parity of that slot's use
    int nt = 0;            // stages this tile has processed
    while (true) {
      const int st = jst;
      if (!wait_warp(bar_full + 8 * st, jph)) {
        ok = false;
        break;
      }
      const int4 md = meta[st];
      if (md.x < 0) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_seen + 8 * st);   // the tag is read
      const int kt = md.y;
      if (kt == 0) {
        decode_pair(md.x, toff, perm, a, it);
        const int ntok = tile == 0 ? it.ntok_a : it.ntok_b;
        q0 = it.q0 + tile * a.BM;
        p0 = it.p0 + tile * a.BM;
        nkt_t = tile == 0 ? it.nkt_a : (it.ntok_b > 0 ? it.nkt : 0);
        const int tok = r / a.G;
        valid = r < a.BM * a.G && tok < ntok;
        prow = valid ? p0 + tok : -1;
        m_used = -INFINITY;
        l = 0.f;
      }
      if (++jst == S) {
        jst = 0;
        jph ^= 1u;
      }
      if (kt >= nkt_t) continue;   // keys past this tile's last position
      // ---- this row of S
      if (!wait_warp(bt, (uint32_t)nt & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kPBN];
      tmem_ld32(trow, *reinterpret_cast<uint32_t(*)[32]>(sr));
      tmem_ld32(trow + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bt + 16);   // the S buffer may be overwritten
      const int tb = kt * kPBN;
      // ---- P = 2^(s f - mu): one packed FFMA per two scores and one ex2 per
      // score, 16-bit; its row sum in fp32 over the rounded values that O
      // sums (mixed-precision adds of the 16-bit halves), so that a row
      // dominated by one key keeps that key's value
      uint32_t pk[kPBN / 2];
      auto p_pass = [&](float f, float mu) -> float {
        float sum8[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) sum8[c] = 0.f;
#pragma unroll
        for (int c = 0; c < kPBN / 2; ++c) {
          float x0 = __uint_as_float(sr[2 * c]), x1 = __uint_as_float(sr[2 * c + 1]);
          ffma2(x0, x1, f, -mu);
          pk[c] = pack2<kBF16>(ex2_approx(x0), ex2_approx(x1));
          sum8[c & 7] = add_pair16<kBF16>(sum8[c & 7], pk[c]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) sum8[c] += sum8[c + 4];
        return (sum8[0] + sum8[1]) + (sum8[2] + sum8[3]);
      };
      // A stage wholly at or before the tile's first position needs no mask;
      // with a positive scale its scores are used raw, f = scale.  Once the
      // row has a reference maximum, such a stage first computes P against
      // it: every P is at most the stage's sum, so a sum of at most 2^kTcTau
      // shows that the reference stays, and the maximum is not needed.
      const bool raw = tb + kPBN - 1 <= p0 && sl2 > 0.f;
      const bool guess = raw && m_used != -INFINITY;
      float alpha = 1.f, ssum = 0.f;
      if (guess) ssum = p_pass(sl2, m_used);
      if (!guess || !(ssum <= kTcTauPow)) {
        // ---- causal mask (a padding row keeps finite scores against cached
        // keys) and maximum; unmasked stages take it on the raw scores,
        // masked ones scale the scores first (f = 1).  Eight partial maxima:
        // one warp per sub-partition leaves no other warp to hide a 64-long
        // chain of dependent instructions; a three-input max takes two
        // scores at a time.
        float mx8[8], f = 1.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) mx8[c] = -INFINITY;
        if (raw) {
#pragma unroll
          for (int c = 0; c < kPBN / 2; ++c)
            mx8[c & 7] = max3f(mx8[c & 7], __uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1]));
          f = sl2;
        } else {
#pragma unroll
          for (int c = 0; c < kPBN / 2; ++c) {
            float v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int t = tb + 2 * c + u;
              const bool in = prow >= 0 ? t <= prow : t < it.T;
              v[u] = in ? __uint_as_float(sr[2 * c + u]) * sl2 : -INFINITY;
              sr[2 * c + u] = __float_as_uint(v[u]);
            }
            mx8[c & 7] = max3f(mx8[c & 7], v[0], v[1]);
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) mx8[c] = fmaxf(mx8[c], mx8[c + 4]);
        float mx = fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3]));
        if (raw) mx *= sl2;
        bool moved = false;
        if (mx > m_used + kTcTau) {   // the exponentials' reference moves
          if (m_used != -INFINITY) alpha = ex2_approx(m_used - mx);
          m_used = mx;
          moved = true;
        }
        // (no row is masked whole at kt 0)
        if (!guess || moved) ssum = p_pass(f, m_used == -INFINITY ? 0.f : m_used);
      }
      l = l * alpha + ssum;
      // the P region's previous use (two stages back) is done: its O += P . V
      // had completed before the score issuer issued these scores
      const uint32_t pe = bt + ((nt & 1) ? 56 : 40);
      tc_fence_after();
      // row r of P into the tile's P region nt % 2 (lane r, two keys a column)
      tmem_st32(trow + 64u + 32u * (uint32_t)(nt & 1), *reinterpret_cast<uint32_t(*)[32]>(pk));
      // ---- rescale this warp's rows of O once the previous stage's
      // O += P . V is done (alpha = 1 leaves a row unchanged)
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        if (nt >= 1 && !wait_warp(bt + ((nt & 1) ? 40 : 56), (uint32_t)((nt - 1) >> 1) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32(trow + 128u + (uint32_t)cc, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(trow + 128u + (uint32_t)cc, o);
        }
        tmem_wait_st();
      }
      // ---- keys past the sequence's end hold no data (NaN, possibly): their
      // V rows are cleared so that P = 0 multiplies zeros (both warpgroups
      // may clear the same rows: they write the same zeros)
      if (tb + kPBN > it.T) {
        const int z0 = max(0, it.T - tb);
        const int per_plane = (kPBN - z0) * 8;   // 16-byte pieces
        const uint32_t vpart = base + (uint32_t)st * a.stage_bytes + (uint32_t)a.kv_bytes;
        const uint32_t vrow = (uint32_t)a.R * 128u, vblk = vrow * (uint32_t)NP;
        for (int e = r; e < per_plane * NP; e += 128) {
          // key z of the stage: row z % R of block z / R's box, plane p
          const int p = e / per_plane, rem = e - p * per_plane;
          const int z = z0 + (rem >> 3);
          const uint32_t addr = vpart + (uint32_t)(z >> a.log2R) * vblk + (uint32_t)p * vrow +
                                (uint32_t)(z & (a.R - 1)) * 128u + (uint32_t)(rem & 7) * 16u;
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();   // the cleared rows, before the tensor core reads them
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bt + ((nt & 1) ? 24 : 32));   // P region nt % 2 is written
      if (kt == nkt_t - 1) {
        // ---- the tile's last stage: out = O / l once O += P . V is done
        if (!wait_warp(pe, (uint32_t)(nt >> 1) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv = 1.f / l;
        uint16_t* orow =
            a.out + ((size_t)(q0 + (valid ? r / a.G : 0)) * a.Hq + (size_t)it.h * a.G + r % a.G) * D;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32(trow + 128u + (uint32_t)cc, o);
          tmem_wait_ld();
          if (valid) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = pack2<kBF16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<uint4*>(orow + cc + 8 * q4) =
                  make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
          }
        }
        tc_fence_before();
        mbar_arrive(bt + 48);   // O may be overwritten by the tile's next item
      }
      ++nt;
    }
    if (!ok) {
      if (lane == 0 && !*abort_flag) set_error(a.err, PA_DEVERR_TIMEOUT);
      if (lane == 0) *abort_flag = 1;
    }
  }

  // ---- teardown: release the tensor memory (every MMA has completed)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTcMma) tmem_dealloc(tmem, kTcTmemCols);
  // the last CTA to finish resets the work counters for the next call
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.ws + 1, 1u) == gridDim.x - 1) {
      a.ws[0] = 0u;
      a.ws[1] = 0u;
      __threadfence();
    }
  }
}

struct PrefillPlan {
  bool bf16, tc;
  int D, G, B, R, nsb, BM, stages, kv_bytes, stage_bytes, ctrl_off, smem_bytes, grid;
  int q_off, q_tx;
};

int ctrl_bytes(int S) { return 32 * S + 4 * (kPMaxSeqs + 1) + 12 + 16 * 8 + 16; }

template <int D, bool BF>
int prepare_kernel(const PrefillPlan& p, int smem_optin, int* per_sm) {
  cudaError_t e = cudaFuncSetAttribute(paged_prefill_kernel<D, BF>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
  if (e != cudaSuccess) return launch_status(e, "cudaFuncSetAttribute (prefill)");
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, paged_prefill_kernel<D, BF>,
                                                    kPThreads, p.smem_bytes);
  return launch_status(e, "occupancy query (prefill)");
}

template <int D, bool BF>
int prepare_tc_kernel(const PrefillPlan& p, int smem_optin, int* per_sm) {
  cudaError_t e = cudaFuncSetAttribute(paged_prefill_tc_kernel<D, BF>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
  if (e != cudaSuccess) return launch_status(e, "cudaFuncSetAttribute (tensor-core prefill)");
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, paged_prefill_tc_kernel<D, BF>,
                                                    kTcThreads, p.smem_bytes);
  return launch_status(e, "occupancy query (tensor-core prefill)");
}

// Plan of the tensor-core kernel: 64-key stages whose K and V parts are
// [plane][64 keys][128 bytes]; each 64-column plane of a block's rows is one
// TMA box of R rows, which must start on 1024 bytes (the 128-byte swizzle), so
// blocks of fewer than 8 tokens take the warp-level kernel.
int make_tc_plan(int Hq, int Hkv, int D, int B, int dtype, int num_seqs, PrefillPlan* out) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(B) || B < 8 || B > 256) return PA_ERR_UNSUPPORTED;
  PrefillPlan p{};
  p.tc = true;
  p.bf16 = dtype == PA_BF16;
  p.D = D;
  p.G = Hq / Hkv;
  if (p.G > 16) return PA_ERR_UNSUPPORTED;
  p.B = B;
  p.R = B < kPBN ? B : kPBN;
  p.nsb = kPBN / p.R;
  p.BM = kPRows / p.G;
  p.kv_bytes = kPBN * D * 2;
  p.stage_bytes = 2 * p.kv_bytes;
  const int qbuf = (D / 64) * 16384;   // one query tile
  DeviceInfo di;
  if (int rc = current_device_info(&di)) return rc;
  // two query tiles (the item's tiles A and B); P lives in tensor memory
  int st = (di.smem_per_block - 1024 - 2 * qbuf - tc_ctrl_bytes(kPMaxStages, num_seqs)) /
           p.stage_bytes;
  if (st > kPMaxStages) st = kPMaxStages;
  if (st < 2) return PA_ERR_UNSUPPORTED;
  p.stages = st;
  p.q_off = st * p.stage_bytes;
  p.ctrl_off = p.q_off + 2 * qbuf;
  p.smem_bytes = 1024 + p.ctrl_off + tc_ctrl_bytes(st, num_seqs);
  p.q_tx = (D / 64) * 128 * p.G * p.BM;
  int per_sm = 0;
  int rc = D == 64 ? (p.bf16 ? prepare_tc_kernel<64, true>(p, di.smem_per_block, &per_sm)
                             : prepare_tc_kernel<64, false>(p, di.smem_per_block, &per_sm))
                   : (p.bf16 ? prepare_tc_kernel<128, true>(p, di.smem_per_block, &per_sm)
                             : prepare_tc_kernel<128, false>(p, di.smem_per_block, &per_sm));
  if (rc != PA_OK) return rc;
  if (per_sm < 1) return PA_ERR_UNSUPPORTED;
  p.grid = di.sm_count * per_sm;
  *out = p;
  return PA_OK;
}

int make_plan(int Hq, int Hkv, int D, int B, int dtype, PrefillPlan* out) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(B) || B < 2 || B > 256) return PA_ERR_UNSUPPORTED;
  PrefillPlan p{};
  p.bf16 = dtype == PA_BF16;
  p.D = D;
  p.G = Hq / Hkv;
  if (p.G > 16) return PA_ERR_UNSUPPORTED;
  p.B = B;
  p.R = B < kPBN ? B : kPBN;
  p.nsb = kPBN / p.R;
  if (p.nsb > 32) return PA_ERR_UNSUPPORTED;
  // the 128-byte swizzled box must start on 1024 bytes
  if ((p.R * D * 2) % 1024 != 0) return PA_ERR_UNSUPPORTED;
  p.BM = kPRows / p.G;
  p.kv_bytes = kPBN * D * 2;
  p.stage_bytes = 2 * p.kv_bytes;
  DeviceInfo di;
  if (int rc = current_device_info(&di)) return rc;
  int st = (di.smem_per_block - 1024 - ctrl_bytes(kPMaxStages)) / p.stage_bytes;
  if (st > kPMaxStages) st = kPMaxStages;
  if (st < 2) return PA_ERR_UNSUPPORTED;
  p.stages = st;
  p.ctrl_off = st * p.stage_bytes;
  p.smem_bytes = 1024 + p.ctrl_off + ctrl_bytes(st);
  int per_sm = 0;
  int rc = D == 64 ? (p.bf16 ? prepare_kernel<64, true>(p, di.smem_per_block, &per_sm)
                             : prepare_kernel<64, false>(p, di.smem_per_block, &per_sm))
                   : (p.bf16 ? prepare_kernel<128, true>(p, di.smem_per_block, &per_sm)
                             : prepare_kernel<128, false>(p, di.smem_per_block, &per_sm));
  if (rc != PA_OK) return rc;
  if (per_sm < 1) return PA_ERR_UNSUPPORTED;
  p.grid = di.sm_count * per_sm;
  *out = p;
  return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

int pa_prefill_workspace_size(size_t* bytes) {
  if (!bytes) return PA_ERR_INVALID_ARG;
  *bytes = 256;
  return PA_OK;
}

int pa_prefill_kernel(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t dtype, int32_t num_seqs, int32_t* kind) {
  if (!kind || num_seqs < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs > kPMaxSeqs) return PA_ERR_UNSUPPORTED;
  // the same choice as pa_prefill's
  PrefillPlan p;
  const int rc_tc = make_tc_plan(num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                                 num_seqs, &p);
  if (rc_tc == PA_OK) {
    *kind = PA_PREFILL_TENSOR_CORE;
    return PA_OK;
  }
  if (rc_tc != PA_ERR_UNSUPPORTED) return rc_tc;
  if (int rc = make_plan(num_q_heads, num_kv_heads, head_dim, block_size, dtype, &p)) return rc;
  *kind = PA_PREFILL_WARP_MMA;
  return PA_OK;
}

int pa_prefill(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, int32_t table_stride, const int32_t* seq_lens,
               const int32_t* query_start, int32_t num_seqs, int64_t total_q,
               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
               int64_t num_blocks, int32_t dtype, float scale, void* out, void* workspace,
               size_t workspace_bytes, int32_t* err_word, pa_stream stream) {
  if (num_seqs < 0 || total_q < 0 || table_stride < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  // the tensor-core kernel where its staging layout allows (blocks of 8 or
  // more tokens), else the warp-level one
  PrefillPlan p;
  const int rc_tc =
      make_tc_plan(num_q_heads, num_kv_heads, head_dim, block_size, dtype, num_seqs, &p);
  if (rc_tc == PA_ERR_UNSUPPORTED) {
    if (int rc = make_plan(num_q_heads, num_kv_heads, head_dim, block_size, dtype, &p)) return rc;
  } else if (rc_tc != PA_OK) {
    return rc_tc;
  }
  if (num_seqs == 0 || total_q == 0) return PA_OK;
  if (num_seqs > kPMaxSeqs) return PA_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start || !out ||
      !workspace)
    return PA_ERR_INVALID_ARG;
  if (num_blocks == 0 || table_stride == 0 || num_blocks > 0xffffffffLL) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace))
    return PA_ERR_INVALID_ARG;
  if (workspace_bytes < 256) return PA_ERR_WORKSPACE;
  CUtensorMap tk, tv, tq;
  if (p.tc) {
    // K: one box per 64-column plane of a block's rows; V: one box per
    // block, all its planes
    if (int rc = encode_pool_plane_map(&tk, k_cache, p.bf16, p.D, p.B, p.R, num_kv_heads,
                                       num_blocks, 1))
      return rc;
    if (int rc = encode_pool_plane_map(&tv, v_cache, p.bf16, p.D, p.B, p.R, num_kv_heads,
                                       num_blocks, p.D / 64))
      return rc;
    if (int rc = encode_q_tile_map(&tq, q, p.bf16, p.D, p.G, num_kv_heads, total_q, p.BM))
      return rc;
  } else {
    DecodePlan mp{};
    mp.bf16 = p.bf16;
    mp.D = p.D;
    mp.B = p.B;
    mp.R = p.R;
    mp.HG = 1;
    mp.swz = true;
    if (int rc = encode_pool_map(&tk, k_cache, mp, num_kv_heads, num_blocks)) return rc;
    if (int rc = encode_pool_map(&tv, v_cache, mp, num_kv_heads, num_blocks)) return rc;
  }
  PrefillArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.bt = block_tables;
  a.seq_lens = seq_lens;
  a.query_start = query_start;
  a.ws = static_cast<uint32_t*>(workspace);
  a.err = err_word;
  a.num_blocks = num_blocks;
  a.num_seqs = num_seqs;
  a.stride = table_stride;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.G = p.G;
  a.B = p.B;
  a.log2B = ilog2(p.B);
  a.BM = p.BM;
  a.R = p.R;
  a.log2R = ilog2(p.R);
  a.nsb = p.nsb;
  a.stages = p.stages;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.hi_log2 = a.log2R + 7;                     // a plane is R rows of 128 bytes
  a.sub_log2 = a.hi_log2 + ilog2(p.D / 64);    // a box is D/64 planes
  a.kv_bytes = p.kv_bytes;
  a.stage_bytes = p.stage_bytes;
  a.ctrl_off = p.ctrl_off;
  a.q_off = p.q_off;
  a.q_tx = p.q_tx;
  clear_stale_error();
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (p.tc) {
    const dim3 g(p.grid), b(kTcThreads);
    const size_t sm = (size_t)p.smem_bytes;
    if (p.D == 64)
      e = p.bf16 ? launch_pdl(paged_prefill_tc_kernel<64, true>, g, b, sm, s, tk, tv, tq, a)
                 : launch_pdl(paged_prefill_tc_kernel<64, false>, g, b, sm, s, tk, tv, tq, a);
    else
      e = p.bf16 ? launch_pdl(paged_prefill_tc_kernel<128, true>, g, b, sm, s, tk, tv, tq, a)
                 : launch_pdl(paged_prefill_tc_kernel<128, false>, g, b, sm, s, tk, tv, tq, a);
    return launch_status(e, "tensor-core prefill kernel launch");
  }
  if (p.D == 64)
    e = p.bf16 ? launch_pdl(paged_prefill_kernel<64, true>, dim3(p.grid), dim3(kPThreads),
                            (size_t)p.smem_bytes, s, tk, tv, a)
               : launch_pdl(paged_prefill_kernel<64, false>, dim3(p.grid), dim3(kPThreads),
                            (size_t)p.smem_bytes, s, tk, tv, a);
  else
    e = p.bf16 ? launch_pdl(paged_prefill_kernel<128, true>, dim3(p.grid), dim3(kPThreads),
                            (size_t)p.smem_bytes, s, tk, tv, a)
               : launch_pdl(paged_prefill_kernel<128, false>, dim3(p.grid), dim3(kPThreads),
                            (size_t)p.smem_bytes, s, tk, tv, a);
  return launch_status(e, "prefill kernel launch");
}

}  // extern "C"
