/*
 * Plain, slow fp64 CPU oracle for paged decode attention and the paged KV
 * cache operations.  TEST INFRASTRUCTURE ONLY: it exists to check the CUDA
 * library and is used by the tests, by the smoke check and by the CPU-baseline
 * leg of the benchmark.  Nothing in the product path may load or call it.
 *
 * It shares no code, header, table or helper with the CUDA library.  Every
 * routine is the textbook definition written out with straight loops:
 * no blocking, no online softmax, no split of the context.
 *
 * Storage conventions (the KV pool as the pages describe it):
 *   one pool per layer for K and one for V, each laid out as
 *   [num_blocks][block_size][num_kv_heads][head_dim]
 *   ("vLLM Framework and Inference Engine Design", section "What is the
 *   essence of vLLM's PagedAttention?", and section "How is vLLM's KV cache
 *   paged?", the per-layer tensor [2, num_blocks, block_size, kv_heads,
 *   head_dim]).  Elements are stored as 16-bit patterns: IEEE-754 binary16
 *   (dtype 0) or bfloat16 (dtype 1).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_F16 0
#define OR_BF16 1

/* ---------------------------------------------------------------------------
 * Element decoding, from the formats' definitions.
 * ------------------------------------------------------------------------- */

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Normal: (-1)^s * 2^(e-15) * (1 + f/1024); subnormal: (-1)^s * 2^-14 * f/1024.
 * Exponent 31 encodes infinity (f == 0) or NaN (f != 0).  Exact in fp64. */
double or_f16_to_f64(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);               /* 2^-14 * f / 2^10 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    }
    return s ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE-754 binary32 (1 sign, 8 exponent bits
 * with bias 127, 7 fraction bits). */
double or_bf16_to_f64(uint16_t b) {
    int s = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);              /* 2^-126 * f / 2^7 */
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp(1.0 + (double)f / 128.0, e - 127);
    }
    return s ? -v : v;
}

static double or_decode(uint16_t x, int dtype) {
    return dtype == OR_BF16 ? or_bf16_to_f64(x) : or_f16_to_f64(x);
}

void or_decode_array(const uint16_t* src, int64_t n, int dtype, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = or_decode(src[i], dtype);
}

/* ---------------------------------------------------------------------------
 * Address translation ("vLLM Framework and Inference Engine Design", section
 * "What is the essence of vLLM's PagedAttention?"):
 *   token t -> logical block j = floor(t / B), slot r = t mod B,
 *   physical block p = block_table[j]; its K and V are K_cache[p][r], V_cache[p][r].
 *   A sequence of T tokens holds ceil(T / B) blocks.
 * ------------------------------------------------------------------------- */

int64_t or_blocks_for(int64_t T, int32_t B) {
    int64_t n = 0;
    /* ceil by counting whole blocks, the definition read literally */
    while (n * (int64_t)B < T) ++n;
    return n;
}

/* Flat slot of token t: block_table[floor(t/B)] * B + (t mod B)
 * ("How is vLLM's KV cache paged?", bullet "Writing": the slot mapping). */
int64_t or_slot(const int32_t* table_row, int64_t t, int32_t B) {
    int64_t j = t / B;
    int64_t r = t % B;
    return (int64_t)table_row[j] * B + r;
}

/* Slot mapping for a list of new tokens given as (sequence index, position). */
void or_slot_mapping(const int32_t* block_tables, int64_t table_stride,
                     const int32_t* token_seq, const int32_t* token_pos, int64_t n,
                     int32_t B, int64_t* slots) {
    for (int64_t k = 0; k < n; ++k) {
        const int32_t* row = block_tables + (int64_t)token_seq[k] * table_stride;
        slots[k] = or_slot(row, token_pos[k], B);
    }
}

/* ---------------------------------------------------------------------------
 * Cache write: each new token's K and V rows ([num_kv_heads][head_dim]) are
 * stored at their flat slot of the pool.  A negative slot marks a padding
 * token that writes nothing (a reading of ours: the pages are silent).
 * ------------------------------------------------------------------------- */
void or_cache_write(uint16_t* k_cache, uint16_t* v_cache,
                    const uint16_t* k, const uint16_t* v,
                    const int64_t* slots, int64_t n, int64_t row_elems) {
    for (int64_t i = 0; i < n; ++i) {
        int64_t s = slots[i];
        if (s < 0) continue;
        for (int64_t e = 0; e < row_elems; ++e) {
            k_cache[s * row_elems + e] = k[i * row_elems + e];
            v_cache[s * row_elems + e] = v[i * row_elems + e];
        }
    }
}

/* ---------------------------------------------------------------------------
 * Copy-on-write block copy ("What operations can cause memory fragmentation,
 * and how does vLLM avoid it?", bullet "Sharing instead of copying"): the whole
 * block src is copied to block dst, K and V.  Pairs are applied in order.
 * ------------------------------------------------------------------------- */
void or_copy_blocks(uint16_t* k_cache, uint16_t* v_cache,
                    const int32_t* pairs, int64_t n, int64_t block_elems) {
    for (int64_t i = 0; i < n; ++i) {
        int64_t src = pairs[2 * i];
        int64_t dst = pairs[2 * i + 1];
        for (int64_t e = 0; e < block_elems; ++e) {
            k_cache[dst * block_elems + e] = k_cache[src * block_elems + e];
            v_cache[dst * block_elems + e] = v_cache[src * block_elems + e];
        }
    }
}

/* ---------------------------------------------------------------------------
 * Block swap between two pools ("vLLM anatomy" / [P3] "Memory Pressure and
 * Preemption": swapping moves physical blocks from GPU memory to the CPU's
 * memory and back): block dst of the destination pool <- block src of the
 * source pool, K and V, for each (src, dst) pair, in order.  block_bytes is
 * the size of one block of one pool.
 * ------------------------------------------------------------------------- */
void or_swap_blocks(const uint8_t* src_k, const uint8_t* src_v, uint8_t* dst_k, uint8_t* dst_v,
                    const int32_t* pairs, int64_t n, int64_t block_bytes) {
    for (int64_t i = 0; i < n; ++i) {
        int64_t src = pairs[2 * i];
        int64_t dst = pairs[2 * i + 1];
        memcpy(dst_k + dst * block_bytes, src_k + src * block_bytes, (size_t)block_bytes);
        memcpy(dst_v + dst * block_bytes, src_v + src * block_bytes, (size_t)block_bytes);
    }
}

/* Gather the first T tokens of one sequence, one KV head, into a contiguous
 * fp64 array out[T][D] by following the block table token by token. */
void or_gather_head(const uint16_t* cache, int dtype, const int32_t* table_row,
                    int64_t T, int32_t B, int32_t H_kv, int32_t D, int32_t h,
                    double* out) {
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = or_slot(table_row, t, B);
        const uint16_t* row = cache + (slot * H_kv + h) * (int64_t)D;
        for (int32_t d = 0; d < D; ++d) out[t * D + d] = or_decode(row[d], dtype);
    }
}

/* Raw 16-bit gather of all heads: out[T][H_kv][D], bit patterns unchanged. */
void or_gather_bits(const uint16_t* cache, const int32_t* table_row, int64_t T,
                    int32_t B, int32_t H_kv, int32_t D, uint16_t* out) {
    int64_t row_elems = (int64_t)H_kv * D;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = or_slot(table_row, t, B);
        memcpy(out + t * row_elems, cache + slot * row_elems,
               (size_t)row_elems * sizeof(uint16_t));
    }
}

/* ---------------------------------------------------------------------------
 * Single-query attention on contiguous fp64 arrays, textbook two-pass softmax
 * ("What is the essence of vLLM's PagedAttention?": scores = q.K^T * scale,
 * weights = softmax(scores), output = weights.V).
 *   q[D], K[T][D], V[T][D] -> out[D]
 *   s_t = scale * sum_d q_d K_td;  w_t = exp(s_t - max s) / sum exp(s - max s)
 *   out_d = sum_t w_t V_td
 * scratch must hold T doubles.
 *
 * If spread is not NULL it receives, per output element, the weighted mean
 * absolute deviation of the values about the output,
 *   spread_d = sum_t w_t |V_td - out_d|.
 * It is not part of the method: it is the scale of the error that perturbing
 * every weight w_t by a relative amount of at most u can cause in out_d (the
 * perturbed output is again a weighted mean, and moves by at most about
 * u * spread_d), which the tests use to bound a kernel's rounding of the
 * weights.
 * ------------------------------------------------------------------------- */
void or_attention_1q(const double* q, const double* K, const double* V,
                     int64_t T, int32_t D, double scale, double* out,
                     double* scratch, double* spread) {
    double m = -INFINITY;
    for (int64_t t = 0; t < T; ++t) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += q[d] * K[t * D + d];
        scratch[t] = scale * dot;
        if (scratch[t] > m) m = scratch[t];
    }
    double z = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        scratch[t] = exp(scratch[t] - m);
        z += scratch[t];
    }
    for (int32_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t t = 0; t < T; ++t) acc += scratch[t] * V[t * D + d];
        out[d] = acc / z;
    }
    if (spread) {
        for (int32_t d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t) acc += scratch[t] * fabs(V[t * D + d] - out[d]);
            spread[d] = acc / z;
        }
    }
}

/* ---------------------------------------------------------------------------
 * Paged single-query decode for a list of sequences.
 *   q        [num_seqs][Hq][D]           (16-bit, dtype)
 *   pools    [num_blocks][B][H_kv][D]    (16-bit, dtype)
 *   block_tables [num_seqs][table_stride] int32, seq_lens[num_seqs] int32
 *   seq_ids  the n_ids sequences to evaluate; out[n_ids][Hq][D] fp64.
 *   spread   NULL, or [n_ids][Hq][D] fp64: each element's weighted mean
 *            absolute deviation (or_attention_1q); zero for a zero-length row.
 * Query head hq reads KV head floor(hq / G), G = Hq / H_kv (contiguous query
 * groups: our reading of grouped-query attention, which the pages name in
 * "How big the KV cache is: a formula and a real measurement" without giving
 * the head mapping).  A sequence of length 0 yields a zero row (our reading).
 * Returns 0, or -1 on an allocation failure.
 * ------------------------------------------------------------------------- */
int or_paged_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                    int dtype, const int32_t* block_tables, int64_t table_stride,
                    const int32_t* seq_lens, const int32_t* seq_ids, int32_t n_ids,
                    int32_t Hq, int32_t H_kv, int32_t D, int32_t B, double scale,
                    double* out, double* spread, int threads) {
    int32_t G = Hq / H_kv;
    int64_t n_work = (int64_t)n_ids * H_kv;
    int failed = 0;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
    for (int64_t w = 0; w < n_work; ++w) {
        int32_t idx = (int32_t)(w / H_kv);
        int32_t h = (int32_t)(w % H_kv);
        int32_t i = seq_ids[idx];
        int64_t T = seq_lens[i];
        double* o = out + (int64_t)idx * Hq * D;
        if (T <= 0) {
            for (int32_t g = 0; g < G; ++g)
                for (int32_t d = 0; d < D; ++d) {
                    o[(int64_t)(h * G + g) * D + d] = 0.0;
                    if (spread) spread[((int64_t)idx * Hq + h * G + g) * D + d] = 0.0;
                }
            continue;
        }
        const int32_t* row = block_tables + (int64_t)i * table_stride;
        double* K = (double*)malloc((size_t)(T * D) * sizeof(double));
        double* V = (double*)malloc((size_t)(T * D) * sizeof(double));
        double* s = (double*)malloc((size_t)T * sizeof(double));
        double* qv = (double*)malloc((size_t)D * sizeof(double));
        if (!K || !V || !s || !qv) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
            or_gather_head(k_cache, dtype, row, T, B, H_kv, D, h, K);
            or_gather_head(v_cache, dtype, row, T, B, H_kv, D, h, V);
            for (int32_t g = 0; g < G; ++g) {
                int32_t hq = h * G + g;
                const uint16_t* qrow = q + ((int64_t)i * Hq + hq) * D;
                for (int32_t d = 0; d < D; ++d) qv[d] = or_decode(qrow[d], dtype);
                or_attention_1q(qv, K, V, T, D, scale, o + (int64_t)hq * D, s,
                                spread ? spread + ((int64_t)idx * Hq + hq) * D : NULL);
            }
        }
        free(K);
        free(V);
        free(s);
        free(qv);
    }
    return failed ? -1 : 0;
}

/* ---------------------------------------------------------------------------
 * Sliding-window paged decode ("vLLM Framework and Inference Engine Design",
 * section "How does it support prompts of arbitrary length? Does it have a
 * sliding window?": in a model trained with sliding-window attention each
 * token attends only to the last W tokens, so only the blocks inside the
 * window are needed and the older ones can be released).  Our reading: the
 * query of position T - 1 attends to tokens [max(0, T - W), T); table entries
 * of blocks wholly before the window may have been released (any value) and
 * are never read.  W <= 0 means no window.  Arguments otherwise as
 * or_paged_decode.
 * ------------------------------------------------------------------------- */
int or_paged_decode_window(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                           int dtype, const int32_t* block_tables, int64_t table_stride,
                           const int32_t* seq_lens, int32_t window, const int32_t* seq_ids,
                           int32_t n_ids, int32_t Hq, int32_t H_kv, int32_t D, int32_t B,
                           double scale, double* out, double* spread, int threads) {
    int32_t G = Hq / H_kv;
    int64_t n_work = (int64_t)n_ids * H_kv;
    int failed = 0;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
    for (int64_t w = 0; w < n_work; ++w) {
        int32_t idx = (int32_t)(w / H_kv);
        int32_t h = (int32_t)(w % H_kv);
        int32_t i = seq_ids[idx];
        int64_t T = seq_lens[i];
        double* o = out + (int64_t)idx * Hq * D;
        if (T <= 0) {
            for (int32_t g = 0; g < G; ++g)
                for (int32_t d = 0; d < D; ++d) {
                    o[(int64_t)(h * G + g) * D + d] = 0.0;
                    if (spread) spread[((int64_t)idx * Hq + h * G + g) * D + d] = 0.0;
                }
            continue;
        }
        int64_t s0 = (window > 0 && T > window) ? T - window : 0;
        int64_t n = T - s0;   /* tokens attended */
        const int32_t* row = block_tables + (int64_t)i * table_stride;
        double* K = (double*)malloc((size_t)(n * D) * sizeof(double));
        double* V = (double*)malloc((size_t)(n * D) * sizeof(double));
        double* s = (double*)malloc((size_t)n * sizeof(double));
        double* qv = (double*)malloc((size_t)D * sizeof(double));
        if (!K || !V || !s || !qv) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
            for (int64_t t = s0; t < T; ++t) {
                int64_t slot = or_slot(row, t, B);
                const uint16_t* kr = k_cache + (slot * H_kv + h) * (int64_t)D;
                const uint16_t* vr = v_cache + (slot * H_kv + h) * (int64_t)D;
                for (int32_t d = 0; d < D; ++d) {
                    K[(t - s0) * D + d] = or_decode(kr[d], dtype);
                    V[(t - s0) * D + d] = or_decode(vr[d], dtype);
                }
            }
            for (int32_t g = 0; g < G; ++g) {
                int32_t hq = h * G + g;
                const uint16_t* qrow = q + ((int64_t)i * Hq + hq) * D;
                for (int32_t d = 0; d < D; ++d) qv[d] = or_decode(qrow[d], dtype);
                or_attention_1q(qv, K, V, n, D, scale, o + (int64_t)hq * D, s,
                                spread ? spread + ((int64_t)idx * Hq + hq) * D : NULL);
            }
        }
        free(K);
        free(V);
        free(s);
        free(qv);
    }
    return failed ? -1 : 0;
}

/* ---------------------------------------------------------------------------
 * Multi-query paged attention for chunked prefill and prefix-cache hits
 * ("vLLM Framework and Inference Engine Design", section "How does it support
 * prompts of arbitrary length?": a long prompt is processed in chunks, mixed
 * with other requests' decode tokens in one batch; "vLLM self-hosted", section
 * "Two phases: prefill and decode").  Sequence i has L_i = query_start[i + 1] -
 * query_start[i] new tokens, already written to the cache, at the end of its
 * seq_lens[i] tokens; new token j sits at position p = seq_lens[i] - L_i + j
 * and attends causally to tokens [0, p] through the block table.  Decode is
 * the case L_i = 1.
 *   q, out   [total_q][Hq][D] (q 16-bit in dtype, out fp64), rows of sequence
 *            i at [query_start[i], query_start[i + 1])
 * ------------------------------------------------------------------------- */
int or_paged_prefill(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                     int dtype, const int32_t* block_tables, int64_t table_stride,
                     const int32_t* seq_lens, const int32_t* query_start, int32_t num_seqs,
                     int32_t Hq, int32_t H_kv, int32_t D, int32_t B, double scale,
                     double* out, double* spread, int threads) {
    int32_t G = Hq / H_kv;
    int64_t n_work = (int64_t)num_seqs * H_kv;
    int failed = 0;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
    for (int64_t w = 0; w < n_work; ++w) {
        int32_t i = (int32_t)(w / H_kv);
        int32_t h = (int32_t)(w % H_kv);
        int64_t T = seq_lens[i];
        int64_t q0 = query_start[i], L = query_start[i + 1] - q0;
        if (L <= 0 || T <= 0 || L > T) continue;
        const int32_t* row = block_tables + (int64_t)i * table_stride;
        double* K = (double*)malloc((size_t)(T * D) * sizeof(double));
        double* V = (double*)malloc((size_t)(T * D) * sizeof(double));
        double* s = (double*)malloc((size_t)T * sizeof(double));
        double* qv = (double*)malloc((size_t)D * sizeof(double));
        if (!K || !V || !s || !qv) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
            or_gather_head(k_cache, dtype, row, T, B, H_kv, D, h, K);
            or_gather_head(v_cache, dtype, row, T, B, H_kv, D, h, V);
            for (int64_t j = 0; j < L; ++j) {
                int64_t p = T - L + j;   /* the token's position: it sees [0, p] */
                for (int32_t g = 0; g < G; ++g) {
                    int32_t hq = h * G + g;
                    const uint16_t* qrow = q + ((q0 + j) * Hq + hq) * D;
                    for (int32_t d = 0; d < D; ++d) qv[d] = or_decode(qrow[d], dtype);
                    or_attention_1q(qv, K, V, p + 1, D, scale, out + ((q0 + j) * Hq + hq) * D, s,
                                    spread ? spread + ((q0 + j) * Hq + hq) * D : NULL);
                }
            }
        }
        free(K);
        free(V);
        free(s);
        free(qv);
    }
    return failed ? -1 : 0;
}

/* The same single-query attention over a contiguous (unpaged) cache
 * K[T][H_kv][D] (fp64), used to check that paging changes only the addressing:
 * "vLLM Framework and Inference Engine Design", section "What is the essence
 * of vLLM's PagedAttention?", has the attention computation as the one place
 * that must learn about blocks, the rest of the model being untouched. */
void or_contiguous_decode(const double* q /*[Hq][D]*/, const double* K, const double* V,
                          int64_t T, int32_t Hq, int32_t H_kv, int32_t D, double scale,
                          double* out /*[Hq][D]*/) {
    int32_t G = Hq / H_kv;
    double* Kh = (double*)malloc((size_t)(T * D + 1) * sizeof(double));
    double* Vh = (double*)malloc((size_t)(T * D + 1) * sizeof(double));
    double* s = (double*)malloc((size_t)(T + 1) * sizeof(double));
    for (int32_t h = 0; h < H_kv; ++h) {
        for (int64_t t = 0; t < T; ++t)
            for (int32_t d = 0; d < D; ++d) {
                Kh[t * D + d] = K[(t * H_kv + h) * D + d];
                Vh[t * D + d] = V[(t * H_kv + h) * D + d];
            }
        for (int32_t g = 0; g < G; ++g) {
            int32_t hq = h * G + g;
            or_attention_1q(q + (int64_t)hq * D, Kh, Vh, T, D, scale, out + (int64_t)hq * D, s,
                            NULL);
        }
    }
    free(Kh);
    free(Vh);
    free(s);
}

/* ---------------------------------------------------------------------------
 * FP8 KV cache ("vLLM Framework and Inference Engine Design", section "How can
 * one customize the tokenizer, cache strategy, or scheduler strategy?", the
 * kv_cache_dtype="fp8" flag: half the KV memory of FP16; "vLLM anatomy",
 * section "Quantization: Reducing Weight & KV Precision": --kv-cache-dtype fp8
 * stores the KV cache in FP8).  The pages name neither the 8-bit format nor a
 * scale convention.  Our reading: the OCP E4M3 format with one scale per
 * tensor (one for K, one for V); a stored code c stands for e4m3(c) * scale,
 * and a value x is stored as c = e4m3_rne_satfinite(float(x) / scale), the
 * division done in IEEE binary32.
 * ------------------------------------------------------------------------- */

/* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits, no
 * infinities.  Exponent field 0: (-1)^s * 2^-6 * f/8 (subnormal); fields
 * 1..15: (-1)^s * 2^(e-7) * (1 + f/8), except S.1111.111, which is NaN.  The
 * largest finite magnitude is 1.75 * 2^8 = 448.  Exact in fp64. */
double or_e4m3_to_f64(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int f = c & 7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0) v = ldexp((double)f / 8.0, -6);
    else v = ldexp(1.0 + (double)f / 8.0, e - 7);
    return s ? -v : v;
}

/* Round half to even of a non-negative double. */
static double or_rne(double q) {
    double fl = floor(q);
    double diff = q - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

/* binary32 -> E4M3 code, round to nearest (ties to even), magnitudes beyond
 * the largest finite value saturate to +-448; NaN gives 0x7F. */
uint8_t or_e4m3_from_f32(float x) {
    if (isnan(x)) return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7e;
    if (a < ldexp(1.0, -6)) {
        /* subnormal spacing 2^-9; a result of 8 is the smallest normal, code 8 */
        double m = or_rne(a / ldexp(1.0, -9));
        return sign | (uint8_t)m;
    }
    int e2;
    frexp(a, &e2);          /* a = fr * 2^e2, fr in [0.5, 1): a in [2^(e2-1), 2^e2) */
    int e = e2 - 1;         /* a in [2^e, 2^(e+1)) */
    double m = or_rne(a / ldexp(1.0, e - 3));   /* in [8, 16] */
    if (m == 16.0) {
        m = 8.0;
        e += 1;
    }
    if (e + 7 > 15 || (e + 7 == 15 && m - 8.0 > 6.0)) return sign | 0x7e;
    return sign | (uint8_t)(((e + 7) << 3) | (int)(m - 8.0));
}

void or_e4m3_encode_array(const float* src, int64_t n, uint8_t* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = or_e4m3_from_f32(src[i]);
}

void or_e4m3_decode_array(const uint8_t* src, int64_t n, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = or_e4m3_to_f64(src[i]);
}

/* Quantizing cache write: pool row at slot_mapping[n] <- codes of k[n], v[n]
 * (16-bit rows of row_elems elements in src_dtype); slot < 0 is skipped. */
void or_cache_write_fp8(uint8_t* k_cache, uint8_t* v_cache, const uint16_t* k,
                        const uint16_t* v, int src_dtype, const int64_t* slots,
                        int64_t n_tok, int64_t row_elems, float k_scale, float v_scale) {
    for (int64_t n = 0; n < n_tok; ++n) {
        int64_t s = slots[n];
        if (s < 0) continue;
        for (int64_t e = 0; e < row_elems; ++e) {
            volatile float kx = (float)or_decode(k[n * row_elems + e], src_dtype);
            volatile float vx = (float)or_decode(v[n * row_elems + e], src_dtype);
            volatile float kq = kx / k_scale;
            volatile float vq = vx / v_scale;
            k_cache[s * row_elems + e] = or_e4m3_from_f32(kq);
            v_cache[s * row_elems + e] = or_e4m3_from_f32(vq);
        }
    }
}

/* Gather of one KV head from an E4M3 pool: out[t][d] = e4m3(code) * scale. */
void or_gather_head_fp8(const uint8_t* cache, double scale, const int32_t* table_row,
                        int64_t T, int32_t B, int32_t H_kv, int32_t D, int32_t h,
                        double* out) {
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = or_slot(table_row, t, B);
        const uint8_t* row = cache + (slot * H_kv + h) * (int64_t)D;
        for (int32_t d = 0; d < D; ++d) out[t * D + d] = or_e4m3_to_f64(row[d]) * scale;
    }
}

/* Paged single-query decode over E4M3 pools: the same textbook attention as
 * or_paged_decode on the dequantized K and V; q (and the output) stay in
 * q_dtype (binary16 or bfloat16). */
int or_paged_decode_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                        int q_dtype, double k_scale, double v_scale,
                        const int32_t* block_tables, int64_t table_stride,
                        const int32_t* seq_lens, const int32_t* seq_ids, int32_t n_ids,
                        int32_t Hq, int32_t H_kv, int32_t D, int32_t B, double scale,
                        double* out, double* spread, int threads) {
    int32_t G = Hq / H_kv;
    int64_t n_work = (int64_t)n_ids * H_kv;
    int failed = 0;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
    for (int64_t w = 0; w < n_work; ++w) {
        int32_t idx = (int32_t)(w / H_kv);
        int32_t h = (int32_t)(w % H_kv);
        int32_t i = seq_ids[idx];
        int64_t T = seq_lens[i];
        double* o = out + (int64_t)idx * Hq * D;
        if (T <= 0) {
            for (int32_t g = 0; g < G; ++g)
                for (int32_t d = 0; d < D; ++d) {
                    o[(int64_t)(h * G + g) * D + d] = 0.0;
                    if (spread) spread[((int64_t)idx * Hq + h * G + g) * D + d] = 0.0;
                }
            continue;
        }
        const int32_t* row = block_tables + (int64_t)i * table_stride;
        double* K = (double*)malloc((size_t)(T * D) * sizeof(double));
        double* V = (double*)malloc((size_t)(T * D) * sizeof(double));
        double* s = (double*)malloc((size_t)T * sizeof(double));
        double* qv = (double*)malloc((size_t)D * sizeof(double));
        if (!K || !V || !s || !qv) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        } else {
            or_gather_head_fp8(k_cache, k_scale, row, T, B, H_kv, D, h, K);
            or_gather_head_fp8(v_cache, v_scale, row, T, B, H_kv, D, h, V);
            for (int32_t g = 0; g < G; ++g) {
                int32_t hq = h * G + g;
                const uint16_t* qrow = q + ((int64_t)i * Hq + hq) * D;
                for (int32_t d = 0; d < D; ++d) qv[d] = or_decode(qrow[d], q_dtype);
                or_attention_1q(qv, K, V, T, D, scale, o + (int64_t)hq * D, s,
                                spread ? spread + ((int64_t)idx * Hq + hq) * D : NULL);
            }
        }
        free(K);
        free(V);
        free(s);
        free(qv);
    }
    return failed ? -1 : 0;
}

int or_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
