"""fp64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and this package never
imports the product.

Two parts:

* ``libpa_oracle.so`` (``pa_oracle.c``): element decoding, address translation,
  slot mapping, cache write, block copy, gather and textbook two-pass softmax
  attention, all in fp64 with straight loops.
* Plain-Python capacity arithmetic printed on the pages (blocks per sequence,
  wasted slots, KV bytes per token, pool sizing, static-batch useful fraction),
  each pinned by the tests to the worked examples the pages print.

Page names used in citations:
  [P1] "vLLM Framework and Inference Engine Design" (vineetganti.com)
  [P3] "vLLM anatomy: high-throughput LLM inference" (karya-semi.vercel.app)
  [P4] "vLLM self-hosted" (sudo.vn)
  [P5] "vLLM" (bibekananda.in)
"""
import ctypes
import math
import os

import numpy as np

from .build import LIB, build_oracle

F16 = 0
BF16 = 1

_lib = None


def lib():
    """Load (building if needed) the C oracle."""
    global _lib
    if _lib is None:
        path = build_oracle()
        L = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        f64p = ctypes.POINTER(ctypes.c_double)
        L.or_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.or_f16_to_f64.restype = ctypes.c_double
        L.or_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.or_bf16_to_f64.restype = ctypes.c_double
        L.or_decode_array.argtypes = [u16p, ctypes.c_int64, ctypes.c_int, f64p]
        L.or_blocks_for.argtypes = [ctypes.c_int64, ctypes.c_int32]
        L.or_blocks_for.restype = ctypes.c_int64
        L.or_slot.argtypes = [i32p, ctypes.c_int64, ctypes.c_int32]
        L.or_slot.restype = ctypes.c_int64
        L.or_slot_mapping.argtypes = [i32p, ctypes.c_int64, i32p, i32p, ctypes.c_int64,
                                      ctypes.c_int32, i64p]
        L.or_cache_write.argtypes = [u16p, u16p, u16p, u16p, i64p, ctypes.c_int64,
                                     ctypes.c_int64]
        L.or_copy_blocks.argtypes = [u16p, u16p, i32p, ctypes.c_int64, ctypes.c_int64]
        L.or_gather_head.argtypes = [u16p, ctypes.c_int, i32p, ctypes.c_int64, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, f64p]
        L.or_gather_bits.argtypes = [u16p, i32p, ctypes.c_int64, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.c_int32, u16p]
        L.or_attention_1q.argtypes = [f64p, f64p, f64p, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_double, f64p, f64p, f64p]
        L.or_paged_decode.argtypes = [u16p, u16p, u16p, ctypes.c_int, i32p, ctypes.c_int64,
                                      i32p, i32p, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_double, f64p, f64p, ctypes.c_int]
        L.or_paged_decode.restype = ctypes.c_int
        L.or_contiguous_decode.argtypes = [f64p, f64p, f64p, ctypes.c_int64, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_double, f64p]
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        L.or_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.or_e4m3_to_f64.restype = ctypes.c_double
        L.or_e4m3_from_f32.argtypes = [ctypes.c_float]
        L.or_e4m3_from_f32.restype = ctypes.c_uint8
        L.or_e4m3_encode_array.argtypes = [f32p, ctypes.c_int64, u8p]
        L.or_e4m3_decode_array.argtypes = [u8p, ctypes.c_int64, f64p]
        L.or_cache_write_fp8.argtypes = [u8p, u8p, u16p, u16p, ctypes.c_int, i64p,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                         ctypes.c_float]
        L.or_gather_head_fp8.argtypes = [u8p, ctypes.c_double, i32p, ctypes.c_int64,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, f64p]
        L.or_paged_decode_fp8.argtypes = [u16p, u8p, u8p, ctypes.c_int, ctypes.c_double,
                                          ctypes.c_double, i32p, ctypes.c_int64, i32p, i32p,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_double, f64p,
                                          f64p, ctypes.c_int]
        L.or_paged_decode_fp8.restype = ctypes.c_int
        L.or_paged_decode_window.argtypes = [u16p, u16p, u16p, ctypes.c_int, i32p,
                                             ctypes.c_int64, i32p, ctypes.c_int32, i32p,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                             f64p, f64p, ctypes.c_int]
        L.or_paged_decode_window.restype = ctypes.c_int
        L.or_swap_blocks.argtypes = [u8p, u8p, u8p, u8p, i32p, ctypes.c_int64, ctypes.c_int64]
        L.or_paged_prefill.argtypes = [u16p, u16p, u16p, ctypes.c_int, i32p, ctypes.c_int64,
                                       i32p, i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_double, f64p,
                                       f64p, ctypes.c_int]
        L.or_paged_prefill.restype = ctypes.c_int
        L.or_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _opt(a):
    """fp64 array pointer, or NULL for None."""
    return ctypes.POINTER(ctypes.c_double)() if a is None else _p(a, ctypes.c_double)


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("expected uint16 bit patterns, got %s" % a.dtype)
    return a


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


# --------------------------------------------------------------------------
# Element decoding
# --------------------------------------------------------------------------

def decode(bits, dtype):
    """16-bit patterns -> exact fp64 values (binary16 for F16, bfloat16 for BF16)."""
    bits = _u16(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().or_decode_array(_p(bits, ctypes.c_uint16), bits.size, int(dtype),
                          _p(out, ctypes.c_double))
    return out


# --------------------------------------------------------------------------
# Address translation and cache operations   [P1 "What is the essence of
# vLLM's PagedAttention?", "How is vLLM's KV cache paged?"]
# --------------------------------------------------------------------------

def blocks_for(T, B):
    """ceil(T / B): blocks held by a sequence of T tokens."""
    return int(lib().or_blocks_for(int(T), int(B)))


def slot(table_row, t, B):
    """block_table[floor(t/B)] * B + (t mod B)."""
    row = _i32(table_row)
    return int(lib().or_slot(_p(row, ctypes.c_int32), int(t), int(B)))


def slot_mapping(block_tables, token_seq, token_pos, B):
    """Flat slots for new tokens given as (sequence index, position)."""
    bt = _i32(block_tables)
    ts = _i32(token_seq)
    tp = _i32(token_pos)
    n = ts.size
    out = np.empty(n, dtype=np.int64)
    lib().or_slot_mapping(_p(bt, ctypes.c_int32), bt.shape[1], _p(ts, ctypes.c_int32),
                          _p(tp, ctypes.c_int32), n, int(B), _p(out, ctypes.c_int64))
    return out


def cache_write(k_cache, v_cache, k, v, slots):
    """In place: pool rows at `slots` <- k, v rows (bit copies; slot < 0 skipped).

    k_cache, v_cache: uint16 [num_blocks, B, H_kv, D]; k, v: uint16 [n, H_kv, D].
    """
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k = _u16(k)
    v = _u16(v)
    s = np.ascontiguousarray(slots, dtype=np.int64)
    row = k_cache.shape[2] * k_cache.shape[3]
    lib().or_cache_write(_p(k_cache, ctypes.c_uint16), _p(v_cache, ctypes.c_uint16),
                         _p(k, ctypes.c_uint16), _p(v, ctypes.c_uint16),
                         _p(s, ctypes.c_int64), s.size, row)


def copy_blocks(k_cache, v_cache, pairs):
    """In place: block dst <- block src for each (src, dst) pair, K and V.

    Pools of 16-bit patterns, or of 8-bit codes (copied as byte pairs).
    """
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    if k_cache.dtype == np.uint8:
        k_cache = k_cache.view(np.uint16)
        v_cache = v_cache.view(np.uint16)
    pr = _i32(pairs).reshape(-1, 2)
    blk = k_cache.shape[1] * k_cache.shape[2] * k_cache.shape[3]
    lib().or_copy_blocks(_p(k_cache, ctypes.c_uint16), _p(v_cache, ctypes.c_uint16),
                         _p(pr, ctypes.c_int32), pr.shape[0], blk)


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs):
    """In place: destination pool block dst <- source pool block src, K and V,
    for each (src, dst) pair (pools of any element type, same block shape)."""
    for a in (src_k, src_v, dst_k, dst_v):
        assert a.flags.c_contiguous
    assert src_k.shape[1:] == dst_k.shape[1:] and src_k.dtype == dst_k.dtype
    pr = _i32(pairs).reshape(-1, 2)
    block_bytes = src_k[0].nbytes
    u8 = ctypes.c_uint8
    lib().or_swap_blocks(_p(src_k.view(np.uint8), u8), _p(src_v.view(np.uint8), u8),
                         _p(dst_k.view(np.uint8), u8), _p(dst_v.view(np.uint8), u8),
                         _p(pr, ctypes.c_int32), pr.shape[0], block_bytes)


def gather_bits(cache, table_row, T):
    """Bit-exact gather of a sequence's first T tokens: uint16 [T, H_kv, D]."""
    cache = _u16(cache)
    nb, B, H, D = cache.shape
    row = _i32(table_row)
    out = np.empty((int(T), H, D), dtype=np.uint16)
    lib().or_gather_bits(_p(cache, ctypes.c_uint16), _p(row, ctypes.c_int32), int(T), B, H, D,
                         _p(out, ctypes.c_uint16))
    return out


def gather_head(cache, dtype, table_row, T, h):
    """fp64 [T, D] of KV head h for a sequence's first T tokens."""
    cache = _u16(cache)
    nb, B, H, D = cache.shape
    row = _i32(table_row)
    out = np.empty((int(T), D), dtype=np.float64)
    lib().or_gather_head(_p(cache, ctypes.c_uint16), int(dtype), _p(row, ctypes.c_int32),
                         int(T), B, H, D, int(h), _p(out, ctypes.c_double))
    return out


# --------------------------------------------------------------------------
# Attention   [P1 "What is the essence of vLLM's PagedAttention?"]
# --------------------------------------------------------------------------

def attention_1q(q, K, V, scale, spread=False):
    """softmax(scale * q.K^T) . V for one query: q [D], K, V [T, D] (fp64).

    With spread=True returns (out, spread), spread[d] = sum_t w_t |V[t, d] -
    out[d]| (the weighted mean absolute deviation about the output)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    T, D = K.shape
    out = np.empty(D, dtype=np.float64)
    scratch = np.empty(max(T, 1), dtype=np.float64)
    sp = np.empty(D, dtype=np.float64) if spread else None
    lib().or_attention_1q(_p(q, ctypes.c_double), _p(K, ctypes.c_double),
                          _p(V, ctypes.c_double), T, D, float(scale),
                          _p(out, ctypes.c_double), _p(scratch, ctypes.c_double), _opt(sp))
    return (out, sp) if spread else out


def paged_decode(q, k_cache, v_cache, dtype, block_tables, seq_lens, scale,
                 seq_ids=None, threads=0, spread=False):
    """fp64 decode output [len(seq_ids), Hq, D].

    q: uint16 [N, Hq, D]; pools uint16 [num_blocks, B, H_kv, D];
    block_tables int32 [N, stride]; seq_lens int32 [N].  Query head hq reads KV
    head hq // (Hq // H_kv).  With spread=True returns (out, spread), spread
    as in attention_1q, per output element.
    """
    q = _u16(q)
    k_cache = _u16(k_cache)
    v_cache = _u16(v_cache)
    N, Hq, D = q.shape
    nb, B, H_kv, D2 = k_cache.shape
    assert D == D2 and Hq % H_kv == 0
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    ids = _i32(np.arange(N) if seq_ids is None else seq_ids)
    out = np.empty((ids.size, Hq, D), dtype=np.float64)
    sp = np.empty_like(out) if spread else None
    rc = lib().or_paged_decode(_p(q, ctypes.c_uint16), _p(k_cache, ctypes.c_uint16),
                               _p(v_cache, ctypes.c_uint16), int(dtype), _p(bt, ctypes.c_int32),
                               bt.shape[1], _p(sl, ctypes.c_int32), _p(ids, ctypes.c_int32),
                               ids.size, Hq, H_kv, D, B, float(scale),
                               _p(out, ctypes.c_double), _opt(sp), int(threads))
    if rc != 0:
        raise MemoryError("oracle decode could not allocate its gather buffers")
    return (out, sp) if spread else out


def paged_decode_window(q, k_cache, v_cache, dtype, block_tables, seq_lens, window, scale,
                        seq_ids=None, threads=0, spread=False):
    """Sliding-window decode [P1 "How does it support prompts of arbitrary
    length? Does it have a sliding window?"]: the query of position T - 1
    attends to tokens [max(0, T - window), T); table entries before the window
    are never read.  window <= 0: full attention."""
    q = _u16(q)
    k_cache = _u16(k_cache)
    v_cache = _u16(v_cache)
    N, Hq, D = q.shape
    nb, B, H_kv, D2 = k_cache.shape
    assert D == D2 and Hq % H_kv == 0
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    ids = _i32(np.arange(N) if seq_ids is None else seq_ids)
    out = np.empty((ids.size, Hq, D), dtype=np.float64)
    sp = np.empty_like(out) if spread else None
    rc = lib().or_paged_decode_window(_p(q, ctypes.c_uint16), _p(k_cache, ctypes.c_uint16),
                                      _p(v_cache, ctypes.c_uint16), int(dtype),
                                      _p(bt, ctypes.c_int32), bt.shape[1], _p(sl, ctypes.c_int32),
                                      int(window), _p(ids, ctypes.c_int32), ids.size, Hq, H_kv, D,
                                      B, float(scale), _p(out, ctypes.c_double), _opt(sp),
                                      int(threads))
    if rc != 0:
        raise MemoryError("oracle decode could not allocate its gather buffers")
    return (out, sp) if spread else out


def paged_prefill(q, k_cache, v_cache, dtype, block_tables, seq_lens, query_start, scale,
                  threads=0, spread=False):
    """Multi-query paged attention (chunked prefill; decode is L_i = 1):
    fp64 out [total_q, Hq, D].  Sequence i's new tokens are q rows
    [query_start[i], query_start[i+1]), sitting at the end of its seq_lens[i]
    cached tokens; token j of them attends causally to [0, T_i - L_i + j]."""
    q = _u16(q)
    k_cache = _u16(k_cache)
    v_cache = _u16(v_cache)
    total, Hq, D = q.shape
    nb, B, H_kv, D2 = k_cache.shape
    assert D == D2 and Hq % H_kv == 0
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    qs = _i32(query_start)
    assert qs.size == sl.size + 1 and qs[-1] == total
    out = np.zeros((total, Hq, D), dtype=np.float64)
    sp = np.zeros_like(out) if spread else None
    rc = lib().or_paged_prefill(_p(q, ctypes.c_uint16), _p(k_cache, ctypes.c_uint16),
                                _p(v_cache, ctypes.c_uint16), int(dtype), _p(bt, ctypes.c_int32),
                                bt.shape[1], _p(sl, ctypes.c_int32), _p(qs, ctypes.c_int32),
                                sl.size, Hq, H_kv, D, B, float(scale), _p(out, ctypes.c_double),
                                _opt(sp), int(threads))
    if rc != 0:
        raise MemoryError("oracle prefill could not allocate its gather buffers")
    return (out, sp) if spread else out


def contiguous_decode(q, K, V, scale):
    """Unpaged single-query attention: q [Hq, D], K, V [T, H_kv, D] (fp64)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    Hq, D = q.shape
    T, H_kv, _ = K.shape
    out = np.empty((Hq, D), dtype=np.float64)
    lib().or_contiguous_decode(_p(q, ctypes.c_double), _p(K, ctypes.c_double),
                               _p(V, ctypes.c_double), T, Hq, H_kv, D, float(scale),
                               _p(out, ctypes.c_double))
    return out


def max_threads():
    return int(lib().or_max_threads())


# --------------------------------------------------------------------------
# FP8 (E4M3) KV cache   [P1 "How can one customize the tokenizer, cache
# strategy, or scheduler strategy?" (kv_cache_dtype="fp8"); P3 "Quantization:
# Reducing Weight & KV Precision" (--kv-cache-dtype fp8)].  Our reading: OCP
# E4M3 codes with one scale per tensor; code = e4m3_rne_satfinite(x / scale)
# with the division in binary32, value = e4m3(code) * scale.
# --------------------------------------------------------------------------

def e4m3_decode(codes):
    """uint8 E4M3 codes -> exact fp64 values (NaN for S.1111.111)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().or_e4m3_decode_array(_p(c, ctypes.c_uint8), c.size, _p(out, ctypes.c_double))
    return out


def e4m3_encode(x):
    """binary32 values -> E4M3 codes (round to nearest even, saturating)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().or_e4m3_encode_array(_p(x, ctypes.c_float), x.size, _p(out, ctypes.c_uint8))
    return out


def cache_write_fp8(k_cache, v_cache, k, v, src_dtype, slots, k_scale, v_scale):
    """In place: pool rows at `slots` <- E4M3 codes of k / k_scale, v / v_scale.

    k_cache, v_cache: uint8 [num_blocks, B, H_kv, D]; k, v: uint16 [n, H_kv, D]
    in src_dtype; slot < 0 skipped.
    """
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k = _u16(k)
    v = _u16(v)
    s = np.ascontiguousarray(slots, dtype=np.int64)
    row = k_cache.shape[2] * k_cache.shape[3]
    lib().or_cache_write_fp8(_p(k_cache, ctypes.c_uint8), _p(v_cache, ctypes.c_uint8),
                             _p(k, ctypes.c_uint16), _p(v, ctypes.c_uint16), int(src_dtype),
                             _p(s, ctypes.c_int64), s.size, row, float(np.float32(k_scale)),
                             float(np.float32(v_scale)))


def gather_head_fp8(cache, scale, table_row, T, h):
    """fp64 [T, D] of KV head h from an E4M3 pool, dequantized."""
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    nb, B, H, D = cache.shape
    row = _i32(table_row)
    out = np.empty((int(T), D), dtype=np.float64)
    lib().or_gather_head_fp8(_p(cache, ctypes.c_uint8), float(scale), _p(row, ctypes.c_int32),
                             int(T), B, H, D, int(h), _p(out, ctypes.c_double))
    return out


def paged_decode_fp8(q, k_cache, v_cache, q_dtype, k_scale, v_scale, block_tables, seq_lens,
                     scale, seq_ids=None, threads=0, spread=False):
    """fp64 decode output [len(seq_ids), Hq, D] over E4M3 pools (uint8);
    with spread=True returns (out, spread) as paged_decode does."""
    q = _u16(q)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint8)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint8)
    N, Hq, D = q.shape
    nb, B, H_kv, D2 = k_cache.shape
    assert D == D2 and Hq % H_kv == 0
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    ids = _i32(np.arange(N) if seq_ids is None else seq_ids)
    out = np.empty((ids.size, Hq, D), dtype=np.float64)
    sp = np.empty_like(out) if spread else None
    rc = lib().or_paged_decode_fp8(_p(q, ctypes.c_uint16), _p(k_cache, ctypes.c_uint8),
                                   _p(v_cache, ctypes.c_uint8), int(q_dtype),
                                   float(np.float32(k_scale)), float(np.float32(v_scale)),
                                   _p(bt, ctypes.c_int32), bt.shape[1], _p(sl, ctypes.c_int32),
                                   _p(ids, ctypes.c_int32), ids.size, Hq, H_kv, D, B,
                                   float(scale), _p(out, ctypes.c_double), _opt(sp),
                                   int(threads))
    if rc != 0:
        raise MemoryError("oracle decode could not allocate its gather buffers")
    return (out, sp) if spread else out


# --------------------------------------------------------------------------
# Capacity arithmetic printed on the pages (plain Python, exact integers)
# --------------------------------------------------------------------------

def static_batch_useful_fraction(prompts, outputs):
    """[P1 "Why is batching multiple requests difficult for traditional
    inference engines?"]  sum(p_i + o_i) / (n * (max p + max o)), as a
    (numerator, denominator) pair of integers."""
    n = len(prompts)
    num = sum(p + o for p, o in zip(prompts, outputs))
    den = n * (max(prompts) + max(outputs))
    return num, den


def wasted_slots_contiguous(lengths, max_len):
    """[P1 "What operations can cause memory fragmentation ...?"]
    sum_i (max_len - T_i): slots a contiguous reservation never uses."""
    return sum(max_len - T for T in lengths)


def allocated_slots_paged(lengths, B):
    """sum_i ceil(T_i / B) * B: slots held under paging."""
    return sum(blocks_for(T, B) * B for T in lengths)


def wasted_slots_paged(lengths, B):
    """sum_i (ceil(T_i / B) * B - T_i); each term is below B."""
    return sum(blocks_for(T, B) * B - T for T in lengths)


def kv_bytes_per_token(layers, kv_heads, head_dim, dtype_bytes):
    """[P4 "How big the KV cache is"]  2 (K and V) * layers * kv_heads *
    head_dim * bytes per element."""
    return 2 * layers * kv_heads * head_dim * dtype_bytes


def block_bytes(layers, block_size, kv_heads, head_dim, dtype_bytes):
    """[P1 "How is vLLM's KV cache paged?"]  2 * L * block_size * H_kv * d * b."""
    return 2 * layers * block_size * kv_heads * head_dim * dtype_bytes


def pool_blocks(budget_bytes, block_nbytes):
    """Whole blocks that fit in a byte budget (floor division)."""
    return budget_bytes // block_nbytes


def requests_that_fit(free_bytes, bytes_per_request):
    """Whole requests that fit in free memory (floor division)."""
    return int(free_bytes // bytes_per_request)


def sliding_window_max_blocks(W, B):
    """[P1 "How does it support prompts of arbitrary length? ..."]  a window of
    W tokens touches at most ceil(W / B) + 1 blocks."""
    return blocks_for(W, B) + 1
