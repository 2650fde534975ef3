"""Thin torch-facing wrappers over the C ABI (argument marshalling only).

Every function takes CUDA tensors, checks dtypes and shapes, passes raw device
pointers, sizes and the current CUDA stream to libpa.so, and raises PAError on
a non-zero status.  Nothing is computed here.
"""
import ctypes

import torch

from . import _lib
from ._lib import PA_BF16, PA_DECODE_AUTO, PA_F16, PA_FP8_E4M3, PA_SWAP_IN, PA_SWAP_OUT


class PAError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = _lib.load().pa_strerror(status)
        super().__init__("%s failed: %s (status %d)" % (what, msg.decode() if msg else "?", status))


def _check(status, what):
    if status != 0:
        raise PAError(status, what)


def _dtype_code(t):
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError("expected float16 or bfloat16, got %s" % t.dtype)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _cuda(t, name):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _pool_shape(k_cache, v_cache):
    _cuda(k_cache, "k_cache")
    _cuda(v_cache, "v_cache")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype or k_cache.dim() != 4:
        raise ValueError("k_cache and v_cache must share one shape [num_blocks, B, H_kv, D]")
    return k_cache.shape


def _fp8_pools(k_cache, v_cache):
    shape = _pool_shape(k_cache, v_cache)
    if k_cache.dtype != torch.uint8:
        raise TypeError("E4M3 pools must be uint8 tensors of codes")
    return shape


def pa_version():
    return _lib.load().pa_version()


def pa_slot_mapping(block_tables, token_seq, token_pos, block_size, num_blocks, out=None,
                    err=None):
    """int64 slots block_tables[seq][pos // B] * B + pos % B for each new token."""
    L = _lib.load()
    for t, n in ((block_tables, "block_tables"), (token_seq, "token_seq"), (token_pos, "token_pos")):
        _cuda(t, n)
        if t.dtype != torch.int32:
            raise TypeError("%s must be int32" % n)
    n_tok = token_seq.numel()
    if token_pos.numel() != n_tok:
        raise ValueError("token_seq and token_pos differ in length")
    if out is None:
        out = torch.empty(n_tok, dtype=torch.int64, device=token_seq.device)
    _check(L.pa_slot_mapping(_ptr(block_tables), block_tables.shape[1], block_tables.shape[0],
                             _ptr(token_seq), _ptr(token_pos), n_tok, int(block_size),
                             int(num_blocks), _ptr(out), _ptr(err), _stream()), "pa_slot_mapping")
    return out


def pa_cache_write(k, v, slot_mapping, k_cache, v_cache, err=None):
    """Store k[n], v[n] ([n_tok, H_kv, D]) at pool slot slot_mapping[n]."""
    L = _lib.load()
    nb, B, H, D = _pool_shape(k_cache, v_cache)
    _cuda(k, "k")
    _cuda(v, "v")
    _cuda(slot_mapping, "slot_mapping")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    n_tok = slot_mapping.numel()
    if k.shape != (n_tok, H, D) or v.shape != (n_tok, H, D):
        raise ValueError("k, v must be [num_tokens, H_kv, D]")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype:
        raise TypeError("k, v and the pools must share a dtype")
    _check(L.pa_cache_write(_ptr(k), _ptr(v), _ptr(slot_mapping), n_tok, _ptr(k_cache),
                            _ptr(v_cache), nb, B, H, D, _dtype_code(k_cache), _ptr(err),
                            _stream()), "pa_cache_write")


def pa_cache_write_mapped(k, v, block_tables, token_seq, token_pos, k_cache, v_cache,
                          slot_mapping=None, err=None):
    """pa_slot_mapping and pa_cache_write in one launch: store k[n], v[n]
    ([n_tok, H_kv, D]) at slot block_tables[seq][pos // B] * B + pos % B of
    new token n; the int64 slots go to slot_mapping when given."""
    L = _lib.load()
    nb, B, H, D = _pool_shape(k_cache, v_cache)
    for t, n in ((block_tables, "block_tables"), (token_seq, "token_seq"), (token_pos, "token_pos")):
        _cuda(t, n)
        if t.dtype != torch.int32:
            raise TypeError("%s must be int32" % n)
    _cuda(k, "k")
    _cuda(v, "v")
    n_tok = token_seq.numel()
    if token_pos.numel() != n_tok:
        raise ValueError("token_seq and token_pos differ in length")
    if k.shape != (n_tok, H, D) or v.shape != (n_tok, H, D):
        raise ValueError("k, v must be [num_tokens, H_kv, D]")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype:
        raise TypeError("k, v and the pools must share a dtype")
    if slot_mapping is not None:
        _cuda(slot_mapping, "slot_mapping")
        if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != n_tok:
            raise ValueError("slot_mapping must be int64 [num_tokens]")
    _check(L.pa_cache_write_mapped(_ptr(k), _ptr(v), _ptr(block_tables), block_tables.shape[1],
                                   block_tables.shape[0], _ptr(token_seq), _ptr(token_pos), n_tok,
                                   _ptr(k_cache), _ptr(v_cache), nb, B, H, D,
                                   _dtype_code(k_cache), _ptr(slot_mapping), _ptr(err), _stream()),
           "pa_cache_write_mapped")
    return slot_mapping


def pa_copy_blocks(pairs, k_cache, v_cache, err=None):
    """Copy pool block src -> dst (K and V) for each row (src, dst) of pairs.

    Pools of float16 / bfloat16 elements, or uint8 E4M3 codes."""
    L = _lib.load()
    nb, B, H, D = _pool_shape(k_cache, v_cache)
    _cuda(pairs, "pairs")
    if pairs.dtype != torch.int32:
        raise TypeError("pairs must be int32 [n, 2]")
    n = pairs.numel() // 2
    code = PA_FP8_E4M3 if k_cache.dtype == torch.uint8 else _dtype_code(k_cache)
    _check(L.pa_copy_blocks(_ptr(pairs), n, _ptr(k_cache), _ptr(v_cache), nb, B, H, D,
                            code, _ptr(err), _stream()), "pa_copy_blocks")


def pa_swap_blocks(pairs, src_k, src_v, dst_k, dst_v, err=None):
    """Copy block src of the source pools to block dst of the destination
    pools for each row (src, dst) of pairs: one pool pair on the GPU, the other
    in host memory the GPU can address (pinned; or any host memory where the
    GPU reads the host's page tables).  The direction follows from which is
    which."""
    L = _lib.load()
    _cuda(pairs, "pairs")
    if pairs.dtype != torch.int32:
        raise TypeError("pairs must be int32 [n, 2]")
    if src_k.is_cuda == dst_k.is_cuda:
        raise ValueError("one pool pair must be on the GPU and the other in pinned host memory")
    dev_k, dev_v, host_k, host_v = (src_k, src_v, dst_k, dst_v) if src_k.is_cuda else \
        (dst_k, dst_v, src_k, src_v)
    for t in (host_k, host_v):
        if not t.is_contiguous():
            raise ValueError("the host pools must be contiguous")
    _pool_shape(dev_k, dev_v)
    if host_k.shape[1:] != dev_k.shape[1:] or host_k.dtype != dev_k.dtype or \
            host_v.shape != host_k.shape or host_v.dtype != host_k.dtype:
        raise ValueError("host and device pools must share the block shape and dtype")
    nbd, B, H, D = dev_k.shape
    code = PA_FP8_E4M3 if dev_k.dtype == torch.uint8 else _dtype_code(dev_k)
    direction = PA_SWAP_OUT if src_k.is_cuda else PA_SWAP_IN
    _check(L.pa_swap_blocks(_ptr(pairs), pairs.numel() // 2, direction, _ptr(dev_k), _ptr(dev_v),
                            nbd, ctypes.c_void_p(host_k.data_ptr()),
                            ctypes.c_void_p(host_v.data_ptr()), host_k.shape[0], B, H, D, code,
                            _ptr(err), _stream()), "pa_swap_blocks")


def pa_cache_write_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, err=None):
    """Quantize k[n], v[n] ([n_tok, H_kv, D], float16 / bfloat16) to E4M3 codes
    (value / scale, round to nearest even, saturating) at pool slot
    slot_mapping[n] of the uint8 pools."""
    L = _lib.load()
    nb, B, H, D = _fp8_pools(k_cache, v_cache)
    _cuda(k, "k")
    _cuda(v, "v")
    _cuda(slot_mapping, "slot_mapping")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    n_tok = slot_mapping.numel()
    if k.shape != (n_tok, H, D) or v.shape != (n_tok, H, D) or k.dtype != v.dtype:
        raise ValueError("k, v must be [num_tokens, H_kv, D] of one dtype")
    _check(L.pa_cache_write_fp8(_ptr(k), _ptr(v), _dtype_code(k), _ptr(slot_mapping), n_tok,
                                _ptr(k_cache), _ptr(v_cache), nb, B, H, D, float(k_scale),
                                float(v_scale), _ptr(err), _stream()), "pa_cache_write_fp8")


def pa_cache_write_fp8_mapped(k, v, block_tables, token_seq, token_pos, k_cache, v_cache,
                              k_scale, v_scale, slot_mapping=None, err=None):
    """pa_slot_mapping and pa_cache_write_fp8 in one launch: E4M3 codes of
    k[n] / k_scale and v[n] / v_scale ([n_tok, H_kv, D], float16 / bfloat16)
    stored at slot block_tables[seq][pos // B] * B + pos % B of new token n;
    the int64 slots go to slot_mapping when given."""
    L = _lib.load()
    nb, B, H, D = _pool_shape(k_cache, v_cache)
    for t, n in ((block_tables, "block_tables"), (token_seq, "token_seq"), (token_pos, "token_pos")):
        _cuda(t, n)
        if t.dtype != torch.int32:
            raise TypeError("%s must be int32" % n)
    _cuda(k, "k")
    _cuda(v, "v")
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("E4M3 pools are uint8 codes")
    n_tok = token_seq.numel()
    if token_pos.numel() != n_tok:
        raise ValueError("token_seq and token_pos differ in length")
    if k.shape != (n_tok, H, D) or v.shape != (n_tok, H, D) or k.dtype != v.dtype:
        raise ValueError("k, v must be [num_tokens, H_kv, D] of one dtype")
    if slot_mapping is not None:
        _cuda(slot_mapping, "slot_mapping")
        if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != n_tok:
            raise ValueError("slot_mapping must be int64 [num_tokens]")
    _check(L.pa_cache_write_fp8_mapped(_ptr(k), _ptr(v), _dtype_code(k), _ptr(block_tables),
                                       block_tables.shape[1], block_tables.shape[0],
                                       _ptr(token_seq), _ptr(token_pos), n_tok, _ptr(k_cache),
                                       _ptr(v_cache), nb, B, H, D, float(k_scale), float(v_scale),
                                       _ptr(slot_mapping), _ptr(err), _stream()),
           "pa_cache_write_fp8_mapped")
    return slot_mapping


def pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                             flags=PA_DECODE_AUTO, num_ctas=0):
    L = _lib.load()
    if isinstance(dtype, torch.dtype):
        dtype = {torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.uint8: PA_FP8_E4M3}[dtype]
    n = ctypes.c_size_t(0)
    _check(L.pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                                      flags, num_ctas, ctypes.byref(n)),
           "pa_decode_workspace_size")
    return n.value


def pa_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, out=None, workspace=None,
              flags=PA_DECODE_AUTO, num_ctas=0, err=None):
    """Paged single-query decode attention: out [N, Hq, D]."""
    L = _lib.load()
    nb, B, H, D = _pool_shape(k_cache, v_cache)
    _cuda(q, "q")
    _cuda(block_tables, "block_tables")
    _cuda(seq_lens, "seq_lens")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    N, Hq, Dq = q.shape
    if Dq != D or q.dtype != k_cache.dtype:
        raise ValueError("q must be [N, Hq, D] in the pool dtype")
    if block_tables.dim() != 2 or block_tables.shape[0] != N or seq_lens.numel() != N:
        raise ValueError("block_tables must be [N, stride] and seq_lens [N]")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = pa_decode_workspace_size(Hq, H, D, B, _dtype_code(q), flags, num_ctas)
        # zero-filled once; the decode leaves it ready for the next call
        workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    _check(L.pa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                       block_tables.shape[1], _ptr(seq_lens), N, Hq, H, D, B, nb,
                       _dtype_code(q), float(scale), _ptr(out), _ptr(workspace),
                       workspace.numel() * workspace.element_size(), int(flags), int(num_ctas),
                       _ptr(err), _stream()), "pa_decode")
    return out


def pa_decode_window(q, k_cache, v_cache, block_tables, seq_lens, scale, window, out=None,
                     workspace=None, flags=PA_DECODE_AUTO, num_ctas=0, err=None):
    """Sliding-window decode: the query of position T - 1 attends to tokens
    [max(0, T - window), T); table entries of blocks before the window are
    never read (released blocks may be -1)."""
    L = _lib.load()
    nb, B, H, D = _pool_shape(k_cache, v_cache)
    _cuda(q, "q")
    _cuda(block_tables, "block_tables")
    _cuda(seq_lens, "seq_lens")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    N, Hq, Dq = q.shape
    if Dq != D or q.dtype != k_cache.dtype:
        raise ValueError("q must be [N, Hq, D] in the pool dtype")
    if block_tables.dim() != 2 or block_tables.shape[0] != N or seq_lens.numel() != N:
        raise ValueError("block_tables must be [N, stride] and seq_lens [N]")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = pa_decode_workspace_size(Hq, H, D, B, _dtype_code(q), flags, num_ctas)
        workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    _check(L.pa_decode_window(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                              block_tables.shape[1], _ptr(seq_lens), N, Hq, H, D, B, nb,
                              _dtype_code(q), float(scale), int(window), _ptr(out),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              int(flags), int(num_ctas), _ptr(err), _stream()),
           "pa_decode_window")
    return out


def pa_decode_fp8(q, k_cache, v_cache, block_tables, seq_lens, scale, k_scale, v_scale, out=None,
                  workspace=None, flags=PA_DECODE_AUTO, num_ctas=0, err=None):
    """Paged decode over uint8 E4M3 pools (value = code * scale): out [N, Hq, D]
    in q's dtype."""
    L = _lib.load()
    nb, B, H, D = _fp8_pools(k_cache, v_cache)
    _cuda(q, "q")
    _cuda(block_tables, "block_tables")
    _cuda(seq_lens, "seq_lens")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    N, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("q must be [N, Hq, D]")
    if block_tables.dim() != 2 or block_tables.shape[0] != N or seq_lens.numel() != N:
        raise ValueError("block_tables must be [N, stride] and seq_lens [N]")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        nbytes = pa_decode_workspace_size(Hq, H, D, B, PA_FP8_E4M3, flags, num_ctas)
        # zero-filled once; the decode leaves it ready for the next call
        workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    _check(L.pa_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                           block_tables.shape[1], _ptr(seq_lens), N, Hq, H, D, B, nb,
                           _dtype_code(q), float(scale), float(k_scale), float(v_scale),
                           _ptr(out), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), int(flags),
                           int(num_ctas), _ptr(err), _stream()), "pa_decode_fp8")
    return out


def pa_prefill(q, k_cache, v_cache, block_tables, seq_lens, query_start, scale, out=None,
               workspace=None, err=None):
    """Multi-query paged attention (chunked prefill, decode tokens allowed):
    q [total_q, Hq, D]; sequence i's new tokens are rows [query_start[i],
    query_start[i+1]), already written at the end of its seq_lens[i] tokens."""
    L = _lib.load()
    nb, B, H, D = _pool_shape(k_cache, v_cache)
    for t, n in ((q, "q"), (block_tables, "block_tables"), (seq_lens, "seq_lens"),
                 (query_start, "query_start")):
        _cuda(t, n)
    for t, n in ((block_tables, "block_tables"), (seq_lens, "seq_lens"),
                 (query_start, "query_start")):
        if t.dtype != torch.int32:
            raise TypeError("%s must be int32" % n)
    total, Hq, Dq = q.shape
    N = seq_lens.numel()
    if Dq != D or q.dtype != k_cache.dtype:
        raise ValueError("q must be [total_q, Hq, D] in the pool dtype")
    if query_start.numel() != N + 1 or block_tables.dim() != 2 or block_tables.shape[0] != N:
        raise ValueError("query_start must be [N + 1] and block_tables [N, stride]")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        n = ctypes.c_size_t(0)
        _check(L.pa_prefill_workspace_size(ctypes.byref(n)), "pa_prefill_workspace_size")
        workspace = torch.zeros(n.value, dtype=torch.uint8, device=q.device)
    _check(L.pa_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                        block_tables.shape[1], _ptr(seq_lens), _ptr(query_start), N, total, Hq, H,
                        D, B, nb, _dtype_code(q), float(scale), _ptr(out), _ptr(workspace),
                        workspace.numel(), _ptr(err), _stream()), "pa_prefill")
    return out


def pa_prefill_kernel(num_q_heads, num_kv_heads, head_dim, block_size, dtype, num_seqs):
    """Which kernel pa_prefill runs for this shape on the current device:
    PA_PREFILL_TENSOR_CORE or PA_PREFILL_WARP_MMA."""
    L = _lib.load()
    kind = ctypes.c_int32(-1)
    _check(L.pa_prefill_kernel(num_q_heads, num_kv_heads, head_dim, block_size, dtype, num_seqs,
                               ctypes.byref(kind)), "pa_prefill_kernel")
    return kind.value


def pa_gather_kv(k_cache, v_cache, block_tables, seq_lens, out_offsets, total_rows,
                 flags=PA_DECODE_AUTO, err=None):
    """Contiguous copies [total_rows, H_kv, D] of every sequence's K and V."""
    L = _lib.load()
    nb, B, H, D = _pool_shape(k_cache, v_cache)
    N = seq_lens.numel()
    k_out = torch.empty((total_rows, H, D), dtype=k_cache.dtype, device=k_cache.device)
    v_out = torch.empty_like(k_out)
    _check(L.pa_gather_kv(_ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                          _ptr(seq_lens), _ptr(out_offsets), N, H, D, B, nb,
                          _dtype_code(k_cache), int(flags), _ptr(k_out), _ptr(v_out), _ptr(err),
                          _stream()), "pa_gather_kv")
    return k_out, v_out


def pa_get_error(err):
    """Synchronize the current stream, return and clear the device error bits."""
    L = _lib.load()
    flags = ctypes.c_int32(0)
    rc = L.pa_get_error(_ptr(err), _stream(), ctypes.byref(flags))
    if rc not in (0, _lib.PA_ERR_DEVICE_INDEX):
        raise PAError(rc, "pa_get_error")
    return flags.value
