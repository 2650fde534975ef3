"""Test harness: one step of the paged decode path through the CUDA library
(C ABI, via the binding) and the same step through the fp64 oracle, on the
same seeded workload.

A step is: copy-on-write block copies (if any), slot mapping, cache write,
decode ("vLLM Framework and Inference Engine Design": K/V are written to their
slots when computed; the query of the newest token then attends over
seq_len tokens, its own included).
"""
import numpy as np
import torch

import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W

# decode tolerance per element: |gpu - oracle| <= ATOL + RTOL * |oracle|
ATOL = 4e-3
RTOL = 1e-2

TORCH_DTYPE = {W.F16: torch.float16, W.BF16: torch.bfloat16}


def to_dev(bits, dtype, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TORCH_DTYPE[dtype])


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class GpuState:
    """The workload's inputs resident on the GPU."""

    def __init__(self, wl, device="cuda"):
        self.wl = wl
        if wl.fp8:   # uint8 E4M3 codes
            self.k_cache = torch.from_numpy(wl.k_cache).to(device)
            self.v_cache = torch.from_numpy(wl.v_cache).to(device)
        else:
            self.k_cache = to_dev(wl.k_cache, wl.dtype, device)
            self.v_cache = to_dev(wl.v_cache, wl.dtype, device)
        self.q = to_dev(wl.q, wl.dtype, device)
        self.k_new = to_dev(wl.k_new, wl.dtype, device)
        self.v_new = to_dev(wl.v_new, wl.dtype, device)
        self.block_tables = torch.from_numpy(wl.block_tables).to(device)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(device)
        self.new_seq = torch.from_numpy(wl.new_seq).to(device)
        self.new_pos = torch.from_numpy(wl.new_pos).to(device)
        self.pairs = torch.from_numpy(np.ascontiguousarray(wl.copy_pairs, np.int32)).to(device)
        self.query_start = (None if wl.query_start is None
                            else torch.from_numpy(wl.query_start).to(device))
        self.err = torch.zeros(1, dtype=torch.int32, device=device)


def gpu_step(st, flags=pa.PA_DECODE_AUTO, num_ctas=0, decode=True):
    """Runs the step; returns (out tensor or None, slot_mapping tensor)."""
    wl = st.wl
    if st.pairs.numel():
        pa.pa_copy_blocks(st.pairs, st.k_cache, st.v_cache, err=st.err)
    slots = pa.pa_slot_mapping(st.block_tables, st.new_seq, st.new_pos, wl.block_size,
                               wl.num_blocks, err=st.err)
    if wl.fp8:
        pa.pa_cache_write_fp8(st.k_new, st.v_new, slots, st.k_cache, st.v_cache, wl.k_scale,
                              wl.v_scale, err=st.err)
    else:
        pa.pa_cache_write(st.k_new, st.v_new, slots, st.k_cache, st.v_cache, err=st.err)
    out = None
    if decode:
        out = gpu_decode(st, st.seq_lens, flags=flags, num_ctas=num_ctas)
    return out, slots


def gpu_decode(st, seq_lens, flags=pa.PA_DECODE_AUTO, num_ctas=0, workspace=None):
    """The decode call of the workload's cache type."""
    wl = st.wl
    if wl.query_start is not None:
        return pa.pa_prefill(st.q, st.k_cache, st.v_cache, st.block_tables, seq_lens,
                             st.query_start, wl.scale, workspace=workspace, err=st.err)
    if wl.window > 0:
        return pa.pa_decode_window(st.q, st.k_cache, st.v_cache, st.block_tables, seq_lens,
                                   wl.scale, wl.window, flags=flags, num_ctas=num_ctas,
                                   workspace=workspace, err=st.err)
    if wl.fp8:
        return pa.pa_decode_fp8(st.q, st.k_cache, st.v_cache, st.block_tables, seq_lens,
                                wl.scale, wl.k_scale, wl.v_scale, flags=flags,
                                num_ctas=num_ctas, workspace=workspace, err=st.err)
    return pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, seq_lens, wl.scale,
                        flags=flags, num_ctas=num_ctas, workspace=workspace, err=st.err)


class OracleState:
    """Host copies of the workload's pools, stepped by the oracle."""

    def __init__(self, wl):
        self.wl = wl
        self.k_cache = wl.k_cache.copy()
        self.v_cache = wl.v_cache.copy()

    def step(self):
        wl = self.wl
        if wl.copy_pairs.size:
            oracle.copy_blocks(self.k_cache, self.v_cache, wl.copy_pairs)
        self.slots = oracle.slot_mapping(wl.block_tables, wl.new_seq, wl.new_pos, wl.block_size)
        if wl.fp8:
            oracle.cache_write_fp8(self.k_cache, self.v_cache, wl.k_new, wl.v_new, wl.dtype,
                                   self.slots, wl.k_scale, wl.v_scale)
        else:
            oracle.cache_write(self.k_cache, self.v_cache, wl.k_new, wl.v_new, self.slots)

    def decode(self, seq_ids=None, threads=0, seq_lens=None):
        wl = self.wl
        sl = wl.seq_lens if seq_lens is None else seq_lens
        if wl.query_start is not None:
            return oracle.paged_prefill(wl.q, self.k_cache, self.v_cache, wl.dtype,
                                        wl.block_tables, sl, wl.query_start, wl.scale,
                                        threads=threads)
        if wl.window > 0:
            return oracle.paged_decode_window(wl.q, self.k_cache, self.v_cache, wl.dtype,
                                              wl.block_tables, sl, wl.window, wl.scale,
                                              seq_ids=seq_ids, threads=threads)
        if wl.fp8:
            return oracle.paged_decode_fp8(wl.q, self.k_cache, self.v_cache, wl.dtype, wl.k_scale,
                                           wl.v_scale, wl.block_tables, sl, wl.scale,
                                           seq_ids=seq_ids, threads=threads)
        return oracle.paged_decode(wl.q, self.k_cache, self.v_cache, wl.dtype, wl.block_tables,
                                   sl, wl.scale, seq_ids=seq_ids, threads=threads)


def gpu_out_f64(out):
    return out.float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, what=""):
    """Element-wise |got - ref| <= ATOL + RTOL * |ref| (the decode tolerance)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError("%s: %d of %d elements out of tolerance (max abs err %.3g); first %s"
                             % (what, int(bad.sum()), bad.size, float(err.max()), idx))
    return float(err.max())
