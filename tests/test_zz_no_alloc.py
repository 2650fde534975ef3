"""pa_decode_noalloc against pa_decode and against the oracle.

pa_decode_noalloc serves callers that cannot allocate device memory: a
runtime whose device memory another allocator already owns, a C program with
no device allocator, a decode loop that cannot afford cudaMalloc's
synchronization.  It runs the decode kernels with their workspace in a fixed
array inside the library.  It launches the same kernels on the same grid as
pa_decode, so its output must match pa_decode's bit for bit; every call
shares the array, so calls in a row (the same shape twice, another shape,
another grid, and back) must each match.

This file is collected last so that, if it fails, a run that stops at the
first failure has already run every other test; it also passes on its own in
a fresh process, where its first call sets the array up.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import GpuState, OracleState, bits_of, check_parity, gpu_step
from paged_kv_cache_72_gb300 import _lib

pytestmark = pytest.mark.gpu


def _noalloc(st, out, num_ctas=0):
    wl = st.wl
    L = _lib.load()
    return L.pa_decode_noalloc(
        ctypes.c_void_p(st.q.data_ptr()), ctypes.c_void_p(st.k_cache.data_ptr()),
        ctypes.c_void_p(st.v_cache.data_ptr()), ctypes.c_void_p(st.block_tables.data_ptr()),
        st.block_tables.shape[1], ctypes.c_void_p(st.seq_lens.data_ptr()), wl.num_seqs,
        wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.num_blocks, wl.dtype,
        wl.scale, ctypes.c_void_p(out.data_ptr()), pa.PA_DECODE_AUTO, num_ctas,
        ctypes.c_void_p(st.err.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_pa_decode_on_calls_in_a_row(cuda_device):
    # long contexts split across thread blocks, so every call counts pieces on
    # the array's counters and merges them
    shapes = {
        "a": W.random_workload(31, W.BF16, 32, 8, 128, 16, [5, 4000, 700, 64, 1, 2500]),
        "b": W.random_workload(32, W.F16, 4, 4, 64, 16, [3000, 17, 129, 900]),
    }
    states, refs = {}, {}
    for key, wl in shapes.items():
        st = GpuState(wl)
        gpu_step(st, decode=False)   # this step's cache write
        assert pa.pa_get_error(st.err) == 0
        ref = OracleState(wl)
        ref.step()
        states[key], refs[key] = st, ref.decode(spread=True)
    # the same shape twice, the other shape, a smaller grid, and back
    for k, (key, ctas) in enumerate([("a", 0), ("a", 0), ("b", 0), ("a", 7), ("a", 0),
                                     ("b", 40)]):
        st, wl = states[key], shapes[key]
        expected = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens,
                                wl.scale, num_ctas=ctas, err=st.err)
        out = torch.full_like(st.q, float("nan"))
        assert _noalloc(st, out, num_ctas=ctas) == 0
        assert pa.pa_get_error(st.err) == 0
        assert np.array_equal(bits_of(out), bits_of(expected)), \
            "call %d (%s, ctas=%d): not bit-identical to pa_decode" % (k, wl.name, ctas)
        check_parity(out, wl, refs[key][0], refs[key][1], "noalloc call %d (%s)" % (k, wl.name))


def test_noalloc_rejects_a_workspace_beyond_its_array(cuda_device):
    wl = W.random_workload(33, W.BF16, 32, 2, 128, 16, [100])
    st = GpuState(wl)
    need = pa.pa_decode_workspace_size(32, 2, 128, 16, W.BF16, num_ctas=2000)
    assert need > _lib.PA_NOALLOC_SCRATCH_BYTES
    out = torch.empty_like(st.q)
    assert _noalloc(st, out, num_ctas=2000) == _lib.PA_ERR_WORKSPACE
