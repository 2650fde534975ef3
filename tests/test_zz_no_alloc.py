"""pa_decode_noalloc against pa_decode.

pa_decode_noalloc serves callers that cannot allocate device memory (a runtime
whose device memory another allocator owns, a C program without a device
allocator, a decode loop that cannot afford cudaMalloc's synchronization): it
runs the decode kernels with their workspace in a fixed array inside the
library.  This file is collected last so that, if it fails, a run that stops at
the first failure has already run every other test; it also passes on its own
in a fresh process, where its first call sets the array up.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import GpuState, assert_close, gpu_out_f64
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


def test_noalloc_matches_pa_decode_on_two_calls(cuda_device):
    cases = [W.random_workload(31, W.BF16, 32, 8, 128, 16, [5, 4000, 700, 64, 1, 2500]),
             W.random_workload(32, W.F16, 4, 4, 64, 16, [3000, 17, 129, 900])]
    for wl in cases:
        st = GpuState(wl)
        ref = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, wl.scale)
        out = torch.empty_like(st.q)
        assert _noalloc(st, out) == 0
        assert pa.pa_get_error(st.err) == 0
        assert_close(gpu_out_f64(out), gpu_out_f64(ref), "noalloc vs pa_decode " + wl.name)


def test_noalloc_rejects_a_workspace_beyond_its_array(cuda_device):
    wl = W.random_workload(33, W.BF16, 32, 2, 128, 16, [100])
    st = GpuState(wl)
    need = pa.pa_decode_workspace_size(32, 2, 128, 16, W.BF16, num_ctas=2000)
    assert need > _lib.PA_NOALLOC_SCRATCH_BYTES
    out = torch.empty_like(st.q)
    assert _noalloc(st, out, num_ctas=2000) == _lib.PA_ERR_WORKSPACE
