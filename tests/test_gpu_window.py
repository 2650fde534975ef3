"""Sliding-window paged decode on the GPU against the fp64 oracle ("vLLM
Framework and Inference Engine Design", section "How does it support prompts of
arbitrary length? Does it have a sliding window?": each token attends only to
the last W tokens; the blocks before the window are released).

Element-wise |gpu - oracle| <= 4e-3 + 1e-2 |oracle| over windows that cut a
block, match a block or chunk edge, exceed the context or keep one token; over
both kernels, head_dim, block size and group size; with the released blocks'
table entries set to -1 and NaN in every slot the decode must not read.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import GpuState, OracleState, assert_close, check_parity, gpu_out_f64, gpu_step

pytestmark = pytest.mark.gpu

LENS = [1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 200, 777, 2049]


def _parity(wl, flags=pa.PA_DECODE_AUTO, num_ctas=0):
    st = GpuState(wl)
    out, _ = gpu_step(st, flags=flags, num_ctas=num_ctas)
    ref = OracleState(wl)
    ref.step()
    expected, spread = ref.decode(spread=True)
    rep = check_parity(out, wl, expected, spread,
                       "window %d flags=%d ctas=%d" % (wl.window, flags, num_ctas), flags=flags)
    assert pa.pa_get_error(st.err) == 0
    return rep["max_abs"]


@pytest.mark.parametrize("window", [1, 7, 16, 17, 100, 128, 129, 1000, 5000])
def test_window_parity_gqa(cuda_device, window):
    wl = W.random_workload(90 + window, W.BF16, 32, 8, 128, 16, LENS, garbage="nan",
                           window=window)
    assert window >= 5000 or np.any(wl.block_tables < 0) or window >= 1000
    _parity(wl)


CASES = [
    # dtype, Hq, Hkv, D, B, window
    (W.F16, 8, 8, 128, 16, 100),    # G = 1: CUDA-core kernel
    (W.BF16, 4, 4, 64, 32, 40),     # a window edge inside a 32-token block, 16-token chunks
    (W.F16, 8, 2, 64, 16, 33),      # 64-token chunks
    (W.BF16, 16, 2, 128, 8, 77),
    (W.F16, 14, 2, 128, 4, 250),
    (W.BF16, 12, 4, 64, 256, 300),
    (W.F16, 6, 3, 128, 4, 65),      # one KV head per group, 128-token chunks
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,B,window", CASES)
def test_window_parity_sweep(cuda_device, dtype, Hq, Hkv, D, B, window):
    wl = W.random_workload(95 + Hq + B, dtype, Hq, Hkv, D, B, LENS, garbage="nan",
                           window=window)
    _parity(wl)
    if Hq == Hkv:
        _parity(wl, flags=pa.PA_DECODE_MMA)


@pytest.mark.parametrize("num_ctas", [1, 5, 300])
def test_window_split_contexts(cuda_device, num_ctas):
    wl = W.random_workload(97, W.BF16, 32, 8, 128, 16, [5000, 3, 4096, 4097, 900, 12000],
                           garbage="nan", window=4096)
    _parity(wl, num_ctas=num_ctas)


def test_window_matches_full_decode_when_it_covers_every_context(cuda_device):
    wl = W.random_workload(98, W.BF16, 8, 2, 128, 16, [10, 100, 300])
    st = GpuState(wl)
    gpu_step(st, decode=False)
    full = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, wl.scale)
    win = pa.pa_decode_window(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens,
                              wl.scale, 300)
    assert torch.equal(full.view(torch.int16), win.view(torch.int16))


def test_window_must_be_positive(cuda_device):
    wl = W.random_workload(99, W.BF16, 8, 2, 64, 16, [10])
    st = GpuState(wl)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_window(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens,
                            wl.scale, 0)
    assert e.value.status == 1
