"""Decode with PA_DECODE_TABLES_READY: the lengths and block tables are read
while the preceding kernel (the cache write of the same step) drains, while
the pools, q, out and the workspace are touched only after it completes.  The
result must match the oracle and be bit-identical to the call without the
flag, on every cache type; empty sequences still get zero rows and bad
lengths are still reported."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import (GpuState, OracleState, assert_close, check_parity, gpu_decode,
                     gpu_out_f64, gpu_step)

pytestmark = pytest.mark.gpu

TR = pa.PA_DECODE_TABLES_READY
LENS = [1, 15, 16, 17, 129, 700, 3000, 2]


def _cases():
    # group sizes 4, 4, 8 and 1 (the CUDA-core kernel); bf16, f16, window, E4M3
    return [
        W.random_workload(2101, W.BF16, 32, 8, 128, 16, LENS, kv_sigma=0.7, garbage="nan"),
        W.random_workload(2102, W.F16, 8, 2, 64, 16, LENS),
        W.random_workload(2103, W.BF16, 8, 1, 128, 16, LENS, window=100),
        W.random_workload(2104, W.BF16, 32, 8, 128, 16, LENS, fp8_scales=(0.05, 0.04)),
        W.random_workload(2108, W.F16, 8, 8, 128, 16, LENS, garbage="nan"),
        W.random_workload(2109, W.BF16, 4, 4, 64, 16, LENS, fp8_scales=(0.03, 0.06)),
    ]


@pytest.mark.parametrize("k", range(6))
def test_parity_and_bits_with_early_tables(cuda_device, k):
    wl = _cases()[k]
    st = GpuState(wl)
    # the step's own cache write precedes the decode: its new rows must be seen
    out, _ = gpu_step(st, flags=TR)
    assert pa.pa_get_error(st.err) == 0
    ref = OracleState(wl)
    ref.step()
    expected, spread = ref.decode(spread=True)
    check_parity(out, wl, expected, spread, "%s tables-ready" % wl.name, flags=TR)
    plain = gpu_decode(st, st.seq_lens)
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))


@pytest.mark.parametrize("num_ctas", [3, 40])
def test_split_contexts_with_early_tables(cuda_device, num_ctas):
    wl = W.random_workload(2105, W.BF16, 32, 8, 128, 16, [5000, 64, 1, 2300])
    st = GpuState(wl)
    out, _ = gpu_step(st, flags=TR, num_ctas=num_ctas)
    ref = OracleState(wl)
    ref.step()
    expected, spread = ref.decode(spread=True)
    check_parity(out, wl, expected, spread, "split, tables-ready", flags=TR)
    assert pa.pa_get_error(st.err) == 0


def test_empty_and_bad_lengths_with_early_tables(cuda_device):
    wl = W.random_workload(2106, W.F16, 8, 2, 64, 16, [1, 40, 1, 17])
    st = GpuState(wl)
    # out starts as garbage: the zero rows are written, not inherited
    out = torch.full_like(st.q, float("nan"))
    sl = torch.tensor([0, 40, 0, 17], dtype=torch.int32, device="cuda")
    pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, sl, wl.scale, out=out,
                 flags=TR, err=st.err)
    assert pa.pa_get_error(st.err) == 0
    o = gpu_out_f64(out)
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    ref = oracle.paged_decode(wl.q, wl.k_cache, wl.v_cache, wl.dtype, wl.block_tables,
                              np.array([0, 40, 0, 17], np.int32), wl.scale)
    assert_close(o, ref, "zero lengths, tables-ready")
    bad = torch.tensor([-3, 40, 10 ** 6, 17], dtype=torch.int32, device="cuda")
    out = pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, bad, wl.scale, flags=TR,
                       err=st.err)
    assert pa.pa_get_error(st.err) == pa.PA_DEVERR_SEQ_LEN
    o = gpu_out_f64(out)
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    assert_close(o[[1, 3]], ref[[1, 3]], "valid rows next to invalid ones, tables-ready")


def test_unknown_flag_bits_are_rejected(cuda_device):
    wl = W.random_workload(2107, W.BF16, 8, 2, 128, 16, [50])
    st = GpuState(wl)
    with pytest.raises(RuntimeError):
        pa.pa_decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, wl.scale,
                     flags=0x200)
