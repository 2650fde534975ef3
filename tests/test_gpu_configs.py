"""The five workloads end to end on the GPU (copy-on-write, slot mapping,
cache write, decode) against the oracle, at full size, each as separate
eager calls (the benchmark's own graph-captured step is checked in
test_gpu_bench_step.py)."""
import numpy as np
import pytest

import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import GpuState, OracleState, bits_of, check_parity, gpu_step

pytestmark = pytest.mark.gpu


def _run(wl, seq_ids=None):
    st = GpuState(wl)
    out, slots = gpu_step(st)
    assert pa.pa_get_error(st.err) == 0
    ref = OracleState(wl)
    ref.step()
    assert np.array_equal(slots.cpu().numpy(), ref.slots)
    expected, spread = ref.decode(seq_ids=seq_ids, spread=True)
    rep = check_parity(out, wl, expected, spread, wl.name, rows=seq_ids)
    return st, ref, rep["max_abs"]


def test_tiny():
    st, ref, _ = _run(W.tiny())
    assert np.array_equal(bits_of(st.k_cache), ref.k_cache)


def test_llama2_7b():
    _run(W.llama2_7b())


def test_llama3_8b_gqa():
    st, ref, _ = _run(W.llama3_8b())
    # the whole pool, not just the written slots, is bit-identical
    assert np.array_equal(bits_of(st.v_cache), ref.v_cache)


def test_qwen2_shared_prefix_copy_on_write():
    wl = W.shared_prefix(garbage="nan")
    assert wl.copy_pairs.shape[0] == 11
    st, ref, _ = _run(wl)
    assert np.array_equal(bits_of(st.k_cache), ref.k_cache)
    assert np.array_equal(bits_of(st.v_cache), ref.v_cache)


def test_70b_long_context_sampled():
    wl = W.long_context_70b()
    ids = np.array([0, 7, 19, 31], np.int32)
    _run(wl, seq_ids=ids)
