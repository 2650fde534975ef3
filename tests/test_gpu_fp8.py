"""FP8 (E4M3) KV cache on the GPU against the fp64 oracle.

The quantizing cache write must produce the oracle's codes bit for bit
(code = e4m3(float32(x) / scale), round to nearest even, saturating); the
decode over E4M3 pools must match the oracle's decode of the dequantized cache
element by element within |gpu - oracle| <= 4e-3 + 1e-2 |oracle|, over
head_dim, query dtype, group size (CUDA-core and tensor-core kernels), block
size, ragged lengths, NaN codes in unread slots and contexts split across
thread blocks.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_72_gb300 as pa
import workloads as W
from harness import GpuState, OracleState, assert_close, check_parity, gpu_out_f64, gpu_step

pytestmark = pytest.mark.gpu

EDGE_LENS = [1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 200, 777]
SCALES = (2.0 ** -6, 2.0 ** -6)


def _parity(wl, flags=pa.PA_DECODE_AUTO, num_ctas=0):
    st = GpuState(wl)
    out, _ = gpu_step(st, flags=flags, num_ctas=num_ctas)
    ref = OracleState(wl)
    ref.step()
    assert np.array_equal(st.k_cache.cpu().numpy(), ref.k_cache), "K codes differ"
    assert np.array_equal(st.v_cache.cpu().numpy(), ref.v_cache), "V codes differ"
    expected, spread = ref.decode(spread=True)
    rep = check_parity(out, wl, expected, spread,
                       "%s flags=%d ctas=%d" % (wl.name, flags, num_ctas), flags=flags)
    assert pa.pa_get_error(st.err) == 0
    return rep["max_abs"]


def test_fp8_cache_write_is_bit_exact_with_saturation_and_ties(cuda_device):
    # small scales push some values past 448 (saturation); f16 and bf16 inputs
    for dtype, scales in ((W.BF16, (0.004, 0.0021)), (W.F16, (2.0 ** -7, 0.05))):
        wl = W.random_workload(51, dtype, 8, 8, 128, 16, [3, 40, 129], fp8_scales=scales)
        st = GpuState(wl)
        gpu_step(st, decode=False)
        ref = OracleState(wl)
        ref.step()
        assert np.array_equal(st.k_cache.cpu().numpy(), ref.k_cache)
        assert np.array_equal(st.v_cache.cpu().numpy(), ref.v_cache)
        assert pa.pa_get_error(st.err) == 0
        # saturation did happen
        codes = st.k_cache.cpu().numpy().reshape(-1)
        assert np.any((codes & 0x7F) == 0x7E)


def test_fp8_slot_mapped_cache_write_is_bit_exact(cuda_device):
    # the one-launch slot mapping + quantizing write gives the oracle's slots
    # and codes (saturation included) and leaves the pools as the two calls do
    for dtype, scales in ((W.BF16, (0.004, 0.0021)), (W.F16, (2.0 ** -7, 0.05))):
        wl = W.random_workload(52, dtype, 8, 8, 128, 16, [3, 40, 129], fp8_scales=scales)
        st = GpuState(wl)
        ref = OracleState(wl)
        ref.step()
        slots = torch.full((wl.new_seq.size,), 7, dtype=torch.int64, device="cuda")
        pa.pa_cache_write_fp8_mapped(st.k_new, st.v_new, st.block_tables, st.new_seq, st.new_pos,
                                     st.k_cache, st.v_cache, wl.k_scale, wl.v_scale,
                                     slot_mapping=slots, err=st.err)
        assert np.array_equal(slots.cpu().numpy(), ref.slots)
        assert np.array_equal(st.k_cache.cpu().numpy(), ref.k_cache)
        assert np.array_equal(st.v_cache.cpu().numpy(), ref.v_cache)
        assert pa.pa_get_error(st.err) == 0
    # a bad table entry: slot -1, nothing written, the block-id bit
    bt = torch.tensor([[9]], dtype=torch.int32, device="cuda")
    one = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.ones(1, 2, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 4, 2, 64, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.zeros(1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_cache_write_fp8_mapped(k, k, bt, one, one, kc, vc, 1.0, 1.0, slot_mapping=slots, err=err)
    assert slots.item() == -1 and not kc.any() and not vc.any()
    assert pa.pa_get_error(err) == pa.PA_DEVERR_BLOCK_ID


CASES = [
    # q dtype, Hq, Hkv, D, B
    (W.BF16, 8, 8, 128, 16),     # G = 1: CUDA-core kernel
    (W.F16, 4, 4, 64, 16),
    (W.BF16, 32, 8, 128, 16),    # the Llama-3-8B shape
    (W.F16, 8, 2, 64, 16),
    (W.BF16, 16, 2, 128, 8),
    (W.F16, 64, 8, 128, 16),     # G = 8
    (W.BF16, 32, 2, 128, 32),    # G = 16: both MMA row halves
    (W.F16, 6, 3, 64, 8),        # H_kv = 3: one KV head per group, 8 boxes a chunk
    (W.BF16, 12, 4, 128, 256),
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,B", CASES)
def test_fp8_decode_parity_sweep(cuda_device, dtype, Hq, Hkv, D, B):
    wl = W.random_workload(60 + Hq + D + B, dtype, Hq, Hkv, D, B, EDGE_LENS, garbage="nan",
                           fp8_scales=SCALES)
    _parity(wl)
    if Hq == Hkv:
        _parity(wl, flags=pa.PA_DECODE_MMA)


@pytest.mark.parametrize("num_ctas", [1, 3, 50, 1000])
def test_fp8_split_contexts(cuda_device, num_ctas):
    lens = [3000, 1, 64, 65, 900, 2048, 5, 4096]
    wl = W.random_workload(71, W.BF16, 32, 8, 128, 16, lens, fp8_scales=SCALES)
    _parity(wl, num_ctas=num_ctas)


def test_fp8_copy_blocks_is_bit_exact(cuda_device):
    wl = W.random_workload(72, W.BF16, 8, 2, 64, 16, [40, 70, 5], fp8_scales=SCALES)
    st = GpuState(wl)
    used = np.unique(wl.block_tables[wl.block_tables >= 0])
    free = np.setdiff1d(np.arange(wl.num_blocks), used)
    pairs = np.stack([used[:3], free[:3]], axis=1).astype(np.int32)
    pa.pa_copy_blocks(torch.from_numpy(pairs).cuda(), st.k_cache, st.v_cache, err=st.err)
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.copy_blocks(kc, vc, pairs)
    assert np.array_equal(st.k_cache.cpu().numpy(), kc)
    assert np.array_equal(st.v_cache.cpu().numpy(), vc)
    assert pa.pa_get_error(st.err) == 0


def test_fp8_scales_are_checked(cuda_device):
    wl = W.random_workload(73, W.BF16, 8, 2, 64, 16, [10], fp8_scales=SCALES)
    st = GpuState(wl)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_fp8(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, wl.scale,
                         0.0, 1.0)
    assert e.value.status == 1
    with pytest.raises(pa.PAError):
        pa.pa_decode_fp8(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens, wl.scale,
                         1.0, float("nan"))
